// Public C entry points (include/fa.h): argument validation, the device
// status word and tensor-map encoding.  The kernels live in fa_fwd.cu,
// fa_bwd.cu and fa_decode.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <cudaTypedefs.h>

#include <mutex>
#include <utility>
#include <vector>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {

// One status word per device (each device that loads the library holds its
// own copy of this variable).
__device__ unsigned g_fa_status;

namespace {

constexpr int kMaxDevices = 64;
unsigned* g_status_ptr[kMaxDevices] = {};
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

unsigned* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_status_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_fa_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<unsigned*>(p);
  }
  return g_status_ptr[dev];
}

fa_status decode_check_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const void* o, int B, int Hq, int Hkv, int d, int block_size,
                            int max_blocks, int num_blocks, int num_splits, float scale) {
  if (B < 1 || Hq < 1 || Hkv < 1 || max_blocks < 1 || num_blocks < 1 || num_splits < 0) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !isfinite(scale)) return FA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || block_size < 16 || block_size % 16 != 0) return FA_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16 || num_splits > 16) return FA_ERR_UNSUPPORTED;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  // the kernels index cache rows and table-row keys in 32-bit integers
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL ||
      static_cast<long long>(max_blocks) * block_size > 0x7fffffffLL)
    return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

namespace {
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle, const void* base, int rank,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);
}  // namespace

bool encode_bf16_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, base, rank, dims,
                     strides_bytes, box);
}

bool encode_f32_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, base, rank, dims,
                     strides_bytes, box);
}

bool encode_f32_sw128_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box) {
  return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B, base, rank, dims,
                     strides_bytes, box);
}

bool set_smem_limit(const void* func, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;  // (kernel, device) pairs already raised
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& e : done)
    if (e.first == func && e.second == dev) return true;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  done.emplace_back(func, dev);
  return true;
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  static int counts[kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev] = n;
  }
  return counts[dev];
}

bool encode_init() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return false;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return true;
}

namespace {
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle, const void* base, int rank,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box) {
  if (!encode_init()) return false;
  cuuint64_t gdim[5];
  cuuint64_t gstr[4];
  cuuint32_t bdim[5];
  cuuint32_t estr[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estr[i] = 1;
    if (i + 1 < rank) gstr[i] = strides_bytes[i];
  }
  CUresult r = g_encode(map, dtype, static_cast<cuuint32_t>(rank), const_cast<void*>(base), gdim, gstr, bdim, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}
}  // namespace

// Lane 0 asks the bounds guard about element 3 of a 3-element extent; no
// memory is touched either way.
__global__ void selftest_bounds_kernel(unsigned* status) {
  if (threadIdx.x == 0) {
    volatile bool ok = FA_IN_BOUNDS(3, 3, status);
    (void)ok;
  }
}

// One CTA waits on an mbarrier that nothing ever completes; the bounded wait
// must give up after `timeout_ns`, latch the timeout bit and let the kernel end.
__global__ void selftest_wait_kernel(unsigned* status, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtx wc{&abort_flag, status, timeout_ns};
  (void)mbar_wait(smem_u32(&bar), 0, wc);
}

}  // namespace fa

using fa::aligned16;

namespace {

bool bad_scale(float s) { return !(s > 0.f) || !isfinite(s); }

int check_attn(const void* Q, const void* K, const void* V, const void* O, const void* LSE, int B, int H, int N, int d,
               float scale) {
  if (B < 1 || H < 1 || N < 0) return FA_ERR_INVALID_ARG;
  if (bad_scale(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (N == 0) return FA_OK;
  if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE)) return FA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if ((static_cast<long long>(N) + 255) / 256 > 65535) return FA_ERR_UNSUPPORTED;
  return FA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

extern "C" {

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_BAD_BLOCK_TABLE: return "FA_ERR_BAD_BLOCK_TABLE";
    case FA_ERR_OUT_OF_BOUNDS: return "FA_ERR_OUT_OF_BOUNDS";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_version(void) { return 109; }

int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d, int causal,
              float scale, const int32_t* kv_lens, void* stream) {
  int st = check_attn(Q, K, V, O, LSE, B, H, N, d, scale);
  if (st != FA_OK || N == 0) return st;
  if (B > 65535) return FA_ERR_UNSUPPORTED;  // batch entries are the grid's z dimension
  return fa::fwd_launch(Q, K, V, O, LSE, B, H, N, d, causal, scale, kv_lens, nullptr, 0,
                        static_cast<cudaStream_t>(stream));
}

int fa_fwd_block_sparse(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                        int causal, float scale, const int32_t* kv_lens, const uint8_t* block_mask,
                        int mask_per_head, void* stream) {
  int st = check_attn(Q, K, V, O, LSE, B, H, N, d, scale);
  if (st != FA_OK || N == 0) return st;
  if (block_mask == nullptr) return FA_ERR_INVALID_ARG;
  if (B > 65535 || N > fa::kBlockSparseMaxN) return FA_ERR_UNSUPPORTED;
  const long long nb = (static_cast<long long>(N) + 127) / 128;
  const long long stride = mask_per_head ? nb * nb : 0;
  return fa::fwd_launch(Q, K, V, O, LSE, B, H, N, d, causal, scale, kv_lens, block_mask, stride,
                        static_cast<cudaStream_t>(stream));
}

int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d, int causal,
           float scale, void* stream) {
  return fa_fwd_ex(Q, K, V, O, LSE, B, H, N, d, causal, scale, nullptr, stream);
}

int fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE, const int32_t* cu_seqlens,
                  int num_seqs, int total, int max_seqlen, int H, int d, int causal, float scale, void* stream) {
  if (num_seqs < 1 || total < 0 || max_seqlen < 0 || H < 1) return FA_ERR_INVALID_ARG;
  if (bad_scale(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (total == 0 || max_seqlen == 0) return FA_OK;
  if (!Q || !K || !V || !O || !LSE || !cu_seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE)) return FA_ERR_INVALID_ARG;
  if (num_seqs > 65535) return FA_ERR_UNSUPPORTED;  // sequences are the grid's z dimension
  if (static_cast<long long>(num_seqs) * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if ((static_cast<long long>(max_seqlen) + 255) / 256 > 65535) return FA_ERR_UNSUPPORTED;
  return fa::fwd_varlen_launch(Q, K, V, O, LSE, cu_seqlens, num_seqs, total, max_seqlen, H, d, causal, scale,
                               static_cast<cudaStream_t>(stream));
}

int fa_paged_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                     const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o, float* lse, int num_seqs,
                     int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int num_blocks, int block_size,
                     int max_blocks, int causal, float scale, void* stream) {
  if (num_seqs < 1 || total_q < 0 || max_seqlen_q < 0 || Hq < 1 || Hkv < 1 || num_blocks < 1 || max_blocks < 1 ||
      block_size < 1)
    return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0 || bad_scale(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  // a 128-key tile is gathered as whole boxes of min(block_size, 128) rows,
  // each a multiple of 8 rows (one 1024-byte swizzle period)
  if (block_size % 8 != 0 || (128 % block_size != 0 && block_size % 128 != 0)) return FA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || static_cast<long long>(num_seqs) * Hq > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size >= 0x7fffffffLL ||
      static_cast<long long>(max_blocks) * block_size >= 0x7fffffffLL)
    return FA_ERR_UNSUPPORTED;
  if ((static_cast<long long>(max_seqlen_q) + 255) / 256 > 65535) return FA_ERR_UNSUPPORTED;
  if (total_q == 0 || max_seqlen_q == 0) return FA_OK;
  if (!q || !k_cache || !v_cache || !block_table || !cu_seqlens_q || !seq_lens_k || !o || !lse)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse))
    return FA_ERR_INVALID_ARG;
  return fa::fwd_paged_launch(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, o, lse, num_seqs, total_q,
                              max_seqlen_q, Hq, Hkv, d, num_blocks, block_size, max_blocks, causal, scale,
                              static_cast<cudaStream_t>(stream));
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (B < 1 || H < 1 || N < 0 || d < 1) return 0;
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t npad = (static_cast<size_t>(N) + 127) / 128 * 128;
  // -D and -LSE2 rows, the fp32 dQ accumulator, the main kernel's work counter
  return 2 * round256(bh * npad * sizeof(float)) + round256(bh * N * d * sizeof(float)) + 256;
}

int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE, void* dQ,
           void* dK, void* dV, int B, int H, int N, int d, int causal, float scale, const int32_t* kv_lens,
           void* workspace, size_t ws_bytes, void* stream) {
  int st = check_attn(Q, K, V, O, LSE, B, H, N, d, scale);
  if (st != FA_OK || N == 0) return st;
  if (!dO || !dQ || !dK || !dV || !workspace) return FA_ERR_INVALID_ARG;
  if (!aligned16(dO) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV)) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
  if (ws_bytes < fa_bwd_workspace_size(B, H, N, d)) return FA_ERR_INVALID_ARG;
  return fa::bwd_launch(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, d, causal, scale, kv_lens, workspace,
                        static_cast<cudaStream_t>(stream));
}

size_t fa_bwd_varlen_workspace_size(int num_seqs, int total, int max_seqlen, int H, int d) {
  if (num_seqs < 1 || total < 0 || max_seqlen < 0 || H < 1 || d < 1) return 0;
  const size_t rows = static_cast<size_t>(num_seqs) * H * ((static_cast<size_t>(max_seqlen) + 127) / 128 * 128);
  return 2 * round256(rows * sizeof(float)) + round256(static_cast<size_t>(total) * H * d * sizeof(float)) + 256;
}

int fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                  void* dQ, void* dK, void* dV, const int32_t* cu_seqlens, int num_seqs, int total, int max_seqlen,
                  int H, int d, int causal, float scale, void* workspace, size_t ws_bytes, void* stream) {
  if (num_seqs < 1 || total < 0 || max_seqlen < 0 || H < 1) return FA_ERR_INVALID_ARG;
  if (bad_scale(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || static_cast<long long>(num_seqs) * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  // (the work-item grid's x extent, key tiles x 8 heads, must fit an int)
  if ((static_cast<long long>(max_seqlen) + 127) / 128 * 8 > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
  if (total == 0 || max_seqlen == 0) return FA_OK;
  if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !cu_seqlens || !workspace)
    return FA_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) || !aligned16(dQ) ||
      !aligned16(dK) || !aligned16(dV))
    return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
  if (ws_bytes < fa_bwd_varlen_workspace_size(num_seqs, total, max_seqlen, H, d)) return FA_ERR_INVALID_ARG;
  return fa::bwd_varlen_launch(Q, K, V, O, dO, LSE, dQ, dK, dV, cu_seqlens, num_seqs, total, max_seqlen, H, d, causal,
                               scale, workspace, static_cast<cudaStream_t>(stream));
}

size_t fa_paged_decode_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B < 1 || Hq < 1 || d < 1 || num_splits < 0 || num_splits > 16) return 0;
  if (num_splits == 1) return 0;  // one split writes the output directly
  const int S = num_splits == 0 ? 16 : num_splits;
  const size_t n = static_cast<size_t>(B) * Hq * S;
  return round256(n * d * sizeof(float)) + round256(n * 2 * sizeof(float));
}

int fa_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d, int block_size,
                    int max_blocks, int num_blocks, int num_splits, float scale, void* workspace, size_t ws_bytes,
                    void* stream) {
  const fa_status st = fa::decode_check_args(q, k_cache, v_cache, block_table, seq_lens, o, B, Hq, Hkv, d, block_size,
                                             max_blocks, num_blocks, num_splits, scale);
  if (st != FA_OK) return st;
  if (num_splits != 1 && !workspace) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return FA_ERR_INVALID_ARG;
  const int S = num_splits == 0 ? 16 : num_splits;
  if (ws_bytes < fa_paged_decode_workspace_size(B, Hq, d, S)) return FA_ERR_INVALID_ARG;
  return fa::decode_launch(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, d, block_size, max_blocks,
                           num_blocks, S, scale, workspace, static_cast<cudaStream_t>(stream));
}

int fa_debug_build(void) {
#ifdef FA_DEBUG
  return 1;
#else
  return 0;
#endif
}

int fa_selftest_bounds(void* stream) {
  unsigned* status = fa::device_status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  fa::selftest_bounds_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status);
  return fa::launch_status();
}

int fa_debug_stall_backward(int item, unsigned timeout_us) {
  if (item < 0 || timeout_us == 0 || timeout_us > 1000000u) return FA_ERR_INVALID_ARG;
  return fa::arm_backward_stall(item, static_cast<unsigned long long>(timeout_us) * 1000ull) ? FA_OK
                                                                                             : FA_ERR_UNSUPPORTED;
}

int fa_debug_stall_forward(int cta, unsigned timeout_us) {
  if (cta < 0 || timeout_us == 0 || timeout_us > 1000000u) return FA_ERR_INVALID_ARG;
  return fa::arm_forward_stall(cta, static_cast<unsigned long long>(timeout_us) * 1000ull) ? FA_OK
                                                                                           : FA_ERR_UNSUPPORTED;
}

int fa_debug_stall_decode(int cta, unsigned timeout_us) {
  if (cta < 0 || timeout_us == 0 || timeout_us > 1000000u) return FA_ERR_INVALID_ARG;
  return fa::arm_decode_stall(cta, static_cast<unsigned long long>(timeout_us) * 1000ull) ? FA_OK
                                                                                         : FA_ERR_UNSUPPORTED;
}

int fa_selftest_wait_timeout(unsigned timeout_us, void* stream) {
  if (timeout_us == 0 || timeout_us > 1000000u) return FA_ERR_INVALID_ARG;
  unsigned* status = fa::device_status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  fa::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, static_cast<unsigned long long>(timeout_us) * 1000ull);
  return fa::launch_status();
}

int fa_get_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, fa::g_fa_status, sizeof(v)) != cudaSuccess) return FA_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
  }
  if (v & fa::kStatusBoundsBit) return FA_ERR_OUT_OF_BOUNDS;
  if (v & fa::kStatusLaunchBit) return FA_ERR_CUDA;
  if (v & fa::kStatusBadArgBit) return FA_ERR_INVALID_ARG;
  if (v & fa::kStatusTimeoutBit) return FA_ERR_TIMEOUT;
  if (v & fa::kStatusBadTableBit) return FA_ERR_BAD_BLOCK_TABLE;
  return FA_OK;
}

}  // extern "C"
