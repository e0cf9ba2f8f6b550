// Host-side plumbing shared by the library's translation units: tensor-map
// encoding through the driver entry point, the per-device status word and
// small launch helpers.  Not part of the public ABI (see include/fa.h).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/fa.h"
#include "fa_status_bits.h"

namespace fa {

// Address of the library's device status word on the current device
// (nullptr if CUDA fails).  Obtained once per device from a file-scope
// __device__ variable; the library allocates no memory for it.
unsigned* device_status_ptr();

// Encode a tiled bf16 tensor map with the 128-byte swizzle.
// dims/strides follow the CUDA driver convention: dims[0] innermost (elements),
// strides_bytes[i] is the stride of dims[i + 1].  Returns false on failure.
bool encode_bf16_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                      const uint32_t* box);

// Encode a tiled fp32 tensor map without swizzle (row-major boxes in shared memory).
bool encode_f32_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                     const uint32_t* box);

// Encode a tiled fp32 tensor map with the 128-byte swizzle (box rows of 32
// elements; in shared memory the 16-byte chunk c of row y sits at chunk c ^ (y % 8)).
bool encode_f32_sw128_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides_bytes, const uint32_t* box);

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

inline fa_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Launchers implemented by the kernel translation units.  Arguments are
// validated by the public entry points before these are called.
fa_status fwd_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                     int causal, float scale, const int32_t* kv_lens, const uint8_t* block_mask,
                     long long mask_stride, cudaStream_t stream);
// largest N the block-sparse forward takes (its key-tile bitmask holds 2048 tiles)
constexpr int kBlockSparseMaxN = 2048 * 128;
fa_status fwd_varlen_launch(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            const int32_t* cu_seqlens, int num_seqs, int total, int max_seqlen, int H, int d,
                            int causal, float scale, cudaStream_t stream);
fa_status fwd_paged_launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                           const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o, float* lse,
                           int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int num_blocks,
                           int block_size, int max_blocks, int causal, float scale, cudaStream_t stream);
fa_status bwd_varlen_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                            const float* LSE, void* dQ, void* dK, void* dV, const int32_t* cu_seqlens, int num_seqs,
                            int total, int max_seqlen, int H, int d, int causal, float scale, void* workspace,
                            cudaStream_t stream);
fa_status bwd_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                     void* dQ, void* dK, void* dV, int B, int H, int N, int d, int causal, float scale,
                     const int32_t* kv_lens, void* workspace, cudaStream_t stream);
// Host setup of the decode kernels on the current device (shared-memory limit),
// done once per device; the graph builder calls it outside any stream capture.
fa_status decode_prepare();
// Raises `func`'s dynamic shared-memory limit to `bytes` on the current device,
// once per (kernel, device); false on failure.
bool set_smem_limit(const void* func, int bytes);
// Number of SMs of the current device (0 if CUDA fails), looked up once per device.
int sm_count();

// FA_DEBUG builds: arm a one-shot stall of the backward main kernel's MMA warp
// before work item `item`, with wait limit `timeout_ns` for that launch;
// false (nothing armed) in release builds.
bool arm_backward_stall(int item, unsigned long long timeout_ns);
// FA_DEBUG builds: arm a one-shot stall of the forward's MMA warp in CTA
// `cta` (linear block index) with wait limit `timeout_ns`; false in release.
bool arm_forward_stall(long long cta, unsigned long long timeout_ns);
// FA_DEBUG builds: arm a one-shot stall of the paged decode split kernel's
// producer in CTA `cta` (linear block index); false in release builds.
bool arm_decode_stall(long long cta, unsigned long long timeout_ns);
// Loads the tensor-map encoder entry point if needed; false if unavailable.
bool encode_init();
// Argument checks shared by every paged-decode entry point (with and without
// a caller workspace); the workspace itself is checked by the caller.
fa_status decode_check_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                            const int32_t* seq_lens, const void* o, int B, int Hq, int Hkv, int d, int block_size,
                            int max_blocks, int num_blocks, int num_splits, float scale);
fa_status decode_launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d, int block_size,
                        int max_blocks, int num_blocks, int num_splits, float scale, void* workspace,
                        cudaStream_t stream);

}  // namespace fa
