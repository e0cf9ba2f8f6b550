// Paged, split-KV, grouped-query decode ("S12 FlashAttention": the paged loop
// of "实现", flash-decoding's split + (m, l, o) merge, and GQA head sharing).
//
// Kernel 1 (split): one CTA per (split s, KV head g, sequence b).  The split's
// logical blocks are gathered through the block table by TMA (each 16-token
// block of KV head g is a 16 x 128 bf16 box, K and V) into an 8-stage shared-
// memory ring.  Four consumer warps take the blocks round-robin; each keeps
// its own online-softmax state for the G = Hq / Hkv query heads of the group
// (one KV read serves all G heads).  The 16-row tensor-core tile holds the G
// heads (rows >= G are zero), so scores and P V are mma.sync m16n8k16
// products; the kernel is bound by the KV stream from HBM, not by them.
// At the end the four warp states merge in shared memory into one partial
// (m, l, o) per (b, head, split), written to the workspace.
//
// With a single split the first kernel finishes the job itself: it normalises
// o by l and writes o and lse, so one launch and no workspace serve short
// contexts (the launch-overhead remark closing the S12 chapter).
//
// Kernel 2 (combine): one warp per (b, query head) merges the splits:
// m = max m_s, l = sum 2^(m_s - m) l_s, o = sum 2^(m_s - m) o_s / l, skipping
// empty splits ("精读笔记 08：FlashAttention" §3.1 merge rule).
//
// All maxima are kept in log2 units of the scaled logit (x = scale log2(e) q.k).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <mutex>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kDMax = 128;         // largest head dimension (64 and 128 are built)
constexpr int kBlk = 16;           // tokens per chunk (one ring stage); cache blocks hold a multiple of it
constexpr int kConsumers = 4;      // consumer warps
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kStages = 8;
constexpr int kHalfBytes = kBlk * 128;           // 16 rows x 128 B (64 bf16)

template <int D>
struct DecCfg {
  static constexpr int kHalves = D / 64;                        // 128-byte halves per row
  static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;  // K halves, then V halves
  static constexpr int kOffBar = kStages * kStageBytes;
  static constexpr int kMergeBytes = kConsumers * (16 * D + 32) * 4;  // per-warp O rows + m, l
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static_assert(kMergeBytes <= kOffBar, "merge scratch reuses the stage ring");
};
// A split covers at least kMinBlocksPerSplit blocks (512 keys) when the batch
// alone fills the GPU (B * Hkv >= kFewUnits), else kMinBlocksPerSplitFew (128
// keys), so a small batch still spreads its keys over enough CTAs.
constexpr int kMinBlocksPerSplit = 32;
constexpr int kMinBlocksPerSplitFew = 8;
constexpr int kFewUnits = 152;

__host__ __device__ inline int splits_for(int nblocks, int max_splits, int min_blocks) {
  int s = (nblocks + min_blocks - 1) / min_blocks;
  return max(1, min(max_splits, s));
}

struct DecArgs {
  const __nv_bfloat16* q;  // [B, Hq, D]
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* part_o;   // [B, Hq, S, D] unnormalised o of each split (rows 512 B, 16-byte aligned)
  float* part_ml;  // [B, Hq, S, 2] m (log2 units), l
  __nv_bfloat16* o;
  float* lse;
  int B, Hq, Hkv, G, max_blocks, num_blocks, S;
  int direct;  // S == 1: the split kernel writes o and lse itself
  int block_size;  // tokens per cache block, a multiple of kBlk
  int min_blocks;  // smallest split, in blocks
  float scale_log2;
  unsigned* status;
#ifdef FA_DEBUG
  long long dbg_stall_cta;            // the producer of this split CTA (linear index) loads nothing (-1: none)
  unsigned long long dbg_timeout_ns;  // wait limit of this launch (0: the default)
#endif
};

#ifdef FA_DEBUG
// One-shot stall armed by fa_debug_stall_decode, taken by the next decode
// launch (host side, not thread-safe: a debug hook).
long long g_dec_stall_cta = -1;
unsigned long long g_dec_stall_timeout_ns = 0;
void take_decode_stall(DecArgs& a) {
  a.dbg_stall_cta = g_dec_stall_cta;
  a.dbg_timeout_ns = g_dec_stall_timeout_ns;
  g_dec_stall_cta = -1;
  g_dec_stall_timeout_ns = 0;
}
#endif

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Address of 16-byte chunk `cd` (0..15 along d) of row `row` in a K or V block
// stored as two 128-byte-swizzled halves of 16 rows.
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int row, int cd) {
  return base + (cd >> 3) * kHalfBytes + row * 128 + ((((cd & 7) ^ (row & 7))) << 4);
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > 50000000ull) break;
  }
}

// kUnit: block_size == 16, so chunk c is simply block table[c] (no division)
template <int D, bool kUnit>
__global__ void __launch_bounds__(kThreads, 3)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const DecArgs a) {
  using C = DecCfg<D>;
  constexpr int kOffBar = C::kOffBar;
  constexpr int kStageBytes = C::kStageBytes;
  // launched as a programmatic dependent: the CTAs may be resident before the
  // previous kernel in the stream has finished, so nothing it may write is
  // read before griddep_wait(); the combine kernel may then be scheduled
  griddep_wait();
  griddep_launch_dependents();
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  // the work is cut into 16-token chunks; chunk c lives in cache block
  // table[c * 16 / block_size] at row (c * 16) % block_size
  const int L = FA_IN_BOUNDS(b, a.B, a.status) ? min(max(a.seq_lens[b], 0), a.max_blocks * a.block_size) : 0;
  const int nb = (L + kBlk - 1) / kBlk;
  const int S_b = splits_for(nb, a.S, a.min_blocks);
  if (s >= S_b) return;  // this sequence uses fewer splits
  const int lo = static_cast<int>((static_cast<long long>(s) * nb) / S_b);
  const int hi = static_cast<int>((static_cast<long long>(s + 1) * nb) / S_b);
  const int nblk = hi - lo;
  const int32_t* table = a.block_table + static_cast<size_t>(b) * a.max_blocks;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * i; };
  auto empty = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (kStages + i); };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + 8 * 2 * kStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
#ifdef FA_DEBUG
  const WaitCtx wc{abort_flag, a.status, a.dbg_timeout_ns != 0 ? a.dbg_timeout_ns : kWaitTimeoutNs};
#else
  const WaitCtx wc{abort_flag, a.status};
#endif

  // per-thread softmax state for rows r0 = lane / 4 and r0 + 8 of the group
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int issued = 0;
      int n_load = nblk;
#ifdef FA_DEBUG
      const long long cta = blockIdx.x + static_cast<long long>(gridDim.x) *
                                             (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z);
      if (cta == a.dbg_stall_cta) n_load = 0;  // injected stall: this warp loads nothing
#endif
      for (int i = 0; i < n_load; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(empty(st), ((i / kStages) & 1) ^ 1, wc)) break;
        const int chunk_key = (lo + i) * kBlk;
        const int te = kUnit ? lo + i : chunk_key / a.block_size;
        const int phys = FA_IN_BOUNDS(static_cast<long long>(b) * a.max_blocks + te,
                                      static_cast<long long>(a.B) * a.max_blocks, a.status)
                             ? __ldg(table + te)
                             : -1;
        if (phys >= 0 && phys < a.num_blocks) {
          mbar_arrive_expect_tx(full(st), kStageBytes);
          const uint32_t dst = sbase + st * kStageBytes;
          const int z = kUnit ? phys * kBlk : phys * a.block_size + chunk_key % a.block_size;
#pragma unroll
          for (int h = 0; h < C::kHalves; ++h) {
            tma_load_3d(dst + h * kHalfBytes, &tmK, full(st), 64 * h, g, z);
            tma_load_3d(dst + (C::kHalves + h) * kHalfBytes, &tmV, full(st), 64 * h, g, z);
          }
        } else {
          atomicOr(a.status, kStatusBadTableBit);
          mbar_arrive(full(st));  // nothing to load: the consumer masks this block
        }
        issued = i + 1;
      }
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int i_last = st + kStages * ((issued - 1 - st) / kStages);
        drain_wait(full(st), (i_last / kStages) & 1);
      }
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int r0 = lane >> 2;
    const int c2 = 2 * (lane & 3);
    const int h0 = g * a.G;
    // Q as the A operand (16 x 128, rows >= G are zero), kept in registers
    uint32_t qa[D / 16][4];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q + (static_cast<size_t>(b) * a.Hq + h0 + r0) * D);
      const uint32_t* q8 = reinterpret_cast<const uint32_t*>(a.q + (static_cast<size_t>(b) * a.Hq + h0 + r0 + 8) * D);
      const bool v0 = r0 < a.G &&
                      FA_IN_BOUNDS(static_cast<long long>(b) * a.Hq + h0 + r0, static_cast<long long>(a.B) * a.Hq, a.status);
      const bool v8 = r0 + 8 < a.G && FA_IN_BOUNDS(static_cast<long long>(b) * a.Hq + h0 + r0 + 8,
                                                   static_cast<long long>(a.B) * a.Hq, a.status);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int col = (16 * ks + c2) >> 1;  // in bf16 pairs
        qa[ks][0] = v0 ? __ldg(q0 + col) : 0u;
        qa[ks][1] = v8 ? __ldg(q8 + col) : 0u;
        qa[ks][2] = v0 ? __ldg(q0 + col + 4) : 0u;
        qa[ks][3] = v8 ? __ldg(q8 + col + 4) : 0u;
      }
    }
    const float sl2 = a.scale_log2;
    // ldmatrix lane roles: matrix m = lane / 8, row i = lane % 8
    const int lm = lane >> 3, li = lane & 7;
    for (int i = warp; i < nblk; i += kConsumers) {
      const int st = i % kStages;
      if (!mbar_wait(full(st), (i / kStages) & 1, wc)) break;
      const uint32_t stK = sbase + st * kStageBytes;
      const uint32_t stV = stK + C::kHalves * kHalfBytes;
      const int te = kUnit ? lo + i : (lo + i) * kBlk / a.block_size;
      const int phys = FA_IN_BOUNDS(static_cast<long long>(b) * a.max_blocks + te,
                                    static_cast<long long>(a.B) * a.max_blocks, a.status)
                           ? __ldg(table + te)
                           : -1;
      const bool bad = !(phys >= 0 && phys < a.num_blocks);
      // ---- S = Q K^T over 16 keys (two n8 tiles)
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t k0, k1, k2, k3;
        const int key = 8 * (lm >> 1) + li;
        ldsm_x4(chunk_addr(stK, key, 2 * ks + (lm & 1)), k0, k1, k2, k3);
        mma_16816(sc[0], qa[ks], k0, k1);
        mma_16816(sc[1], qa[ks], k2, k3);
      }
      // ---- mask keys past the sequence end (and whole skipped blocks)
      const int kbase = (lo + i) * kBlk + c2;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kidx = kbase + 8 * nt + (e & 1);
          sc[nt][e] = (bad || kidx >= L) ? -INFINITY : sc[nt][e] * sl2;
        }
      // ---- online softmax for rows r0 (e = 0, 1) and r0 + 8 (e = 2, 3)
      float alpha[2];
      uint32_t pa[4];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        float mx = fmaxf(fmaxf(sc[0][2 * rr], sc[0][2 * rr + 1]), fmaxf(sc[1][2 * rr], sc[1][2 * rr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run[rr], mx);
        const float sub = (m_new == -INFINITY) ? 0.f : m_new;
        alpha[rr] = ex2_approx(m_run[rr] - sub);
        m_run[rr] = m_new;
        const float p0 = ex2_approx(sc[0][2 * rr] - sub), p1 = ex2_approx(sc[0][2 * rr + 1] - sub);
        const float p2 = ex2_approx(sc[1][2 * rr] - sub), p3 = ex2_approx(sc[1][2 * rr + 1] - sub);
        l_run[rr] = l_run[rr] * alpha[rr] + ((p0 + p1) + (p2 + p3));
        pa[rr] = pack_bf16x2(p0, p1);      // keys 0-7 : a0a1 (row r0) / a2a3 (row r0+8)
        pa[2 + rr] = pack_bf16x2(p2, p3);  // keys 8-15: a4a5 / a6a7
      }
#pragma unroll
      for (int dn = 0; dn < D / 8; ++dn) {
        acc[dn][0] *= alpha[0];
        acc[dn][1] *= alpha[0];
        acc[dn][2] *= alpha[1];
        acc[dn][3] *= alpha[1];
      }
      // ---- O += P V  (V^T fragments through ldmatrix.trans)
#pragma unroll
      for (int dn2 = 0; dn2 < D / 16; ++dn2) {
        uint32_t v0, v1, v2, v3;
        const int key = 8 * (lm & 1) + li;
        ldsm_x4_t(chunk_addr(stV, key, 2 * dn2 + (lm >> 1)), v0, v1, v2, v3);
        mma_16816(acc[2 * dn2], pa, v0, v1);
        mma_16816(acc[2 * dn2 + 1], pa, v2, v3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty(st));
    }
    // quad-reduce the row sums (each lane summed its own key columns)
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 1);
      l_run[rr] += __shfl_xor_sync(0xffffffffu, l_run[rr], 2);
    }
  }

  // ---------------------------------------------------------------- merge warps
  __syncthreads();  // every stage consumed; the ring becomes merge scratch
  float* sO = reinterpret_cast<float*>(smem);               // [warp][16][D]
  float* sML = sO + kConsumers * 16 * D;                   // [warp][16][2]
  if (warp < kConsumers) {
    const int r0 = lane >> 2, c2 = 2 * (lane & 3);
    float* w = sO + warp * 16 * D;
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      *reinterpret_cast<float2*>(w + r0 * D + 8 * dn + c2) = make_float2(acc[dn][0], acc[dn][1]);
      *reinterpret_cast<float2*>(w + (r0 + 8) * D + 8 * dn + c2) = make_float2(acc[dn][2], acc[dn][3]);
    }
    if ((lane & 3) == 0) {
      sML[(warp * 16 + r0) * 2 + 0] = m_run[0];
      sML[(warp * 16 + r0) * 2 + 1] = l_run[0];
      sML[(warp * 16 + r0 + 8) * 2 + 0] = m_run[1];
      sML[(warp * 16 + r0 + 8) * 2 + 1] = l_run[1];
    }
  }
  __syncthreads();
  if (threadIdx.x < D) {
    const int dcol = threadIdx.x;
    for (int r = 0; r < a.G; ++r) {
      float m = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) m = fmaxf(m, sML[(w * 16 + r) * 2]);
      float o = 0.f, l = 0.f;
      if (m != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          const float wm = sML[(w * 16 + r) * 2];
          const float f = ex2_approx(wm - m);  // 0 for warps that saw nothing
          o += f * sO[(w * 16 + r) * D + dcol];
          l += f * sML[(w * 16 + r) * 2 + 1];
        }
      }
      if (a.direct) {
        const size_t row = static_cast<size_t>(b) * a.Hq + g * a.G + r;
        if (!FA_IN_BOUNDS(static_cast<long long>(row), static_cast<long long>(a.B) * a.Hq, a.status)) continue;
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        a.o[row * D + dcol] = __float2bfloat16_rn(o * inv);
        if (a.lse != nullptr && dcol == 0)
          a.lse[row] = (l > 0.f) ? (m + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
        continue;
      }
      const size_t idx = (static_cast<size_t>(b) * a.Hq + g * a.G + r) * a.S + s;
      if (!FA_IN_BOUNDS(static_cast<long long>(idx), static_cast<long long>(a.B) * a.Hq * a.S, a.status)) continue;
      a.part_o[idx * D + dcol] = o;
      if (dcol == 0) {
        a.part_ml[2 * idx] = m;
        a.part_ml[2 * idx + 1] = l;
      }
    }
  }
}

// One warp per (b, query head): merge the sequence's split states; each lane
// handles D / 32 consecutive entries of o.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecArgs a) {
  constexpr int kPer = D / 32;
  griddep_wait();  // the split kernel's partial states are complete and visible
  griddep_launch_dependents();
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= a.B * a.Hq) return;
  const int b = gw / a.Hq;
  const int L = FA_IN_BOUNDS(b, a.B, a.status) ? min(max(a.seq_lens[b], 0), a.max_blocks * a.block_size) : 0;
  const int S_b = splits_for((L + kBlk - 1) / kBlk, a.S, a.min_blocks);
  const float* po = a.part_o + static_cast<size_t>(gw) * a.S * D;
  const float* pml = a.part_ml + static_cast<size_t>(gw) * a.S * 2;
  float m = -INFINITY;
  if (!FA_IN_BOUNDS(static_cast<long long>(gw) * a.S + S_b - 1, static_cast<long long>(a.B) * a.Hq * a.S, a.status))
    return;
  for (int s = 0; s < S_b; ++s)
    if (pml[2 * s + 1] > 0.f) m = fmaxf(m, pml[2 * s]);
  float o[kPer];
#pragma unroll
  for (int e = 0; e < kPer; ++e) o[e] = 0.f;
  float l = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < S_b; ++s) {
      const float ls = pml[2 * s + 1];
      if (!(ls > 0.f)) continue;
      const float f = ex2_approx(pml[2 * s] - m);
      const float* src = po + static_cast<size_t>(s) * D + kPer * lane;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        o[0] += f * v.x;
        o[1] += f * v.y;
        o[2] += f * v.z;
        o[3] += f * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        o[0] += f * v.x;
        o[1] += f * v.y;
      }
      l += f * ls;
    }
  }
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  __nv_bfloat16* dst = a.o + static_cast<size_t>(gw) * D + kPer * lane;
  if constexpr (kPer == 4) {
    uint2 w;
    w.x = pack_bf16x2(o[0] * inv, o[1] * inv);
    w.y = pack_bf16x2(o[2] * inv, o[3] * inv);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(o[0] * inv, o[1] * inv);
  }
  if (a.lse != nullptr && lane == 0)
    a.lse[gw] = (l > 0.f) ? (m + lg2_approx(l)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

fa_status decode_prepare() {
  auto raise = [](const void* f, int bytes) { return set_smem_limit(f, bytes); };
  const bool ok = raise(reinterpret_cast<const void*>(&decode_split_kernel<128, true>), DecCfg<128>::kSmemBytes) &&
                  raise(reinterpret_cast<const void*>(&decode_split_kernel<128, false>), DecCfg<128>::kSmemBytes) &&
                  raise(reinterpret_cast<const void*>(&decode_split_kernel<64, true>), DecCfg<64>::kSmemBytes) &&
                  raise(reinterpret_cast<const void*>(&decode_split_kernel<64, false>), DecCfg<64>::kSmemBytes);
  return ok ? FA_OK : FA_ERR_CUDA;
}

namespace {
template <int D>
fa_status decode_launch_d(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                          const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int block_size,
                          int max_blocks, int num_blocks, int num_splits, float scale, void* workspace,
                          cudaStream_t stream) {
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv),
                            static_cast<uint64_t>(num_blocks) * block_size};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Hkv) * D * 2};
  const uint32_t box[3] = {64, 1, kBlk};
  CUtensorMap tk, tv;
  if (!encode_bf16_tmap(&tk, k_cache, 3, dims, strides, box) || !encode_bf16_tmap(&tv, v_cache, 3, dims, strides, box))
    return FA_ERR_CUDA;
  if (decode_prepare() != FA_OK) return FA_ERR_CUDA;
  unsigned* status = device_status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  DecArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  const size_t n_part = static_cast<size_t>(B) * Hq * num_splits;
  a.part_o = static_cast<float*>(workspace);
  a.part_ml = a.part_o + ((n_part * D + 63) & ~static_cast<size_t>(63));
  a.o = static_cast<__nv_bfloat16*>(o);
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.max_blocks = max_blocks;
  a.num_blocks = num_blocks;
  a.S = num_splits;
  a.direct = num_splits == 1 ? 1 : 0;
  a.block_size = block_size;
  a.min_blocks = (static_cast<long long>(B) * Hkv >= kFewUnits) ? kMinBlocksPerSplit : kMinBlocksPerSplitFew;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
#ifdef FA_DEBUG
  take_decode_stall(a);
#endif
  // Both kernels are programmatic dependents of whatever precedes them in the
  // stream: their launch and start-up overlap the previous kernel's tail (a
  // decode step is a chain of short kernels, one pair per layer).
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_splits, Hkv, B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = DecCfg<D>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e = (block_size == kBlk) ? cudaLaunchKernelEx(&cfg, decode_split_kernel<D, true>, tk, tv, a)
                                       : cudaLaunchKernelEx(&cfg, decode_split_kernel<D, false>, tk, tv, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  if (a.direct) return launch_status();
  cfg.gridDim = dim3(ceil_div(static_cast<long long>(B) * Hq, 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  if (cudaLaunchKernelEx(&cfg, decode_combine_kernel<D>, a) != cudaSuccess) {
    cudaGetLastError();
    return FA_ERR_CUDA;
  }
  return launch_status();
}
}  // namespace

fa_status decode_launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                        const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d, int block_size,
                        int max_blocks, int num_blocks, int num_splits, float scale, void* workspace,
                        cudaStream_t stream) {
  if (block_size < kBlk || block_size % kBlk != 0) return FA_ERR_UNSUPPORTED;
  if (d == 128)
    return decode_launch_d<128>(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, block_size,
                                max_blocks, num_blocks, num_splits, scale, workspace, stream);
  if (d == 64)
    return decode_launch_d<64>(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, block_size,
                               max_blocks, num_blocks, num_splits, scale, workspace, stream);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa

// ---------------------------------------------------------------------------
// Paged decode without a caller workspace.
//
// Some callers cannot call cudaMalloc at the point where they decode: an
// inference-engine plugin whose device memory is handed out by the engine at
// build time and which may not allocate while enqueuing work, or a serving
// loop that must not allocate because cudaMalloc/cudaFree can synchronise the
// device and stall every other stream.  Such callers cannot pass the split
// workspace fa_paged_decode needs, so this variant keeps the split partials in
// a fixed file-scope device array.
//
// Capacity: B * Hq * num_splits <= kNoAllocMaxStates partial states at d = 128
// (fp32 o [states, 128] followed by fp32 (m, l) [states, 2]: 16.25 MiB).  Every
// device that loads the library holds one copy of the array until the process
// exits.  All calls on a device share it and it keeps the last call's
// contents; nothing in it needs to start at zero, because the split kernel
// writes every partial state that the combine kernel later reads.  Calls that
// overlap on the GPU (different streams, or different host threads without
// ordering) race on the array.
namespace fa {
namespace {

constexpr size_t kNoAllocMaxStates = 32768;
static __device__ __align__(256) float g_decode_scratch[kNoAllocMaxStates * (kDMax + 2)];

std::mutex g_scratch_mu;
float* g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the host-side symbol is only a stand-in, not a device address).
// The lookup is not made while `stream` is being captured into a graph: the
// call then returns nullptr (FA_ERR_CUDA to the caller) and leaves the capture
// untouched.
float* decode_scratch_ptr(cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  return g_scratch_ptr[dev];
}

}  // namespace

bool arm_decode_stall(long long cta, unsigned long long timeout_ns) {
#ifdef FA_DEBUG
  g_dec_stall_cta = cta;
  g_dec_stall_timeout_ns = timeout_ns;
  return true;
#else
  (void)cta;
  (void)timeout_ns;
  return false;
#endif
}
}  // namespace fa

extern "C" int fa_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                       const int32_t* block_table, const int32_t* seq_lens, void* o, float* lse, int B,
                                       int Hq, int Hkv, int d, int block_size, int max_blocks, int num_blocks,
                                       int num_splits, float scale, void* stream) {
  const fa_status st = fa::decode_check_args(q, k_cache, v_cache, block_table, seq_lens, o, B, Hq, Hkv, d,
                                             block_size, max_blocks, num_blocks, num_splits, scale);
  if (st != FA_OK) return st;
  const int S = num_splits == 0 ? 16 : num_splits;
  if (static_cast<size_t>(B) * Hq * S > fa::kNoAllocMaxStates) return FA_ERR_UNSUPPORTED;  // scratch too small
  float* scratch = fa::decode_scratch_ptr(static_cast<cudaStream_t>(stream));
  if (scratch == nullptr) return FA_ERR_CUDA;
  return fa::decode_launch(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, d, block_size, max_blocks,
                           num_blocks, S, scale, scratch, static_cast<cudaStream_t>(stream));
}
