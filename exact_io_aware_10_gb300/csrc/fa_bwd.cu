// Backward attention by recomputation on sm_103a ("精读笔记 08：FlashAttention"
// §3.3: keep O and the row statistics, rebuild the score tiles on chip; the
// IO-explained page: recomputation trades extra FLOPs for fewer HBM accesses).  With P recomputed as
// P = exp(scale Q K^T - LSE), the gradients of sum(dO * O) are
//     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
//     dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches on one stream:
//  1. bwd_pre_kernel   -D_i = -sum_c dO_ic O_ic and -LSE_i * log2(e) into padded
//                      fp32 rows (0 / -inf past N), and dQacc <- 0.
//  2. bwd_main_kernel  one CTA per (128-key tile j, batch*head); the grid runs
//                      over groups of four heads so the CTAs in flight share a
//                      few heads' Q, dO and dQ accumulator in L2.  K_j and V_j stay in shared
//                      memory; the CTA streams the query tiles i that see
//                      tile j and, per tile, runs five tcgen05 MMAs with fp32
//                      accumulators in TMEM:
//                        S^T  = K_j Q_i^T          (TMEM cols   0..127)
//                        dP^T = V_j dO_i^T         (TMEM cols 128..255)
//                        dV_j += P^T dO_i          (A = P^T, bf16 in TMEM over S^T)
//                        dK_j += dS^T Q_i          (A = dS^T: d = 128 bf16 in TMEM next
//                                                   to P^T, d = 64 from shared memory)
//                        dQ_i^T = K_j^T dS^T       (d = 128: lanes = head dim, over dP^T)
//                        dQ_i   = dS K_j           (d = 64: lanes = queries, over dP^T)
//                      MMA order per tile: dV_i, dQ_i, dK_i, S_{i+1}, dP_{i+1}:
//                      dQ_i is read out as soon as it is done (at d = 128 it is
//                      the only reader of the shared-memory dS^T, so its
//                      completion also frees that buffer for dQ staging), and
//                      the next tile's scores run while dQ_i is staged.
//                      dQ_i is added into the fp32 accumulator in L2 by TMA
//                      bulk reductions of boxes staged in shared memory: at
//                      d = 128 one 128 x 32 box per compute warpgroup, at
//                      d = 64 two swizzled 32 x 32 boxes per TMEM lane quarter.
//  3. bwd_dq_kernel    dQ = bf16(dQacc).
//
// Roles of the main kernel (20 warps = 5 warpgroups): warps 0-15 compute
// (thread = key row of S^T / dP^T / dK / dV; warpgroup h takes query columns
// 32h..32h+31 and head-dim columns h*d/4.. of dK/dV), warp 16 loads (TMA),
// warp 17 issues the MMAs, warp 18 folds the next query tile's load
// into the dS barrier (Q watcher), warp 19 idle; the fifth warpgroup hands
// registers to the compute warps.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kThreads = 640;
constexpr uint32_t kRegsCompute = 96;  // 4 x 128 x 96 + 128 x 96 = 640 x 96 (the launch pool)
constexpr uint32_t kRegsOther = 96;
constexpr int kTile = 128;  // keys per CTA and queries per step
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int kSub = D / 64;
  static constexpr int kSubBytes = kTile * 128;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kPBytes = kTile * kTile * 2;
  static constexpr int kSlots = 3;  // Q_i, Q_{i+1} and dO_i tiles
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  static constexpr int kOffP = kOffV + kTileBytes;  // dS^T (bf16, 128 x 128)
  static constexpr int kOffRing = kOffP + kPBytes;  // Q slots 0-1, then the dO slot
  // dQ staging for the TMA reductions.  d = 128: 16 KB (32 queries x 128 fp32)
  // per compute warpgroup, warpgroups 0-1 here, 2-3 in the dS^T buffer (idle
  // while dQ is read out).  d = 64: 8 KB (32 queries x 64 fp32) per TMEM lane
  // quarter, as two 128-byte-swizzled halves of 32 columns.
  static constexpr int kOffStage = kOffRing + kSlots * kTileBytes;
  static constexpr int kStageBytes = (D == 128) ? 2 * 16384 : 4 * 8192;
  static constexpr int kOffSide = kOffStage + kStageBytes;  // 2 x (-LSE2[128], -D[128])
  static constexpr int kOffBar = kOffSide + 2 * 1024;
  static constexpr int kUsedBytes = kOffBar + 256;
  static constexpr int kSmemBytes = (kUsedBytes + 1024 <= 232448) ? kUsedBytes + 1024 : 232448;
  static constexpr int kMaxPad = kSmemBytes - kUsedBytes;  // alignment padding the allocation can absorb
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D, kColDQ = 128;
};

enum : int {
  BAR_KV = 0,
  BAR_Q_FULL = 1,   // + slot (2)
  BAR_DO_FULL = 3,
  BAR_Q_EMPTY = 4,  // + slot (2)
  BAR_DO_EMPTY = 6,
  BAR_SIDE_FULL = 7,   // + 2
  BAR_SIDE_EMPTY = 9,  // + 2
  BAR_S = 11,
  BAR_P = 12,
  BAR_DP = 13,
  BAR_DS = 14,
  BAR_DQ_FULL = 15,
  BAR_DQ_READ = 16,
  BAR_FINAL = 17,
  BAR_DRAIN = 18,
  kNumBars = 19,
};
constexpr int kOffTmemSlot = kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kComputeWarps = 16;
// warp 18 folds the wait for the next query tile into the dS barrier
// (measured: 2 % faster at d = 128; at d = 64 2 % slower while dQ went out as
// per-thread reductions, 1.4-2.3 % faster with the staged TMA reductions)
template <int D>
constexpr bool kQWatch = true;
constexpr int kHeadGroup = 4;  // heads whose CTAs are interleaved in the grid

struct BwdArgs {
  float* Dpad;      // [BH, Npad] -D, 0 past N
  float* Lpad;      // [BH, Npad] -LSE * log2(e), -inf past N
  float* dQacc;     // [BH, N, D] fp32
  void* dK;         // [BH, N, D] bf16
  void* dV;
  const int32_t* kv_lens;
  int H, BH, N, Npad, nq;
  int causal;
  float scale;
  float scale_log2;
  unsigned* status;
  // packed ragged batch (nullptr: dense): Q/K/V/O/dO/dQ/dK/dV and dQacc are
  // [total, H, D], LSE is [H, total]; "batch entry" b is sequence b, rows
  // cu_seqlens[b] .. cu_seqlens[b+1]-1, and N is the longest sequence.  Kept
  // last: the dense kernel's register allocation is sensitive to the layout.
  const int32_t* cu_seqlens;
  int total;
};

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > 50000000ull) break;
  }
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Rows of sequence b in a packed batch: [tok0, tok0 + len).  The offsets must
// be non-decreasing, start at 0, end at total, and no sequence may be longer
// than N (the longest sequence the launch was sized for); otherwise len = -1.
__device__ __forceinline__ int packed_range(const BwdArgs& a, int b, int& tok0) {
  tok0 = a.cu_seqlens[b];
  const int tok1 = a.cu_seqlens[b + 1];
  const int nseq = a.BH / a.H;
  if (tok0 < 0 || tok1 < tok0 || tok1 > a.total || tok1 - tok0 > a.N || (b == 0 && tok0 != 0) ||
      (b == nseq - 1 && tok1 != a.total))
    return -1;
  return tok1 - tok0;
}

// --------------------------------------------------------------------------- 1. preprocess
// -D = -rowsum(dO * O) in fp32, -LSE in log2 units, dQacc row = 0.  A row is
// read by D / 8 lanes with 16-byte loads (16 lanes at d = 128, 8 at d = 64),
// so one warp covers 32 / (D / 8) rows; the partial sums are combined by
// shuffles within each row's lanes.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ O,
                                                      const __nv_bfloat16* __restrict__ dO,
                                                      const float* __restrict__ LSE, BwdArgs a, int BH) {
  constexpr int kLanesPerRow = D / 8;               // 16-byte chunks of a bf16 row
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;  // 2 (d = 128) or 4 (d = 64)
  const int lane = threadIdx.x & 31;
  const int sub = lane % kLanesPerRow;
  const long long gw = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const long long gr = gw * kRowsPerWarp + lane / kLanesPerRow;  // row over [BH, Npad]
  const long long rows = static_cast<long long>(BH) * a.Npad;
  const bool have = gr < rows;
  const int bh = have ? static_cast<int>(gr / a.Npad) : 0;
  const int r = have ? static_cast<int>(gr % a.Npad) : 0;
  int len = a.N;
  int tok0 = 0;
  if (a.cu_seqlens != nullptr && have) {
    len = packed_range(a, bh / a.H, tok0);
    if (len < 0) {
      if (r == 0 && sub == 0) atomicOr(a.status, kStatusBadArgBit);
      len = 0;
    }
  }
  const bool live = have && r < len;
  float acc = 0.f;
  size_t row = 0;
  if (live) {
    // [B, H, N, D] rows, or [total, H, D] rows when packed (LSE [H, total])
    row = a.cu_seqlens != nullptr ? static_cast<size_t>(tok0 + r) * a.H + bh % a.H
                                  : static_cast<size_t>(bh) * a.N + r;
    const uint4 o = *reinterpret_cast<const uint4*>(O + row * D + 8 * sub);
    const uint4 g = *reinterpret_cast<const uint4*>(dO + row * D + 8 * sub);
    const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&o);
    const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 of = __bfloat1622float2(o2[i]);
      const float2 gf = __bfloat1622float2(g2[i]);
      acc = fmaf(of.x, gf.x, acc);
      acc = fmaf(of.y, gf.y, acc);
    }
    float4* q = reinterpret_cast<float4*>(a.dQacc + row * D + 8 * sub);
    q[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    q[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (have && sub == 0) {
    if (live) {
      const size_t lrow = a.cu_seqlens != nullptr ? static_cast<size_t>(bh % a.H) * a.total + tok0 + r : row;
      a.Dpad[gr] = -acc;
      a.Lpad[gr] = -LSE[lrow] * kLog2e;
    } else {
      a.Dpad[gr] = 0.f;
      a.Lpad[gr] = -INFINITY;
    }
  }
}

// --------------------------------------------------------------------------- 3. dQ convert
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float* __restrict__ dQacc, __nv_bfloat16* __restrict__ dQ,
                                                     long long n4) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 v = reinterpret_cast<const float4*>(dQacc)[i];
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  reinterpret_cast<uint2*>(dQ)[i] = w;
}

// --------------------------------------------------------------------------- 2. main
// kPacked selects the packed ragged-batch layout at compile time, so the dense
// instantiation carries none of its indexing.
template <int D, bool kPacked>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  {
    // the tiles need a 1024-byte aligned base; refuse (and report) rather than overrun
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad > static_cast<uint32_t>(C::kMaxPad)) {
      if (threadIdx.x == 0) atomicOr(a.status, kStatusLaunchBit);
      return;
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t barbase = sbase + C::kOffBar;
  auto bar = [&](int i) -> uint32_t { return barbase + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // grid: y = group of kHeadGroup heads, x = key tile * kHeadGroup + head in
  // group: the CTAs in flight share a few heads' Q, dO and dQ accumulator in L2,
  // and within a group the key tiles with most query tiles (causal) start first
  const int bh = blockIdx.y * kHeadGroup + static_cast<int>(blockIdx.x % kHeadGroup);
  if (bh >= a.BH) return;
  const int b = bh / a.H;
  const int j = static_cast<int>(blockIdx.x / kHeadGroup);
  const int head = bh % a.H;
  // N = rows of this batch entry (dense) or sequence (packed); tok0 = its first token
  int n_rows = a.N, tok0 = 0;
  if constexpr (kPacked) {
    n_rows = packed_range(a, b, tok0);
    if (n_rows < 0 || j * kTile >= n_rows) return;  // bad offsets (reported by the preprocess) or past the end
  }
  const int N = n_rows;
  int kv_len = N;
  if (a.kv_lens != nullptr) kv_len = min(max(a.kv_lens[b], 0), N);
  const bool live = j * kTile < kv_len;  // any unmasked key in this tile
  const int i0 = a.causal ? j : 0;
  const int nq = kPacked ? (N + kTile - 1) / kTile : a.nq;
  const int nt = live ? (nq - i0) : 0;  // query tiles to visit
  // TMA coordinates (y, z) of 128 rows from `row`: dense maps are (d, N, B*H)
  // -> (row, bh), packed maps (d, H, total) -> (head, tok0 + row)
#define BWD_CRD(row) (kPacked ? head : (row)), (kPacked ? tok0 + (row) : bh)

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_Q_FULL + s), 1);
      mbar_init(bar(BAR_Q_EMPTY + s), 1);
      mbar_init(bar(BAR_SIDE_FULL + s), 1);
      mbar_init(bar(BAR_SIDE_EMPTY + s), kComputeWarps);
    }
    mbar_init(bar(BAR_DO_FULL), 1);
    mbar_init(bar(BAR_DO_EMPTY), 1);
    mbar_init(bar(BAR_S), 1);
    mbar_init(bar(BAR_P), kComputeWarps);
    mbar_init(bar(BAR_DP), 1);
    mbar_init(bar(BAR_DS), kComputeWarps + (kQWatch<D> ? 1 : 0));  // + the Q watcher
    mbar_init(bar(BAR_DQ_FULL), 1);
    mbar_init(bar(BAR_DQ_READ), kComputeWarps);
    mbar_init(bar(BAR_FINAL), 1);
    mbar_init(bar(BAR_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, a.status};
  const size_t side_row = static_cast<size_t>(bh) * a.Npad;

  if (warp >= kComputeWarps) {
    regs_dealloc<kRegsOther>();
    if (warp == kComputeWarps) {
      // ---------------------------------------------------------- producer
      if (lane == 0 && nt > 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdO);
        mbar_arrive_expect_tx(bar(BAR_KV), 2 * C::kTileBytes);
        for (int s = 0; s < C::kSub; ++s) {
          tma_load_3d(sbase + C::kOffK + s * C::kSubBytes, &tmK, bar(BAR_KV), s * 64, BWD_CRD(j * kTile));
          tma_load_3d(sbase + C::kOffV + s * C::kSubBytes, &tmV, bar(BAR_KV), s * 64, BWD_CRD(j * kTile));
        }
        int side_issued = 0, q_issued = 0, o_issued = 0;
        for (int it = 0; it < nt; ++it) {
          const int i = i0 + it;
          const int sd = it & 1;
          if (!mbar_wait(bar(BAR_SIDE_EMPTY + sd), ((it >> 1) & 1) ^ 1, wc)) break;
          mbar_arrive_expect_tx(bar(BAR_SIDE_FULL + sd), 1024);
          bulk_load(sbase + C::kOffSide + sd * 1024, a.Lpad + side_row + i * kTile, 512, bar(BAR_SIDE_FULL + sd));
          bulk_load(sbase + C::kOffSide + sd * 1024 + 512, a.Dpad + side_row + i * kTile, 512,
                    bar(BAR_SIDE_FULL + sd));
          side_issued = it + 1;
          // Q_i into Q slot it % 2 (free once dK of tile it-2 is done)
          if (!mbar_wait(bar(BAR_Q_EMPTY + sd), ((it >> 1) & 1) ^ 1, wc)) break;
          mbar_arrive_expect_tx(bar(BAR_Q_FULL + sd), C::kTileBytes);
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d(sbase + C::kOffRing + sd * C::kTileBytes + s * C::kSubBytes, &tmQ, bar(BAR_Q_FULL + sd),
                        s * 64, BWD_CRD(i * kTile));
          q_issued = it + 1;
          // dO_i into the dO slot (free once dV of tile it-1 is done)
          if (!mbar_wait(bar(BAR_DO_EMPTY), (it & 1) ^ 1, wc)) break;
          mbar_arrive_expect_tx(bar(BAR_DO_FULL), C::kTileBytes);
          for (int s = 0; s < C::kSub; ++s)
            tma_load_3d(sbase + C::kOffRing + 2 * C::kTileBytes + s * C::kSubBytes, &tmdO, bar(BAR_DO_FULL), s * 64,
                        BWD_CRD(i * kTile));
          o_issued = it + 1;
        }
        drain_wait(bar(BAR_KV), 0);
        for (int s = 0; s < 2 && s < q_issued; ++s) {
          const int it_last = s + 2 * ((q_issued - 1 - s) / 2);
          drain_wait(bar(BAR_Q_FULL + s), (it_last >> 1) & 1);
        }
        for (int s = 0; s < 2 && s < side_issued; ++s) {
          const int it_last = s + 2 * ((side_issued - 1 - s) / 2);
          drain_wait(bar(BAR_SIDE_FULL + s), (it_last >> 1) & 1);
        }
        if (o_issued > 0) drain_wait(bar(BAR_DO_FULL), (o_issued - 1) & 1);
      }
    } else if (warp == kComputeWarps + 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0 && nt > 0) {
        constexpr uint32_t idSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t idKN = idesc_bf16_f32(128, D, false, true);     // dV (TS), dK
        const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sP = sbase + C::kOffP;
        auto q_addr = [&](int it) { return sbase + C::kOffRing + (it & 1) * C::kTileBytes; };
        const uint32_t aO = sbase + C::kOffRing + 2 * C::kTileBytes;
        // Descriptors are built once per operand tile (K-major and MN-major views)
        // and advanced by immediates, so the issuing thread keeps the tensor pipe fed.
        const uint64_t kK = sdesc_sw128(sK, 16, 1024), kV = sdesc_sw128(sV, 16, 1024);
        const uint64_t kP = sdesc_sw128(sP, 16, 1024), kO = sdesc_sw128(aO, 16, 1024);
        const uint64_t mK = sdesc_sw128(sK, C::kSubBytes, 1024), mP = sdesc_sw128(sP, C::kSubBytes, 1024);
        const uint64_t mO = sdesc_sw128(aO, C::kSubBytes, 1024);
        const uint64_t kQ0 = sdesc_sw128(q_addr(0), 16, 1024), mQ0 = sdesc_sw128(q_addr(0), C::kSubBytes, 1024);
        auto kq = [&](int it) { return sdesc_advance(kQ0, (it & 1) * C::kTileBytes); };
        auto mq = [&](int it) { return sdesc_advance(mQ0, (it & 1) * C::kTileBytes); };
        // A and B both K-major, K extent = D (head dim)
        auto mma_kmajor_d = [&](uint32_t dcol, uint64_t da, uint64_t db) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::kSubBytes + (k & 3) * 32;
            mma_ss(tmem + dcol, sdesc_advance(da, off), sdesc_advance(db, off), idSS, k > 0 ? 1u : 0u);
          }
        };
        bool ok = mbar_wait(bar(BAR_KV), 0, wc);
        // prologue: S_0 and dP_0
        if (ok) ok = mbar_wait(bar(BAR_Q_FULL + 0), 0, wc);
        if (ok) {
          tc_fence_after();
          mma_kmajor_d(C::kColS, kK, kq(0));
          mma_commit(bar(BAR_S));
          ok = mbar_wait(bar(BAR_DO_FULL), 0, wc);
        }
        if (ok) {
          tc_fence_after();
          mma_kmajor_d(C::kColDP, kV, kO);
          mma_commit(bar(BAR_DP));
        }
        for (int it = 0; ok && it < nt; ++it) {
          const bool next = it + 1 < nt;
          // dV_j += P^T dO_i  (P^T packed bf16 in TMEM: warpgroup h's 32 queries in cols 32h..32h+15)
          if (!(ok = mbar_wait(bar(BAR_P), it & 1, wc))) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            const uint32_t acol = 32 * (k >> 1) + 8 * (k & 1);
            mma_ts(tmem + C::kColDV, tmem + C::kColS + acol, sdesc_advance(mO, k * 2048), idKN,
                   (it > 0 || k > 0) ? 1u : 0u);
          }
          mma_commit(bar(BAR_DO_EMPTY));
          // dK_j += dS^T Q_i  and  dQ_i over the dP^T columns
          if (!(ok = mbar_wait(bar(BAR_DS), it & 1, wc))) break;
          tc_fence_after();
          auto issue_dk = [&]() {
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k) {
              const uint32_t aoff = (k >> 2) * C::kSubBytes + (k & 3) * 32;
              mma_ss(tmem + C::kColDK, sdesc_advance(kP, aoff), sdesc_advance(mq(it), k * 2048), idKN,
                     (it > 0 || k > 0) ? 1u : 0u);
            }
          };
          if constexpr (D == 128) {
            // dQ_i first: it is the only reader of the shared-memory dS^T, so
            // DQ_FULL also frees that buffer for dQ staging; then dK_i with
            // A = dS^T from TMEM (packed bf16 next to P^T, as for dV)
            constexpr uint32_t idQT = idesc_bf16_f32(128, 128, true, true);  // A = K^T, B = dS^T
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k)
              mma_ss(tmem + C::kColDQ, sdesc_advance(mK, k * 2048), sdesc_advance(mP, k * 2048), idQT,
                     k > 0 ? 1u : 0u);
            mma_commit(bar(BAR_DQ_FULL));
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k) {
              const uint32_t acol = 32 * (k >> 1) + 16 + 8 * (k & 1);
              mma_ts(tmem + C::kColDK, tmem + C::kColS + acol, sdesc_advance(mq(it), k * 2048), idKN,
                     (it > 0 || k > 0) ? 1u : 0u);
            }
          } else {
            // d = 64: dQ first, so its read-out and staged reductions (own
            // staging buffer, not the dS^T one) start while dK runs
            constexpr uint32_t idNN = idesc_bf16_f32(128, D, true, true);  // A = dS, B = K
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k)
              mma_ss(tmem + C::kColDQ, sdesc_advance(mP, k * 2048), sdesc_advance(mK, k * 2048), idNN,
                     k > 0 ? 1u : 0u);
            mma_commit(bar(BAR_DQ_FULL));
            issue_dk();
          }
          mma_commit(bar(BAR_Q_EMPTY + (it & 1)));
          // S_{i+1} = K_j Q_{i+1}^T over the S^T columns (after dV has read P^T).
          // Issued behind dK_i and dQ_i, so dQ_i reaches the compute warps (which
          // read it out next) without waiting for S_{i+1}.
          if (next) {
            // with the watcher: Q_i+1 has landed, the DS(i) barrier waited for above
            // completes only after the Q watcher has seen it
            if (!kQWatch<D> &&
                !(ok = mbar_wait(bar(BAR_Q_FULL + ((it + 1) & 1)), ((it + 1) >> 1) & 1, wc)))
              break;
            if (!kQWatch<D>) tc_fence_after();
            mma_kmajor_d(C::kColS, kK, kq(it + 1));
            mma_commit(bar(BAR_S));
          }
          // dP_{i+1} = V_j dO_{i+1}^T over the dP^T columns (after dQ_i has been read out)
          if (next) {
            if (!(ok = mbar_wait(bar(BAR_DO_FULL), (it + 1) & 1, wc))) break;
            if (!(ok = mbar_wait(bar(BAR_DQ_READ), it & 1, wc))) break;
            tc_fence_after();
            mma_kmajor_d(C::kColDP, kV, kO);
            mma_commit(bar(BAR_DP));
          }
        }
        if (ok) mma_commit(bar(BAR_FINAL));
        mma_commit(bar(BAR_DRAIN));
        drain_wait(bar(BAR_DRAIN), 0);
      }
    } else if (kQWatch<D> && warp == kComputeWarps + 2) {
      // ---------------------------------------------------------- Q watcher
      // Adds one arrival to DS(i), after Q_i+1 has landed, so the issuing
      // thread's wait for dS_i also covers the next query tile (one barrier
      // wait fewer per tile on the issuing thread).  It arrives for tile i only
      // once DS(i - 1) has completed, so it never arrives twice in one phase.
      if (lane == 0) {
        for (int it = 0; it < nt; ++it) {
          if (it > 0 && !mbar_wait(bar(BAR_DS), static_cast<uint32_t>(it - 1) & 1u, wc)) break;
          if (it + 1 < nt &&
              !mbar_wait(bar(BAR_Q_FULL + ((it + 1) & 1)), static_cast<uint32_t>((it + 1) >> 1) & 1u, wc))
            break;
          mbar_arrive(bar(BAR_DS));
        }
      }
    }
  } else {
    regs_alloc<kRegsCompute>();
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;  // warpgroup: query columns 32 grp .. 32 grp + 31
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // key row (S^T, dP^T, dK, dV); head-dim row of dQ^T (d = 128)
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int key = j * kTile + r;
    const bool key_ok = key < kv_len;
    // this thread's 32 query columns of dS^T: sub-tile grp / 2, 16-byte chunks 4 (grp & 1) .. +3
    const uint32_t dsrow = sbase + C::kOffP + (grp >> 1) * C::kSubBytes + r * 128;
    const int swz = r & 7;
    const float2 sl2v = make_float2(a.scale_log2, a.scale_log2);
    const float2 scv = make_float2(a.scale, a.scale);
    bool aborted = false;
    for (int it = 0; it < nt; ++it) {
      const int i = i0 + it;
      const int sd = it & 1;
      if (!mbar_wait(bar(BAR_SIDE_FULL + sd), (it >> 1) & 1, wc) || !mbar_wait(bar(BAR_S), it & 1, wc)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const float* nlse2 = reinterpret_cast<const float*>(smem + C::kOffSide + sd * 1024) + grp * 32;  // -LSE2
      const float* ndsum = nlse2 + 128;                                                                // -D
      // ---- P^T = exp2(S^T * scale * log2e - LSE2[q]) on this thread's 32 query columns
      float p[32];
      {
        uint32_t sv[32];
        tmem_ld32(tmem + lane_off + C::kColS + grp * 32, sv);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(nlse2 + c);
          const float2 x0 = ffma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2v,
                                  make_float2(l4.x, l4.y));
          const float2 x1 = ffma2(make_float2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2v,
                                  make_float2(l4.z, l4.w));
          p[c + 0] = ex2_approx(x0.x);
          p[c + 1] = ex2_approx(x0.y);
          p[c + 2] = ex2_approx(x1.x);
          p[c + 3] = ex2_approx(x1.y);
        }
        // causal: key > query is masked; queries past N have -LSE2 = -inf -> 0
        const int qlo = i * kTile + grp * 32;
        const int first_vis = a.causal ? (key - qlo) : 0;  // columns c >= first_vis are visible
        if (!key_ok || first_vis > 0) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (!key_ok || c < first_vis) p[c] = 0.f;
        }
      }
      {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(p[2 * c], p[2 * c + 1]);
        tmem_st16(tmem + lane_off + C::kColS + grp * 32, pk);  // over this thread's own S^T columns
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P));
      // ---- dS^T = scale * P^T * (dP^T - D[q])  -> shared memory (bf16)
      if (!mbar_wait(bar(BAR_DP), it & 1, wc)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      {
        uint32_t dv[32];
        tmem_ld32(tmem + lane_off + C::kColDP + grp * 32, dv);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(ndsum + c);
          const float2 g0 = fadd2(make_float2(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), make_float2(d4.x, d4.y));
          const float2 g1 =
              fadd2(make_float2(__uint_as_float(dv[c + 2]), __uint_as_float(dv[c + 3])), make_float2(d4.z, d4.w));
          const float2 ds0 = fmul2(fmul2(make_float2(p[c], p[c + 1]), scv), g0);
          const float2 ds1 = fmul2(fmul2(make_float2(p[c + 2], p[c + 3]), scv), g1);
          p[c] = ds0.x;
          p[c + 1] = ds0.y;
          p[c + 2] = ds1.x;
          p[c + 3] = ds1.y;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_SIDE_EMPTY + sd));
      if constexpr (D == 128) {
        // the previous tile's dQ reductions of warpgroups 2-3 read staging inside
        // the dS^T buffer: their reads must be done before any warp overwrites it
        if (it > 0) {
          if (grp >= 2 && q4 == 0 && lane == 0) bulk_wait_read_all();
          named_barrier_sync(1, 32 * kComputeWarps);
        }
      }
      // d = 128: dS^T also goes to TMEM, next to P^T (columns 32 grp + 16 ..):
      // dK_i reads it from there, so only dQ_i reads the shared-memory copy
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) pk[c] = pack_bf16x2(p[16 * h + 2 * c], p[16 * h + 2 * c + 1]);
        if constexpr (D == 128) tmem_st8(tmem + lane_off + C::kColS + grp * 32 + 16 + 8 * h, pk);
#pragma unroll
        for (int c8 = 0; c8 < 2; ++c8) {
          const int chunk = 4 * (grp & 1) + 2 * h + c8;
          st_shared_v4(dsrow + (((chunk ^ swz)) << 4), pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2], pk[4 * c8 + 3]);
        }
      }
      if constexpr (D == 128) tmem_st_wait();
      fence_proxy_async_smem();
      if constexpr (D == 128) tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_DS));
      // ---- dQ_i += this tile's contribution
      if (!mbar_wait(bar(BAR_DQ_FULL), it & 1, wc)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      if constexpr (D == 128) {
        // dQ^T: lane = head-dim index r, columns = this warpgroup's 32 queries.
        // The TMEM columns are released as soon as the values are in registers;
        // the warpgroup then stages its 32 x 128 fp32 box (row-major) and one
        // thread adds it into dQacc with a TMA reduction in L2.
        uint32_t rr[32];
        tmem_ld32(tmem + lane_off + C::kColDQ + grp * 32, rr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_DQ_READ));
        const int q0 = i * kTile + grp * 32;
        const uint32_t stg = (grp < 2) ? sbase + C::kOffStage + grp * 16384 : sbase + C::kOffP + (grp - 2) * 16384;
        const bool leader = (q4 == 0 && lane == 0);
        if (grp < 2 && it > 0 && leader) bulk_wait_read_all();  // this staging slot's previous reduction
        named_barrier_sync(2 + grp, 128);
#pragma unroll
        for (int q = 0; q < 32; ++q) st_shared_f32(stg + q * 512 + r * 4, __uint_as_float(rr[q]));
        fence_proxy_async_smem();
        named_barrier_sync(2 + grp, 128);
        if (leader && q0 < N) {
          // rows past a packed sequence carry exact zeros (their P is 0)
          tma_reduce_add_3d(&tmdQ, stg, 0, BWD_CRD(q0));
          bulk_commit();
        }
        continue;  // DQ_READ already signalled
      } else {
        // dQ: lane = query row r, columns = this warpgroup's 16 head-dim
        // entries.  The four warps of one TMEM lane quarter (q4, one per
        // warpgroup) stage their 32 queries x 64 fp32 in shared memory, two
        // 128-byte-swizzled halves of 32 columns (conflict-free 16-byte
        // stores), and one of them adds the box into dQacc with two TMA
        // reductions in L2.
        uint32_t rr[16];
        tmem_ld16(tmem + lane_off + C::kColDQ + grp * 16, rr);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_DQ_READ));
        const uint32_t stg = sbase + C::kOffStage + q4 * 8192;
        const bool leader = (grp == 0 && lane == 0);
        if (it > 0 && leader) bulk_wait_read_all();  // this staging box's previous reductions
        named_barrier_sync(2 + q4, 128);
        const uint32_t srow = stg + (grp >> 1) * 4096 + lane * 128;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(srow + ((((grp & 1) * 4 + c) ^ (lane & 7)) << 4), rr[4 * c], rr[4 * c + 1], rr[4 * c + 2],
                       rr[4 * c + 3]);
        fence_proxy_async_smem();
        named_barrier_sync(2 + q4, 128);
        const int q0 = i * kTile + q4 * 32;
        if (leader && q0 < N) {
          // rows past a packed sequence carry exact zeros (their P is 0)
          tma_reduce_add_3d(&tmdQ, stg, 0, BWD_CRD(q0));
          tma_reduce_add_3d(&tmdQ, stg + 4096, 32, BWD_CRD(q0));
          bulk_commit();
        }
        continue;  // DQ_READ already signalled
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_DQ_READ));
    }
    if (lane == 0) bulk_wait_read_all();  // staging must outlive the reductions' reads
    // ---- epilogue: dV_j, dK_j rows (thread = key row r), head-dim columns of this warpgroup
    if (!aborted) {
      const bool have = nt > 0;
      if (have && !mbar_wait(bar(BAR_FINAL), 0, wc)) aborted = true;
      if (!aborted) {
        tc_fence_after();
        constexpr int kCols = D / 4;
        const bool in_range = key < N;
        const size_t krow = kPacked ? static_cast<size_t>(tok0 + key) * a.H + head : static_cast<size_t>(bh) * N + key;
        const size_t rowoff = krow * D + grp * kCols;
#pragma unroll
        for (int which = 0; which < 2; ++which) {
          uint8_t* out = static_cast<uint8_t*>(which ? a.dK : a.dV) + rowoff * 2;
          const uint32_t col = (which ? C::kColDK : C::kColDV) + grp * kCols;
          uint32_t rr[kCols];
          if (have) {
            if constexpr (kCols == 32) {
              tmem_ld32(tmem + lane_off + col, rr);
            } else {
              tmem_ld16(tmem + lane_off + col, rr);
            }
          } else {
#pragma unroll
            for (int c = 0; c < kCols; ++c) rr[c] = 0u;
          }
          if (in_range) {
            uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
            for (int q = 0; q < kCols / 8; ++q)
              dst[q] = make_uint4(pack_bf16x2(__uint_as_float(rr[8 * q + 0]), __uint_as_float(rr[8 * q + 1])),
                                  pack_bf16x2(__uint_as_float(rr[8 * q + 2]), __uint_as_float(rr[8 * q + 3])),
                                  pack_bf16x2(__uint_as_float(rr[8 * q + 4]), __uint_as_float(rr[8 * q + 5])),
                                  pack_bf16x2(__uint_as_float(rr[8 * q + 6]), __uint_as_float(rr[8 * q + 7])));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}
#undef BWD_CRD

template <int D>
fa_status bwd_launch_d(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, int B, int H, int N, int causal, float scale,
                       const int32_t* kv_lens, void* workspace, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int BH = B * H;
  const int nq = ceil_div(N, kTile);
  const int Npad = nq * kTile;
  const size_t side = (static_cast<size_t>(BH) * Npad * sizeof(float) + 255) & ~static_cast<size_t>(255);
  BwdArgs a;
  a.Dpad = static_cast<float*>(workspace);
  a.Lpad = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + side);
  a.dQacc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 2 * side);
  a.dK = dK;
  a.dV = dV;
  a.kv_lens = kv_lens;
  a.cu_seqlens = nullptr;
  a.total = 0;
  a.H = H;
  a.BH = BH;
  a.N = N;
  a.Npad = Npad;
  a.nq = nq;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.status = device_status_ptr();
  if (a.status == nullptr) return FA_ERR_CUDA;

  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(N) * D * 2};
  const uint32_t box[3] = {64, kTile, 1};
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!encode_bf16_tmap(&tq, Q, 3, dims, strides, box) || !encode_bf16_tmap(&tk, K, 3, dims, strides, box) ||
      !encode_bf16_tmap(&tv, V, 3, dims, strides, box) || !encode_bf16_tmap(&tdo, dO, 3, dims, strides, box))
    return FA_ERR_CUDA;
  // fp32 dQ accumulator as head-dim x 32-query boxes for the TMA reductions:
  // d = 128 one plain 128-column box, d = 64 two 128-byte-swizzled 32-column boxes
  const uint64_t qstrides[2] = {static_cast<uint64_t>(D) * 4, static_cast<uint64_t>(N) * D * 4};
  const uint32_t qbox[3] = {D == 128 ? 128u : 32u, 32, 1};
  if (!(D == 128 ? encode_f32_tmap(&tdq, a.dQacc, 3, dims, qstrides, qbox)
                 : encode_f32_sw128_tmap(&tdq, a.dQacc, 3, dims, qstrides, qbox)))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&bwd_main_kernel<D, false>), C::kSmemBytes))
    return FA_ERR_CUDA;
  const long long pre_rows = static_cast<long long>(BH) * Npad;
  bwd_pre_kernel<D><<<static_cast<unsigned>((pre_rows + 8 * (256 / D) - 1) / (8 * (256 / D))), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, a, BH);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const dim3 grid(nq * kHeadGroup, ceil_div(BH, kHeadGroup));
  bwd_main_kernel<D, false><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const long long n4 = static_cast<long long>(BH) * N * D / 4;
  bwd_dq_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(a.dQacc,
                                                                             static_cast<__nv_bfloat16*>(dQ), n4);
  return launch_status();
}

template <int D>
fa_status bwd_varlen_launch_d(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                              const float* LSE, void* dQ, void* dK, void* dV, const int32_t* cu_seqlens, int num_seqs,
                              int total, int max_seqlen, int H, int causal, float scale, void* workspace,
                              cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int BH = num_seqs * H;
  const int nq = ceil_div(max_seqlen, kTile);
  const int Npad = nq * kTile;
  const size_t side = (static_cast<size_t>(BH) * Npad * sizeof(float) + 255) & ~static_cast<size_t>(255);
  BwdArgs a;
  a.Dpad = static_cast<float*>(workspace);
  a.Lpad = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + side);
  a.dQacc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 2 * side);
  a.dK = dK;
  a.dV = dV;
  a.kv_lens = nullptr;
  a.cu_seqlens = cu_seqlens;
  a.total = total;
  a.H = H;
  a.BH = BH;
  a.N = max_seqlen;
  a.Npad = Npad;
  a.nq = nq;
  a.causal = causal ? 1 : 0;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.status = device_status_ptr();
  if (a.status == nullptr) return FA_ERR_CUDA;
  // packed [total, H, D]: TMA dims (D, H, total), 128 consecutive tokens of one head
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(H), static_cast<uint64_t>(total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(H) * D * 2};
  const uint32_t box[3] = {64, 1, kTile};
  CUtensorMap tq, tk, tv, tdo, tdq;
  if (!encode_bf16_tmap(&tq, Q, 3, dims, strides, box) || !encode_bf16_tmap(&tk, K, 3, dims, strides, box) ||
      !encode_bf16_tmap(&tv, V, 3, dims, strides, box) || !encode_bf16_tmap(&tdo, dO, 3, dims, strides, box))
    return FA_ERR_CUDA;
  const uint64_t qstrides[2] = {static_cast<uint64_t>(D) * 4, static_cast<uint64_t>(H) * D * 4};
  const uint32_t qbox[3] = {D == 128 ? 128u : 32u, 1, 32};
  if (!(D == 128 ? encode_f32_tmap(&tdq, a.dQacc, 3, dims, qstrides, qbox)
                 : encode_f32_sw128_tmap(&tdq, a.dQacc, 3, dims, qstrides, qbox)))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&bwd_main_kernel<D, true>), C::kSmemBytes))
    return FA_ERR_CUDA;
  const long long pre_rows = static_cast<long long>(BH) * Npad;
  bwd_pre_kernel<D><<<static_cast<unsigned>((pre_rows + 8 * (256 / D) - 1) / (8 * (256 / D))), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, a, BH);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const dim3 grid(nq * kHeadGroup, ceil_div(BH, kHeadGroup));
  bwd_main_kernel<D, true><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, tdo, tdq, a);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  const long long n4 = static_cast<long long>(total) * H * D / 4;
  bwd_dq_kernel<<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, stream>>>(a.dQacc,
                                                                             static_cast<__nv_bfloat16*>(dQ), n4);
  return launch_status();
}

}  // namespace

fa_status bwd_varlen_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                            const float* LSE, void* dQ, void* dK, void* dV, const int32_t* cu_seqlens, int num_seqs,
                            int total, int max_seqlen, int H, int d, int causal, float scale, void* workspace,
                            cudaStream_t stream) {
  if (d == 64)
    return bwd_varlen_launch_d<64>(Q, K, V, O, dO, LSE, dQ, dK, dV, cu_seqlens, num_seqs, total, max_seqlen, H,
                                   causal, scale, workspace, stream);
  if (d == 128)
    return bwd_varlen_launch_d<128>(Q, K, V, O, dO, LSE, dQ, dK, dV, cu_seqlens, num_seqs, total, max_seqlen, H,
                                    causal, scale, workspace, stream);
  return FA_ERR_UNSUPPORTED;
}

fa_status bwd_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                     void* dQ, void* dK, void* dV, int B, int H, int N, int d, int causal, float scale,
                     const int32_t* kv_lens, void* workspace, cudaStream_t stream) {
  if (d == 64) return bwd_launch_d<64>(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, causal, scale, kv_lens, workspace, stream);
  if (d == 128) return bwd_launch_d<128>(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, causal, scale, kv_lens, workspace, stream);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
