// Backward attention by recomputation on sm_103a ("精读笔记 08：FlashAttention"
// §3.3: keep O and the row statistics, rebuild the score tiles on chip; the
// IO-explained page: recomputation trades extra FLOPs for fewer HBM accesses).  With P recomputed as
// P = exp(scale Q K^T - LSE), the gradients of sum(dO * O) are
//     dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
//     dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches on one stream, the second and third as programmatic
// dependents of the one before (their launch and set-up overlap its tail;
// griddepcontrol.wait precedes every read of its results):
//  1. bwd_pre_kernel   -D_i = -sum_c dO_ic O_ic and -LSE_i * log2(e) into padded
//                      fp32 rows (0 / -inf past N), dQacc <- 0 and the main
//                      kernel's work counter <- 0.
//  2. bwd_main_kernel  one persistent CTA per SM; its work items are the
//                      (128-key tile j, batch*head) pairs, taken in order from a
//                      counter in the workspace: groups of heads (16, 8 or 4 by
//                      the L2 budget), within a group the key tiles with most
//                      query tiles first, so
//                      the items in flight share a few heads' Q, dO and dQ
//                      accumulator in L2.  K_j and V_j stay in shared
//                      memory (d = 64, short items: two K, V buffers, so the
//                      next item's load overlaps this one); the CTA streams the query tiles i that see
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
// 32h..32h+31 and head-dim columns h*d/4.. of dK/dV), warp 16 takes the work
// items from the counter and loads (TMA), warp 17 issues the MMAs, warp 18 folds the next query tile's load
// into the dS barrier (Q watcher), warp 19 idle; the fifth warpgroup hands
// registers to the compute warps.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include <utility>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kThreads = 640;
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
  // d = 64 has room for a second K, V pair: consecutive work items alternate
  // between the two, so the next item's K and V load while the current one runs
  static constexpr int kKVBufs = (D == 64) ? 2 : 1;
  static constexpr int kOffKV1 = (kOffBar + 256 + 1023) / 1024 * 1024;
  static constexpr int kUsedBytes = (kKVBufs == 2) ? kOffKV1 + 2 * kTileBytes : kOffBar + 256;
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
constexpr int kComputeWarps = 16;
constexpr int kAltMaxTiles = 8;  // d = 64: items of at most this many query tiles alternate K, V buffers
// warp 18 folds the wait for the next query tile into the dS barrier
// (measured: 2 % faster at d = 128; at d = 64 2 % slower while dQ went out as
// per-thread reductions, 1.4-2.3 % faster with the staged TMA reductions)
template <int D>
constexpr bool kQWatch = true;
// Heads whose work items are interleaved: the items in flight then share
// those heads' Q, dO and fp32 dQ accumulator (N d 8 bytes a head) in L2.  The
// largest of 16, 8 and 4 heads whose share fits kL2HeadBudget, well inside the
// 129 MB L2 (a share the size of L2 already doubles the main kernel's DRAM
// traffic through dQ reductions that miss it); 8 for the packed layout
// (measured best on the long ragged mix).
constexpr double kL2HeadBudget = 96.0 * 1024 * 1024;
inline int bwd_head_group(int N, int D, bool packed) {
  if (packed) return 8;
  for (int g = 16; g > 4; g /= 2)
    if (static_cast<double>(g) * N * D * 8.0 <= kL2HeadBudget) return g;
  return 4;
}
// register split of the main kernel: d = 64 gives the compute warps 104 (their
// item and tile state spills at 96), d = 128 keeps 96 / 96 (the issuing thread
// spills at 64)
template <int D>
constexpr uint32_t kRegsCompute = (D == 64) ? 104 : 96;
template <int D>
constexpr uint32_t kRegsOther = (D == 64) ? 64 : 96;  // 4 x 128 x compute + 128 x other <= 640 x 96 (the launch pool)

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
  // persistent main kernel: work-item counter (zeroed by the preprocess), the
  // number of items and the x extent of the item grid (key tiles x heads per group)
  unsigned* sched;
  int n_items, gx;
#ifdef FA_DEBUG
  // extents for the debug bounds checks: batch entries (sequences), rows of
  // Q/K/V/O/dO/dQ/dK/dV and dQacc (D elements each) and of LSE, elements of
  // each of the -D and -LSE2 row buffers
  int dbg_nb;
  long long dbg_rows, dbg_side;
  int dbg_stall_item;                   // the MMA warp stops before this work item (-1: never)
  unsigned long long dbg_timeout_ns;    // wait limit of this launch (0: the default)
#endif
};

#ifdef FA_DEBUG
// One-shot stall armed by fa_debug_stall_backward, taken by the next launch
// of the main kernel (host side, not thread-safe: a debug hook).
int g_stall_item = -1;
unsigned long long g_stall_timeout_ns = 0;
void take_backward_stall(BwdArgs& a) {
  a.dbg_stall_item = g_stall_item;
  a.dbg_timeout_ns = g_stall_timeout_ns;
  g_stall_item = -1;
  g_stall_timeout_ns = 0;
}
#endif

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
  tok0 = 0;
  if (!FA_IN_BOUNDS(b + 1, a.dbg_nb + 1, a.status)) return -1;
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
  // the main kernel (which waits for this grid's completion before it reads
  // anything written here) may be scheduled once every CTA has started
  griddep_launch_dependents();
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
  if (a.sched != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *a.sched = 0u;
  bool live = have && r < len;
  float acc = 0.f;
  size_t row = 0;
  if (live) {
    // [B, H, N, D] rows, or [total, H, D] rows when packed (LSE [H, total])
    row = a.cu_seqlens != nullptr ? static_cast<size_t>(tok0 + r) * a.H + bh % a.H
                                  : static_cast<size_t>(bh) * a.N + r;
    live = FA_IN_BOUNDS(static_cast<long long>(row), a.dbg_rows, a.status);
  }
  if (live) {
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
      a.Lpad[gr] = FA_IN_BOUNDS(static_cast<long long>(lrow), a.dbg_rows, a.status) ? -LSE[lrow] * kLog2e : 0.f;
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
  griddep_wait();  // a programmatic dependent of the main kernel: its reductions are complete
  if (i >= n4) return;
  const float4 v = reinterpret_cast<const float4*>(dQacc)[i];
  uint2 w;
  w.x = pack_bf16x2(v.x, v.y);
  w.y = pack_bf16x2(v.z, v.w);
  reinterpret_cast<uint2*>(dQ)[i] = w;
}

// --------------------------------------------------------------------------- 2. main (persistent)
// One CTA per SM takes work items -- the (key tile, batch*head) pairs of the
// one-CTA-per-item grid, in the same order (longest causal work first within
// each group of heads) -- from a counter in the workspace that the preprocess
// zeroes, so each item's fixed costs overlap the previous one: the next item's
// K/V, Q and dO loads and its first S and dP MMAs are issued while the compute
// warps read out and store the previous item's dK and dV, and no CTA launch,
// barrier set-up or TMEM allocation separates two items.  Barrier phases run on
// across items: per-tile barriers by the CTA's running count of query tiles,
// per-item ones (K/V, FINAL and their releases) by its count of items with work.
enum : int {
  BAR_SCHED_FULL = kNumBars,       // + slot (2): an item index published
  BAR_SCHED_EMPTY = kNumBars + 2,  // + slot (2): every consumer has read it
  BAR_KV_EMPTY = kNumBars + 4,     // the item's last MMA has read K and V
  BAR_DKV_FREE = kNumBars + 5,     // the item's dK and dV read out of TMEM
  BAR_KV1 = kNumBars + 6,          // d = 64: the second K, V pair (BAR_KV, BAR_KV_EMPTY: the first)
  BAR_KV_EMPTY1 = kNumBars + 7,
  kNumBarsP = kNumBars + 8,
};
constexpr int kOffTmemSlotP = kNumBarsP * 8;
constexpr int kOffAbortP = kOffTmemSlotP + 4;
constexpr int kOffSchedP = kOffAbortP + 4;  // two int item slots
static_assert(kOffSchedP + 8 <= 256, "barrier block");

// Work item -> (batch*head, key tile) and its query-tile range; false for an
// item with nothing to do (a head past B*H, a key tile past its packed
// sequence, or bad offsets, which the preprocess reports).
template <bool kPacked>
struct BwdItem {
  int bh, b, j, head, tok0, N, kv_len, i0, nt;
  __device__ __forceinline__ bool decode(const BwdArgs& a, int item) {
    const int hg = a.gx / a.nq;  // heads per group
    const int x = item % a.gx, y = item / a.gx;
    bh = y * hg + x % hg;
    if (bh >= a.BH) return false;
    b = bh / a.H;
    j = x / hg;
    head = bh % a.H;
    int n_rows = a.N;
    tok0 = 0;
    if constexpr (kPacked) {
      n_rows = packed_range(a, b, tok0);
      if (n_rows < 0 || j * kTile >= n_rows) return false;
    }
    N = n_rows;
    kv_len = N;
    if (a.kv_lens != nullptr && FA_IN_BOUNDS(b, a.dbg_nb, a.status)) kv_len = min(max(a.kv_lens[b], 0), N);
    const bool live = j * kTile < kv_len;
    i0 = a.causal ? j : 0;
    const int nq = kPacked ? (N + kTile - 1) / kTile : a.nq;
    nt = live ? (nq - i0) : 0;
    return true;
  }
};

template <int D, bool kPacked>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_main_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                       const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                       const __grid_constant__ CUtensorMap tmdV, const BwdArgs a) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  {
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
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + kOffTmemSlotP);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + kOffAbortP);
  volatile int* sched_slot = reinterpret_cast<volatile int*>(smem + C::kOffBar + kOffSchedP);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#define BWD_CRD(row) (kPacked ? w.head : (row)), (kPacked ? w.tok0 + (row) : w.bh)

  if (threadIdx.x == 0) {
    mbar_init(bar(BAR_KV), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(BAR_Q_FULL + s), 1);
      mbar_init(bar(BAR_Q_EMPTY + s), 1);
      mbar_init(bar(BAR_SIDE_FULL + s), 1);
      mbar_init(bar(BAR_SIDE_EMPTY + s), kComputeWarps);
      mbar_init(bar(BAR_SCHED_FULL + s), 1);
      mbar_init(bar(BAR_SCHED_EMPTY + s), kComputeWarps + 1 + (kQWatch<D> ? 1 : 0));
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
    mbar_init(bar(BAR_KV_EMPTY), 1);
    mbar_init(bar(BAR_KV1), 1);
    mbar_init(bar(BAR_KV_EMPTY1), 1);
    mbar_init(bar(BAR_DKV_FREE), kComputeWarps);
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
  // launched as a programmatic dependent of the preprocess: the set-up above
  // overlaps its tail; its outputs (work counter, -D and -LSE2 rows, zeroed
  // accumulator) are complete and visible from here on
  griddep_wait();
  const uint32_t tmem = *tmem_slot;
#ifdef FA_DEBUG
  const WaitCtx wc{abort_flag, a.status, a.dbg_timeout_ns != 0 ? a.dbg_timeout_ns : kWaitTimeoutNs};
#else
  const WaitCtx wc{abort_flag, a.status};
#endif
  // consumers read item k from slot k & 1 once SCHED_FULL has completed for it
  // (the compute warps' version ignores the abort flag, like their other waits)
  auto take_item_alike = [&](int k, int& item) -> bool {
    if (!mbar_wait_alike(bar(BAR_SCHED_FULL + (k & 1)), static_cast<uint32_t>(k >> 1) & 1u, wc)) return false;
    item = sched_slot[k & 1];
    return true;
  };
  auto take_item = [&](int k, int& item) -> bool {
    if (!mbar_wait(bar(BAR_SCHED_FULL + (k & 1)), static_cast<uint32_t>(k >> 1) & 1u, wc)) return false;
    item = sched_slot[k & 1];
    return true;
  };
  // K, V buffer of the kf-th item with work, and how many times it was used before
  // (alternating only pays for short items: at most kAltMaxTiles query tiles)
  const bool kv_alt = C::kKVBufs == 2 && a.nq <= kAltMaxTiles;
  auto kv_slot = [&](int kf) { return kv_alt ? (kf & 1) : 0; };
  auto kv_use = [&](int kf) { return kv_alt ? (kf >> 1) : kf; };
  auto kv_full = [&](int slot) { return bar(slot ? BAR_KV1 : BAR_KV); };
  auto kv_empty = [&](int slot) { return bar(slot ? BAR_KV_EMPTY1 : BAR_KV_EMPTY); };

  if (warp >= kComputeWarps) {
    regs_dealloc<kRegsOther<D>>();
    if (warp == kComputeWarps) {
      // ---------------------------------------------------------- producer (and scheduler)
      if (lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmdO);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        int cur = static_cast<int>(atomicAdd(a.sched, 1u));
        sched_slot[0] = cur;
        mbar_arrive(bar(BAR_SCHED_FULL + 0));
        int gs = 0, kf = 0, side_issued = 0, q_issued = 0, o_issued = 0, kv_issued = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
          const int item = cur;
          if (item >= a.n_items) break;
          // publish item k + 1 in slot (k + 1) & 1 once every consumer has read
          // item k - 1 from it
          if (k >= 1 && !mbar_wait(bar(BAR_SCHED_EMPTY + ((k + 1) & 1)), static_cast<uint32_t>((k - 1) >> 1) & 1u,
                                   wc)) {
            ok = false;
            break;
          }
          cur = static_cast<int>(atomicAdd(a.sched, 1u));
          sched_slot[(k + 1) & 1] = cur;
          mbar_arrive(bar(BAR_SCHED_FULL + ((k + 1) & 1)));
          BwdItem<kPacked> w;
          if (!w.decode(a, item) || w.nt == 0) continue;
          const size_t side_row = static_cast<size_t>(w.bh) * a.Npad;
          // K_j, V_j once the last MMA of the item that used this buffer before has read it
          const int ks = kv_slot(kf), ku = kv_use(kf);
          if (ku > 0 && !mbar_wait(kv_empty(ks), static_cast<uint32_t>(ku - 1) & 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t kvb = sbase + (ks ? C::kOffKV1 : C::kOffK);
          mbar_arrive_expect_tx(kv_full(ks), 2 * C::kTileBytes);
          for (int s = 0; s < C::kSub; ++s) {
            tma_load_3d(kvb + s * C::kSubBytes, &tmK, kv_full(ks), s * 64, BWD_CRD(w.j * kTile));
            tma_load_3d(kvb + C::kTileBytes + s * C::kSubBytes, &tmV, kv_full(ks), s * 64, BWD_CRD(w.j * kTile));
          }
          kv_issued = kf + 1;
          for (int it = 0; it < w.nt; ++it) {
            const int g = gs + it;
            const int i = w.i0 + it;
            const int sd = g & 1;
            if (!mbar_wait(bar(BAR_SIDE_EMPTY + sd), ((g >> 1) & 1) ^ 1, wc)) {
              ok = false;
              break;
            }
            if (FA_IN_BOUNDS(static_cast<long long>(side_row) + i * kTile + kTile - 1, a.dbg_side, a.status)) {
              mbar_arrive_expect_tx(bar(BAR_SIDE_FULL + sd), 1024);
              bulk_load(sbase + C::kOffSide + sd * 1024, a.Lpad + side_row + i * kTile, 512,
                        bar(BAR_SIDE_FULL + sd));
              bulk_load(sbase + C::kOffSide + sd * 1024 + 512, a.Dpad + side_row + i * kTile, 512,
                        bar(BAR_SIDE_FULL + sd));
            } else {
              mbar_arrive(bar(BAR_SIDE_FULL + sd));  // no copy: complete the phase
            }
            side_issued = g + 1;
            if (!mbar_wait(bar(BAR_Q_EMPTY + sd), ((g >> 1) & 1) ^ 1, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(BAR_Q_FULL + sd), C::kTileBytes);
            for (int s = 0; s < C::kSub; ++s)
              tma_load_3d(sbase + C::kOffRing + sd * C::kTileBytes + s * C::kSubBytes, &tmQ, bar(BAR_Q_FULL + sd),
                          s * 64, BWD_CRD(i * kTile));
            q_issued = g + 1;
            if (!mbar_wait(bar(BAR_DO_EMPTY), (g & 1) ^ 1, wc)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(BAR_DO_FULL), C::kTileBytes);
            for (int s = 0; s < C::kSub; ++s)
              tma_load_3d(sbase + C::kOffRing + 2 * C::kTileBytes + s * C::kSubBytes, &tmdO, bar(BAR_DO_FULL),
                          s * 64, BWD_CRD(i * kTile));
            o_issued = g + 1;
          }
          gs += w.nt;
          kf += 1;
        }
        // every issued copy lands before the CTA can exit
        const int kv_bufs = kv_alt ? 2 : 1;
        for (int s = 0; s < kv_bufs && s < kv_issued; ++s) {
          const int last = s + kv_bufs * ((kv_issued - 1 - s) / kv_bufs);  // its last item
          drain_wait(kv_full(s), static_cast<uint32_t>(kv_use(last)) & 1u);
        }
        for (int s = 0; s < 2 && s < q_issued; ++s) {
          const int last = s + 2 * ((q_issued - 1 - s) / 2);
          drain_wait(bar(BAR_Q_FULL + s), (last >> 1) & 1);
        }
        for (int s = 0; s < 2 && s < side_issued; ++s) {
          const int last = s + 2 * ((side_issued - 1 - s) / 2);
          drain_wait(bar(BAR_SIDE_FULL + s), (last >> 1) & 1);
        }
        if (o_issued > 0) drain_wait(bar(BAR_DO_FULL), (o_issued - 1) & 1);
      }
    } else if (warp == kComputeWarps + 1) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idSS = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t idKN = idesc_bf16_f32(128, D, false, true);     // dV (TS), dK
        const uint32_t sK = sbase + C::kOffK, sV = sbase + C::kOffV, sP = sbase + C::kOffP;
        auto q_addr = [&](int g) { return sbase + C::kOffRing + (g & 1) * C::kTileBytes; };
        const uint32_t aO = sbase + C::kOffRing + 2 * C::kTileBytes;
        const uint64_t kK0 = sdesc_sw128(sK, 16, 1024), kV0 = sdesc_sw128(sV, 16, 1024);
        const uint64_t kP = sdesc_sw128(sP, 16, 1024), kO = sdesc_sw128(aO, 16, 1024);
        const uint64_t mK0 = sdesc_sw128(sK, C::kSubBytes, 1024), mP = sdesc_sw128(sP, C::kSubBytes, 1024);
        const uint64_t mO = sdesc_sw128(aO, C::kSubBytes, 1024);
        const uint64_t kQ0 = sdesc_sw128(q_addr(0), 16, 1024), mQ0 = sdesc_sw128(q_addr(0), C::kSubBytes, 1024);
        auto kq = [&](int g) { return sdesc_advance(kQ0, (g & 1) * C::kTileBytes); };
        auto mq = [&](int g) { return sdesc_advance(mQ0, (g & 1) * C::kTileBytes); };
        auto mma_kmajor_d = [&](uint32_t dcol, uint64_t da, uint64_t db) {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * C::kSubBytes + (k & 3) * 32;
            mma_ss(tmem + dcol, sdesc_advance(da, off), sdesc_advance(db, off), idSS, k > 0 ? 1u : 0u);
          }
        };
        int gs = 0, kf = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
          int item = 0;
          if (!(ok = take_item(k, item))) break;
          mbar_arrive(bar(BAR_SCHED_EMPTY + (k & 1)));
          if (item >= a.n_items) break;
#ifdef FA_DEBUG
          if (item == a.dbg_stall_item) {  // injected stall: this warp issues nothing more
            ok = false;
            break;
          }
#endif
          BwdItem<kPacked> w;
          if (!w.decode(a, item) || w.nt == 0) continue;
          const int nt = w.nt;
          const int ks = kv_slot(kf);
          if (!(ok = mbar_wait(kv_full(ks), static_cast<uint32_t>(kv_use(kf)) & 1u, wc))) break;
          // descriptors of this item's K, V buffer: the first pair's advanced by the offset
          // (start address in 16-byte units, the descriptor's low bits)
          const uint32_t kvo = ks ? static_cast<uint32_t>((C::kOffKV1 - C::kOffK) >> 4) : 0u;
          // (formed at each use, not kept live: the issuing thread's registers are tight)
          auto at_kv = [&](uint64_t d0) {
            if constexpr (C::kKVBufs == 1) return d0;
            uint64_t r;
            asm volatile("add.u64 %0, %1, %2;" : "=l"(r) : "l"(d0), "l"(static_cast<uint64_t>(kvo)));
            return r;
          };
          // prologue: S_0 and dP_0; dP_0 overwrites the previous item's last dQ
          if (!(ok = mbar_wait(bar(BAR_Q_FULL + (gs & 1)), (gs >> 1) & 1, wc))) break;
          tc_fence_after();
          mma_kmajor_d(C::kColS, at_kv(kK0), kq(gs));
          mma_commit(bar(BAR_S));
          if (!(ok = mbar_wait(bar(BAR_DO_FULL), gs & 1, wc))) break;
          if (gs > 0 && !(ok = mbar_wait(bar(BAR_DQ_READ), (gs - 1) & 1, wc))) break;
          tc_fence_after();
          mma_kmajor_d(C::kColDP, at_kv(kV0), kO);
          mma_commit(bar(BAR_DP));
          for (int it = 0; ok && it < nt; ++it) {
            const int g = gs + it;
            const bool next = it + 1 < nt;
            if (!(ok = mbar_wait(bar(BAR_P), g & 1, wc))) break;
            // the item's first dV and dK overwrite the accumulators: the
            // previous item's dK and dV must have been read out
            if (it == 0 && kf > 0 && !(ok = mbar_wait(bar(BAR_DKV_FREE), static_cast<uint32_t>(kf - 1) & 1u, wc)))
              break;
            tc_fence_after();
#pragma unroll
            for (int k2 = 0; k2 < kTile / 16; ++k2) {
              const uint32_t acol = 32 * (k2 >> 1) + 8 * (k2 & 1);
              mma_ts(tmem + C::kColDV, tmem + C::kColS + acol, sdesc_advance(mO, k2 * 2048), idKN,
                     (it > 0 || k2 > 0) ? 1u : 0u);
            }
            mma_commit(bar(BAR_DO_EMPTY));
            if (!(ok = mbar_wait(bar(BAR_DS), g & 1, wc))) break;
            tc_fence_after();
            if constexpr (D == 128) {
              constexpr uint32_t idQT = idesc_bf16_f32(128, 128, true, true);  // A = K^T, B = dS^T
#pragma unroll
              for (int k2 = 0; k2 < kTile / 16; ++k2)
                mma_ss(tmem + C::kColDQ, sdesc_advance(at_kv(mK0), k2 * 2048), sdesc_advance(mP, k2 * 2048), idQT,
                       k2 > 0 ? 1u : 0u);
              mma_commit(bar(BAR_DQ_FULL));
#pragma unroll
              for (int k2 = 0; k2 < kTile / 16; ++k2) {
                const uint32_t acol = 32 * (k2 >> 1) + 16 + 8 * (k2 & 1);
                mma_ts(tmem + C::kColDK, tmem + C::kColS + acol, sdesc_advance(mq(g), k2 * 2048), idKN,
                       (it > 0 || k2 > 0) ? 1u : 0u);
              }
            } else {
              constexpr uint32_t idNN = idesc_bf16_f32(128, D, true, true);  // A = dS, B = K
#pragma unroll
              for (int k2 = 0; k2 < kTile / 16; ++k2)
                mma_ss(tmem + C::kColDQ, sdesc_advance(mP, k2 * 2048), sdesc_advance(at_kv(mK0), k2 * 2048), idNN,
                       k2 > 0 ? 1u : 0u);
              mma_commit(bar(BAR_DQ_FULL));
#pragma unroll
              for (int k2 = 0; k2 < kTile / 16; ++k2) {
                const uint32_t aoff = (k2 >> 2) * C::kSubBytes + (k2 & 3) * 32;
                mma_ss(tmem + C::kColDK, sdesc_advance(kP, aoff), sdesc_advance(mq(g), k2 * 2048), idKN,
                       (it > 0 || k2 > 0) ? 1u : 0u);
              }
            }
            mma_commit(bar(BAR_Q_EMPTY + (g & 1)));
            if (next) {
              // with the watcher, DS(g) completed only after Q of tile g + 1 landed
              if (!kQWatch<D> && !(ok = mbar_wait(bar(BAR_Q_FULL + ((g + 1) & 1)), ((g + 1) >> 1) & 1, wc)))
                break;
              if (!kQWatch<D>) tc_fence_after();
              mma_kmajor_d(C::kColS, at_kv(kK0), kq(g + 1));
              mma_commit(bar(BAR_S));
              if (!(ok = mbar_wait(bar(BAR_DO_FULL), (g + 1) & 1, wc))) break;
              if (!(ok = mbar_wait(bar(BAR_DQ_READ), g & 1, wc))) break;
              tc_fence_after();
              mma_kmajor_d(C::kColDP, at_kv(kV0), kO);
              mma_commit(bar(BAR_DP));
            }
          }
          if (!ok) break;
          mma_commit(bar(BAR_FINAL));
          mma_commit(kv_empty(ks));
          gs += nt;
          kf += 1;
        }
        mma_commit(bar(BAR_DRAIN));
        drain_wait(bar(BAR_DRAIN), 0);
      }
    } else if (kQWatch<D> && warp == kComputeWarps + 2) {
      // ---------------------------------------------------------- Q watcher
      // One arrival on DS(g) per tile g, after Q of tile g + 1 (same item) has
      // landed and only once DS(g - 1) has completed.
      if (lane == 0) {
        int gs = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
          int item = 0;
          if (!(ok = take_item(k, item))) break;
          mbar_arrive(bar(BAR_SCHED_EMPTY + (k & 1)));
          if (item >= a.n_items) break;
          BwdItem<kPacked> w;
          if (!w.decode(a, item) || w.nt == 0) continue;
          for (int it = 0; it < w.nt; ++it) {
            const int g = gs + it;
            if (g > 0 && !(ok = mbar_wait(bar(BAR_DS), static_cast<uint32_t>(g - 1) & 1u, wc))) break;
            if (it + 1 < w.nt &&
                !(ok = mbar_wait(bar(BAR_Q_FULL + ((g + 1) & 1)), static_cast<uint32_t>((g + 1) >> 1) & 1u, wc)))
              break;
            mbar_arrive(bar(BAR_DS));
          }
          gs += w.nt;
        }
      }
    }
  } else {
    regs_alloc<kRegsCompute<D>>();
    // ------------------------------------------------------------ compute warps
    const int grp = warp >> 2;  // warpgroup: query columns 32 grp .. 32 grp + 31
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;  // key row (S^T, dP^T, dK, dV); head-dim row of dQ^T (d = 128)
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t dsrow = sbase + C::kOffP + (grp >> 1) * C::kSubBytes + r * 128;
    const int swz = r & 7;
    const float2 sl2v = make_float2(a.scale_log2, a.scale_log2);
    const float2 scv = make_float2(a.scale, a.scale);
    // The compute warps wait on the same phases in the same order and hold
    // named barriers between their waits.  Their waits ignore the CTA's abort
    // flag and give up only at their own limit, so a phase that never
    // completes stops all of them at the same wait and none is left at a
    // barrier for a thread that has gone.
    bool aborted = false;
    int gs = 0, kf = 0;
    for (int k = 0; !aborted; ++k) {
      int item = 0;
      if (!take_item_alike(k, item)) {
        aborted = true;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_SCHED_EMPTY + (k & 1)));
      if (item >= a.n_items) break;
      BwdItem<kPacked> w;
      if (!w.decode(a, item)) continue;
      const int N = w.N;
      const int nt = w.nt;
      const int key = w.j * kTile + r;
      const bool key_ok = key < w.kv_len;
      for (int it = 0; it < nt; ++it) {
        const int g = gs + it;
        const int i = w.i0 + it;
        const int sd = g & 1;
        if (!mbar_wait_alike(bar(BAR_SIDE_FULL + sd), (g >> 1) & 1, wc) || !mbar_wait_alike(bar(BAR_S), g & 1, wc)) {
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
        if (!mbar_wait_alike(bar(BAR_DP), g & 1, wc)) {
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
            const float2 g0 =
                fadd2(make_float2(__uint_as_float(dv[c]), __uint_as_float(dv[c + 1])), make_float2(d4.x, d4.y));
            const float2 g1 = fadd2(make_float2(__uint_as_float(dv[c + 2]), __uint_as_float(dv[c + 3])),
                                    make_float2(d4.z, d4.w));
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
          if (g > 0) {
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
            st_shared_v4(dsrow + (((chunk ^ swz)) << 4), pk[4 * c8], pk[4 * c8 + 1], pk[4 * c8 + 2],
                         pk[4 * c8 + 3]);
          }
        }
        if constexpr (D == 128) tmem_st_wait();
        fence_proxy_async_smem();
        if constexpr (D == 128) tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_DS));
        // ---- dQ_i += this tile's contribution
        if (!mbar_wait_alike(bar(BAR_DQ_FULL), g & 1, wc)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        if constexpr (D == 128) {
          // dQ^T: lane = head-dim index r, columns = this warpgroup's 32 queries;
          // staged as one 32 x 128 fp32 box per warpgroup, added by a TMA reduction
          uint32_t rr[32];
          tmem_ld32(tmem + lane_off + C::kColDQ + grp * 32, rr);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_DQ_READ));
          const int q0 = i * kTile + grp * 32;
          const uint32_t stg =
              (grp < 2) ? sbase + C::kOffStage + grp * 16384 : sbase + C::kOffP + (grp - 2) * 16384;
          const bool leader = (q4 == 0 && lane == 0);
          if (grp < 2 && g > 0 && leader) bulk_wait_read_all();  // this staging slot's previous reduction
          named_barrier_sync(2 + grp, 128);
#pragma unroll
          for (int q = 0; q < 32; ++q) st_shared_f32(stg + q * 512 + r * 4, __uint_as_float(rr[q]));
          fence_proxy_async_smem();
          named_barrier_sync(2 + grp, 128);
          if (leader && q0 < N) {
            tma_reduce_add_3d(&tmdQ, stg, 0, BWD_CRD(q0));
            bulk_commit();
          }
        } else {
          // dQ: lane = query row, columns = this warpgroup's 16 head-dim entries;
          // the four warps of a TMEM lane quarter stage 32 queries x 64 fp32 as
          // two 128-byte-swizzled halves, added by two TMA reductions
          uint32_t rr[16];
          tmem_ld16(tmem + lane_off + C::kColDQ + grp * 16, rr);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(BAR_DQ_READ));
          const uint32_t stg = sbase + C::kOffStage + q4 * 8192;
          const bool leader = (grp == 0 && lane == 0);
          if (g > 0 && leader) bulk_wait_read_all();  // this staging box's previous reductions
          named_barrier_sync(2 + q4, 128);
          const uint32_t srow = stg + (grp >> 1) * 4096 + lane * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_shared_v4(srow + ((((grp & 1) * 4 + c) ^ (lane & 7)) << 4), rr[4 * c], rr[4 * c + 1],
                         rr[4 * c + 2], rr[4 * c + 3]);
          fence_proxy_async_smem();
          named_barrier_sync(2 + q4, 128);
          const int q0 = i * kTile + q4 * 32;
          if (leader && q0 < N) {
            tma_reduce_add_3d(&tmdQ, stg, 0, BWD_CRD(q0));
            tma_reduce_add_3d(&tmdQ, stg + 4096, 32, BWD_CRD(q0));
            bulk_commit();
          }
        }
      }
      if (aborted) break;
      // ---- epilogue: dV_j, dK_j rows (thread = key row r), head-dim columns of
      // this warpgroup; TMEM is released for the next item before the stores
      const bool have = nt > 0;
      if (have && !mbar_wait_alike(bar(BAR_FINAL), static_cast<uint32_t>(kf) & 1u, wc)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      constexpr int kCols = D / 4;
      // packed bf16 pairs of this thread's dV and dK columns
      uint32_t pv[kCols / 2], pk2[kCols / 2];
      if (have) {
        {
          uint32_t rr[kCols];
          if constexpr (kCols == 32) tmem_ld32(tmem + lane_off + C::kColDV + grp * kCols, rr);
          else tmem_ld16(tmem + lane_off + C::kColDV + grp * kCols, rr);
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) pv[c] = pack_bf16x2(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1]));
        }
        {
          uint32_t rr[kCols];
          if constexpr (kCols == 32) tmem_ld32(tmem + lane_off + C::kColDK + grp * kCols, rr);
          else tmem_ld16(tmem + lane_off + C::kColDK + grp * kCols, rr);
#pragma unroll
          for (int c = 0; c < kCols / 2; ++c) pk2[c] = pack_bf16x2(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1]));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(BAR_DKV_FREE));
      } else {
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) pv[c] = pk2[c] = 0u;
      }
      if constexpr (kPacked) {
        // packed: rows past the sequence belong to the next one, so each
        // thread stores its own row
        const size_t krow = static_cast<size_t>(w.tok0 + key) * a.H + w.head;
        if (key < N && FA_IN_BOUNDS(static_cast<long long>(krow), a.dbg_rows, a.status)) {
          const size_t rowoff = (krow * D + grp * kCols) * 2;
          uint4* dv_dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.dV) + rowoff);
          uint4* dk_dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.dK) + rowoff);
#pragma unroll
          for (int q = 0; q < kCols / 8; ++q) {
            dv_dst[q] = make_uint4(pv[4 * q], pv[4 * q + 1], pv[4 * q + 2], pv[4 * q + 3]);
            dk_dst[q] = make_uint4(pk2[4 * q], pk2[4 * q + 1], pk2[4 * q + 2], pk2[4 * q + 3]);
          }
        }
      } else {
        // dense: dV and dK are staged as 128-byte-swizzled tiles and written by
        // TMA stores (rows past N clipped), full lines instead of 16-byte
        // pieces 2 d bytes apart.  d = 128: dV in the dQ staging buffer, dK in
        // the dS^T buffer, one 64-column sub-tile per warpgroup leader, each in
        // the region its own next dQ staging reuses; d = 64: both in the
        // staging buffer, 64-row halves by the four lane-quarter leaders.
        const bool qleader = (D == 128) ? (q4 == 0 && lane == 0) : (grp == 0 && lane == 0);
        // the last tile's dQ reductions have read their staging boxes
        if (qleader) bulk_wait_read_all();
        named_barrier_sync(1, 32 * kComputeWarps);
        const uint32_t vbase = sbase + C::kOffStage;
        const uint32_t kbase = (D == 128) ? sbase + C::kOffP : sbase + C::kOffStage + kTile * 128;
#pragma unroll
        for (int h2 = 0; h2 < kCols / 8; ++h2) {
          // 16-byte chunk of this thread's columns: d = 128: sub-tile grp / 2,
          // chunks 4 (grp & 1) + h2; d = 64: chunks 2 grp + h2 of the one sub-tile
          const int sub = (D == 128) ? (grp >> 1) : 0;
          const int chunk = (D == 128) ? 4 * (grp & 1) + h2 : 2 * grp + h2;
          const uint32_t off = sub * C::kSubBytes + r * 128 + ((chunk ^ swz) << 4);
          st_shared_v4(vbase + off, pv[4 * h2], pv[4 * h2 + 1], pv[4 * h2 + 2], pv[4 * h2 + 3]);
          st_shared_v4(kbase + off, pk2[4 * h2], pk2[4 * h2 + 1], pk2[4 * h2 + 2], pk2[4 * h2 + 3]);
        }
        fence_proxy_async_smem();
        named_barrier_sync(1, 32 * kComputeWarps);
        if (qleader) {
          const int row0 = w.j * kTile;
          if constexpr (D == 128) {
            // warpgroups 0-1: dV sub-tile grp; 2-3: dK sub-tile grp - 2
            if (grp < 2)
              tma_store_3d(&tmdV, vbase + grp * C::kSubBytes, 64 * grp, row0, w.bh);
            else
              tma_store_3d(&tmdK, kbase + (grp - 2) * C::kSubBytes, 64 * (grp - 2), row0, w.bh);
          } else {
            // lane quarters 0-1: dV rows 64 q4 ..; 2-3: dK rows 64 (q4 - 2) ..
            if (q4 < 2)
              tma_store_3d(&tmdV, vbase + q4 * 64 * 128, 0, row0 + 64 * q4, w.bh);
            else
              tma_store_3d(&tmdK, kbase + (q4 - 2) * 64 * 128, 0, row0 + 64 * (q4 - 2), w.bh);
          }
          bulk_commit();
        }
      }
      if (have) {
        gs += nt;
        kf += 1;
      }
    }
    if (lane == 0) bulk_wait_read_all();  // staging must outlive the reductions' reads
  }

  griddep_launch_dependents();  // the dQ conversion may start launching (it waits for completion)
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}
#undef BWD_CRD

// Launches `kernel` as a programmatic dependent of the work before it in the
// stream: it may be scheduled before that work completes and must wait for it
// (griddepcontrol.wait) before touching its results.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args&&... args) {
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) cudaGetLastError();
  return e;
}

// The scheduler counter of the persistent kernel: 256 bytes after the fp32 dQ
// accumulator (elements floats) in the workspace, whose -D and -LSE2 rows take
// `side` bytes each.
inline unsigned* bwd_sched_ptr(void* workspace, size_t side, size_t elements) {
  const size_t acc = (elements * sizeof(float) + 255) & ~static_cast<size_t>(255);
  return reinterpret_cast<unsigned*>(static_cast<uint8_t*>(workspace) + 2 * side + acc);
}

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
#ifdef FA_DEBUG
  a.dbg_nb = B;
  a.dbg_rows = static_cast<long long>(BH) * N;
  a.dbg_side = static_cast<long long>(BH) * Npad;
  take_backward_stall(a);
#endif
  a.status = device_status_ptr();
  if (a.status == nullptr) return FA_ERR_CUDA;

  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(BH)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(N) * D * 2};
  const uint32_t box[3] = {64, kTile, 1};
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
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
  // work items: (key tile, batch*head) pairs, key tile * heads per group + head
  // in group fastest, then the group of heads
  const int hg = bwd_head_group(N, D, false);
  a.gx = nq * hg;
  a.n_items = a.gx * ceil_div(BH, hg);
  a.sched = bwd_sched_ptr(workspace, side, static_cast<size_t>(BH) * N * D);
  // dK, dV as TMA store targets: 64-column boxes of a key tile's rows (d = 64:
  // 64-row halves)
  const uint32_t sbox[3] = {64, D == 128 ? 128u : 64u, 1};
  if (!encode_bf16_tmap(&tdk, dK, 3, dims, strides, sbox) || !encode_bf16_tmap(&tdv, dV, 3, dims, strides, sbox))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&bwd_main_kernel<D, false>), C::kSmemBytes))
    return FA_ERR_CUDA;
  const long long pre_rows = static_cast<long long>(BH) * Npad;
  bwd_pre_kernel<D><<<static_cast<unsigned>((pre_rows + 8 * (256 / D) - 1) / (8 * (256 / D))), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, a, BH);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  // one persistent CTA per SM (fewer when there are fewer work items)
  const int ctas = min(a.n_items, max(sm_count(), 1));
  if (launch_dependent(bwd_main_kernel<D, false>, dim3(ctas), dim3(kThreads), C::kSmemBytes, stream, tq, tk, tv, tdo,
                       tdq, tdk, tdv, a) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long n4 = static_cast<long long>(BH) * N * D / 4;
  if (launch_dependent(bwd_dq_kernel, dim3(static_cast<unsigned>((n4 + 255) / 256)), dim3(256), 0, stream,
                       static_cast<const float*>(a.dQacc), static_cast<__nv_bfloat16*>(dQ), n4) != cudaSuccess)
    return FA_ERR_CUDA;
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
#ifdef FA_DEBUG
  a.dbg_nb = num_seqs;
  a.dbg_rows = static_cast<long long>(total) * H;
  a.dbg_side = static_cast<long long>(BH) * Npad;
  take_backward_stall(a);
#endif
  a.status = device_status_ptr();
  if (a.status == nullptr) return FA_ERR_CUDA;
  // packed [total, H, D]: TMA dims (D, H, total), 128 consecutive tokens of one head
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(H), static_cast<uint64_t>(total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(H) * D * 2};
  const uint32_t box[3] = {64, 1, kTile};
  CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv;
  if (!encode_bf16_tmap(&tq, Q, 3, dims, strides, box) || !encode_bf16_tmap(&tk, K, 3, dims, strides, box) ||
      !encode_bf16_tmap(&tv, V, 3, dims, strides, box) || !encode_bf16_tmap(&tdo, dO, 3, dims, strides, box))
    return FA_ERR_CUDA;
  const uint64_t qstrides[2] = {static_cast<uint64_t>(D) * 4, static_cast<uint64_t>(H) * D * 4};
  const uint32_t qbox[3] = {D == 128 ? 128u : 32u, 1, 32};
  if (!(D == 128 ? encode_f32_tmap(&tdq, a.dQacc, 3, dims, qstrides, qbox)
                 : encode_f32_sw128_tmap(&tdq, a.dQacc, 3, dims, qstrides, qbox)))
    return FA_ERR_CUDA;
  // work items: (key tile, batch*head) pairs, key tile * heads per group + head
  // in group fastest, then the group of heads
  const int hg = bwd_head_group(max_seqlen, D, true);
  a.gx = nq * hg;
  a.n_items = a.gx * ceil_div(BH, hg);
  a.sched = bwd_sched_ptr(workspace, side, static_cast<size_t>(total) * H * D);
  // (the packed kernel stores dK, dV row by row; these maps are not used)
  if (!encode_bf16_tmap(&tdk, dK, 3, dims, strides, box) || !encode_bf16_tmap(&tdv, dV, 3, dims, strides, box))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&bwd_main_kernel<D, true>), C::kSmemBytes))
    return FA_ERR_CUDA;
  const long long pre_rows = static_cast<long long>(BH) * Npad;
  bwd_pre_kernel<D><<<static_cast<unsigned>((pre_rows + 8 * (256 / D) - 1) / (8 * (256 / D))), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(O), static_cast<const __nv_bfloat16*>(dO), LSE, a, BH);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_CUDA;
  // one persistent CTA per SM (fewer when there are fewer work items)
  const int ctas = min(a.n_items, max(sm_count(), 1));
  if (launch_dependent(bwd_main_kernel<D, true>, dim3(ctas), dim3(kThreads), C::kSmemBytes, stream, tq, tk, tv, tdo,
                       tdq, tdk, tdv, a) != cudaSuccess)
    return FA_ERR_CUDA;
  const long long n4 = static_cast<long long>(total) * H * D / 4;
  if (launch_dependent(bwd_dq_kernel, dim3(static_cast<unsigned>((n4 + 255) / 256)), dim3(256), 0, stream,
                       static_cast<const float*>(a.dQacc), static_cast<__nv_bfloat16*>(dQ), n4) != cudaSuccess)
    return FA_ERR_CUDA;
  return launch_status();
}

}  // namespace

bool arm_backward_stall(int item, unsigned long long timeout_ns) {
#ifdef FA_DEBUG
  g_stall_item = item;
  g_stall_timeout_ns = timeout_ns;
  return true;
#else
  (void)item;
  (void)timeout_ns;
  return false;
#endif
}

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
