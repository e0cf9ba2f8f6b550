// Forward attention on sm_103a: one CTA owns two 128-row query tiles of one
// (batch, head) and streams all visible 128-key K/V tiles through shared
// memory, computing
//     S = Q K^T      (tcgen05 MMA, operands in shared memory, fp32 accumulator in TMEM)
//     online softmax (one thread per query row, registers only); P is written
//                    back as packed bf16 over the first 64 columns of its S tile
//     O += P V       (tcgen05 MMA with A = P read from TMEM, B = V from shared memory)
// so no score tile ever reaches device memory ("精读笔记 08：FlashAttention",
// §3.2 tiling and §3.4 fusion; the recurrence is §3.1 / S12 "核心思路").
//
// Roles (12 warps = 3 warpgroups):
//   warps 0-3  softmax + epilogue for query tile 0 (TMEM lanes 0..127)
//   warps 4-7  softmax + epilogue for query tile 1
//   warp 8     TMA producer: Q tiles once, then K_j, V_j into a slot ring
//   warp 9     MMA issuer (one thread)
//   warp 10    K/V watcher (d = 128): waits for each key tile's K/V group and
//              adds one arrival to query tile 0's P barrier, so the MMA
//              issuer's wait for P(0, j) also covers the ring (one barrier
//              wait fewer per key tile on the issuing thread)
//   warp 11    idle (it completes the third warpgroup)
// The third warpgroup gives registers to the two softmax warpgroups
// (setmaxnreg), so each softmax thread holds its 128 scores without spilling.
// MMA order per key tile j:  PV(0, j), S(0, j+1), PV(1, j), S(1, j+1), so the
// tensor core works on one query tile while the other one's softmax runs.
//
// Online softmax with a stale reference max: a row keeps the reference m_ref
// (log2 units) it last rescaled to; a tile whose max exceeds m_ref by more
// than kRescaleLog2 moves the reference and rescales O (in TMEM) and l by
// alpha = 2^(m_ref_old - m_ref_new).  Otherwise p = 2^(x - m_ref) <= 2^8 and
// nothing is rescaled.  O and l share the reference, so O / l is exact
// (the S12 page's point: a single multiplication corrects all that has been
// accumulated before the maximum moved).
// A row whose running max is still -inf subtracts 0 instead of -inf, which
// avoids exp(-inf - -inf) = NaN on fully masked tiles (S12 warning).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>

#include "fa_internal.h"
#include "sm103.cuh"

namespace fa {
namespace {

constexpr int kThreads = 384;
constexpr uint32_t kRegsSoftmax = 200;  // 2 x 128 x 200 + 128 x 96 = 63488 <= 384 x 168 (the launch pool)
constexpr uint32_t kRegsOther = 96;
constexpr int kRows = 128;   // query rows per tile = TMEM lanes
constexpr int kKeys = 128;   // keys per K/V tile
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int kSub = D / 64;                // 128-byte swizzle sub-tiles per row
  static constexpr int kSubBytes = kRows * 128;      // one sub-tile: 128 rows x 128 B
  static constexpr int kTileBytes = kRows * D * 2;   // Q/K/V tile
  static constexpr int kSlots = (D == 128) ? 5 : 8;  // K/V ring slots
  // The ring is filled and released in groups: group 0 = K_0, group p = V_{p-1}
  // and K_p, the pair the MMA issuer consumes together (one barrier wait and
  // one release per key tile).  Group p reuses slots of group p - kAhead, so
  // kAhead groups are in flight; kGroupBars barrier pairs rotate.
  static constexpr int kAhead = kSlots / 2;
  // d = 128: warp 10 folds each key tile's K/V wait into the P(0, j) barrier
  // (measured: 2.5-3.6 % faster at d = 128, 3 % slower at d = 64)
  static constexpr bool kWatch = (D == 128);
  static constexpr int kGroupBars = kAhead + 1;
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  static constexpr int kOffMask = kOffBar + 256;  // block-sparse key-tile bitmasks and counts
  static constexpr int kSmemBytes = kOffMask + 1024 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns: S of tile t at 128 t, O of tile t at 256 + D t
  __device__ static constexpr uint32_t col_s(int t) { return 128u * static_cast<uint32_t>(t); }
  __device__ static constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(D * t); }
};

// barrier indices (8 bytes each) inside the barrier block
enum : int {
  BAR_Q = 0,
  BAR_KV_FULL = 1,    // + group barrier (max 8)
  BAR_KV_EMPTY = 9,   // + group barrier
  BAR_S_FULL = 17,    // + tile
  BAR_P_FULL = 19,    // + tile
  BAR_O_FINAL = 21,   // + tile
  BAR_DRAIN = 23,
  kNumBars = 24,
};
constexpr int kOffTmemSlot = kNumBars * 8;
// block-sparse: bitmasks over at most kMaskWords * 32 key tiles (union of the
// CTA's two query tiles, then each tile's own row), then the two stream counts
constexpr int kMaskWords = 64;
constexpr int kOffAbort = kOffTmemSlot + 4;

struct FwdArgs {
  void* O;
  float* LSE;
  // dense: keys visible per batch entry (nullptr: all N); paged: kv_len of
  // each sequence (cached prefix + its query chunk)
  const int32_t* kv_lens;
  // packed ragged batch: Q/O are [total, H, D], LSE is [H, total] and
  // sequence s owns tokens cu_seqlens[s] .. cu_seqlens[s+1]-1 (nullptr: dense)
  const int32_t* cu_seqlens;
  int total;
  int H, N;
  int head_group;  // heads whose CTAs are interleaved in the grid (its x extent)
  int causal;
  float scale_log2;  // scale * log2(e)
  unsigned* status;
  // paged K/V (nullptr: K/V laid out like Q): key t of sequence s and KV head
  // g is cache row block_table[s][t / block_size] * block_size + t % block_size
  // of the (D, Hkv, num_rows) tensor maps; query head h reads KV head h / group
  const int32_t* block_table;
  int max_blocks, block_size, box_rows, num_rows, num_blocks, group;
  // block-sparse (nullptr: dense): uint8 [nqb, nkb] per (batch, head), 1 keeps
  // the 128 x 128 score tile; mask_stride = bytes between (batch, head) masks
  // (0: one mask for all)
  const uint8_t* block_mask;
  long long mask_stride;
  int nkb;
#ifdef FA_DEBUG
  // extents for the debug bounds checks: batch entries (sequences), rows of
  // O (D elements each), elements of LSE, bytes of the block mask
  int dbg_nb;
  long long dbg_o_rows, dbg_lse_len, dbg_mask_bytes;
  long long dbg_stall_cta;            // the MMA warp of this CTA (linear index) issues nothing (-1: none)
  unsigned long long dbg_timeout_ns;  // wait limit of this launch (0: the default)
#endif
};

#ifdef FA_DEBUG
// One-shot stall armed by fa_debug_stall_forward, taken by the next forward
// launch (host side, not thread-safe: a debug hook).
long long g_fwd_stall_cta = -1;
unsigned long long g_fwd_stall_timeout_ns = 0;
void take_forward_stall(FwdArgs& a) {
  a.dbg_stall_cta = g_fwd_stall_cta;
  a.dbg_timeout_ns = g_fwd_stall_timeout_ns;
  g_fwd_stall_cta = -1;
  g_fwd_stall_timeout_ns = 0;
}
#endif

// Wait for a barrier phase ignoring the abort flag, for at most ~50 ms; used
// only on the exit path to let in-flight asynchronous work land.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > 50000000ull) break;
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV, const FwdArgs args) {
  using C = FwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t barbase = sbase + C::kOffBar;
  auto bar = [&](int i) -> uint32_t { return barbase + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffBar + kOffTmemSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // grid (heads of a group, query-tile pairs, batch entry or sequence x head
  // group): the heads of a group run side by side, so concurrent CTAs share
  // their K/V in L2.  A group is every head of a batch entry unless those
  // heads' K/V would not fit in L2 together (long N), then fewer heads.
  const int hgrp = args.head_group;
  const int ngrp = (args.H + hgrp - 1) / hgrp;
  const int head = static_cast<int>(blockIdx.z % ngrp) * hgrp + static_cast<int>(blockIdx.x);
  if (head >= args.H) return;  // the last group of a head count hgrp does not divide
  const int bh = static_cast<int>(blockIdx.z / ngrp) * args.H + head;  // dense: batch * H + head; packed: sequence * H + head
  const int b = bh / args.H;
  const int mblk = gridDim.y - 1 - blockIdx.y;  // longest causal work first
  const int N = args.N;
  const bool packed = args.cu_seqlens != nullptr;

  const bool paged = args.block_table != nullptr;
  const int kv_head = paged ? head / args.group : head;

  // rows of this (sequence, head): Lq query rows; kv_len visible keys; query
  // row r sits at key position qoff + r (causal masks keys past it: qoff = 0
  // is the square top-left mask, qoff = kv_len - Lq the bottom-right one of a
  // query chunk at the end of its context); tok0 = first query token (packed)
  // kv_lens: the dense key-padding lengths or the paged context lengths
  const int kv_given =
      (args.kv_lens != nullptr && FA_IN_BOUNDS(b, args.dbg_nb, args.status)) ? args.kv_lens[b] : N;
  int Lq = N, kv_len = N, tok0 = 0, qoff = 0;
  if (packed) {
    if (!FA_IN_BOUNDS(b + 1, args.dbg_nb + 1, args.status)) return;
    tok0 = args.cu_seqlens[b];
    const int tok1 = args.cu_seqlens[b + 1];
    kv_len = paged ? kv_given : tok1 - tok0;
    // offsets must be non-decreasing within [0, total], no sequence may be
    // longer than the max_seqlen the grid covers, and a paged context must fit
    // its block-table row; otherwise nothing is written for this sequence and
    // the status word records the bad argument
    if (tok0 < 0 || tok1 < tok0 || tok1 > args.total || tok1 - tok0 > static_cast<int>(gridDim.y) * 2 * kRows ||
        (paged && (kv_len < 0 || kv_len > args.max_blocks * args.block_size))) {
      if (blockIdx.y == 0 && threadIdx.x == 0) atomicOr(args.status, kStatusBadArgBit);
      return;
    }
    Lq = tok1 - tok0;
    qoff = kv_len - Lq;
  } else {
    kv_len = min(max(kv_given, 0), N);
  }
  if (packed && 2 * mblk * kRows >= Lq) return;  // whole CTA past this sequence's end
  int n_t[2];
  bool valid_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qt = 2 * mblk + t;
    valid_t[t] = qt * kRows < Lq;
    int end = kv_len;
    if (args.causal) end = min(end, qoff + qt * kRows + kRows);
    n_t[t] = (valid_t[t] && end > 0) ? (end + kKeys - 1) / kKeys : 0;
  }
  // Block-sparse: the CTA streams the key tiles that either query tile keeps
  // (the union of its two mask rows, each cut to the tile's causal / key-length
  // range).  A tile kept only for the other query tile is computed fully masked.
  // n_t becomes the number of streamed tiles within tile t's range (a prefix of
  // the stream, as for the dense tile counts).
  const bool sparse = args.block_mask != nullptr;
  uint32_t* mwords = reinterpret_cast<uint32_t*>(smem + C::kOffMask);  // [3][kMaskWords]
  int* mcount = reinterpret_cast<int*>(smem + C::kOffMask + 3 * kMaskWords * 4);
  if (sparse && warp == 10) {
    const uint8_t* mrow = args.block_mask + static_cast<size_t>(bh) * args.mask_stride;
    int c0 = 0, c1 = 0;
    for (int w = lane; w < kMaskWords; w += 32) {
      uint32_t r0 = 0, r1 = 0;
      if (32 * w < n_t[1] || 32 * w < n_t[0]) {
#pragma unroll 4
        for (int bt = 0; bt < 32; ++bt) {
          const int j = 32 * w + bt;
          if (j < n_t[0] &&
              FA_IN_BOUNDS(bh * args.mask_stride + (2LL * mblk) * args.nkb + j, args.dbg_mask_bytes, args.status) &&
              mrow[static_cast<size_t>(2 * mblk) * args.nkb + j])
            r0 |= 1u << bt;
          if (j < n_t[1] &&
              FA_IN_BOUNDS(bh * args.mask_stride + (2LL * mblk + 1) * args.nkb + j, args.dbg_mask_bytes,
                           args.status) &&
              mrow[static_cast<size_t>(2 * mblk + 1) * args.nkb + j])
            r1 |= 1u << bt;
        }
      }
      const uint32_t u = r0 | r1;
      mwords[w] = u;
      mwords[kMaskWords + w] = r0;
      mwords[2 * kMaskWords + w] = r1;
      // streamed tiles inside each query tile's range
      const int lo0 = n_t[0] - 32 * w, lo1 = n_t[1] - 32 * w;
      const uint32_t rng0 = lo0 >= 32 ? ~0u : (lo0 <= 0 ? 0u : (1u << lo0) - 1u);
      const uint32_t rng1 = lo1 >= 32 ? ~0u : (lo1 <= 0 ? 0u : (1u << lo1) - 1u);
      c0 += __popc(u & rng0);
      c1 += __popc(u & rng1);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      c0 += __shfl_xor_sync(0xffffffffu, c0, off);
      c1 += __shfl_xor_sync(0xffffffffu, c1, off);
    }
    if (lane == 0) {
      mcount[0] = c0;
      mcount[1] = c1;
    }
  }
  // first streamed key tile at or after `from` (sparse); bounded by the words
  auto next_kt = [&](int from) -> int {
    int w = from >> 5;
    if (w >= kMaskWords) return 0;
    uint32_t x = mwords[w] & (~0u << (from & 31));
    while (x == 0 && w + 1 < kMaskWords) x = mwords[++w];
    return x == 0 ? 0 : (w << 5) + __ffs(x) - 1;
  };

  // the producer thread sets up the barriers and, unless the key tiles come
  // from a block mask counted above, issues both Q tiles' copies at once (and,
  // for K/V in the Q layout, the first key tile's K), so their latency
  // overlaps the rest of the set-up
  const bool early_k = !sparse && !paged && max(n_t[0], n_t[1]) > 0;
  if (warp == 8 && lane == 0) {
    mbar_init(bar(BAR_Q), 1);
    for (int s = 0; s < C::kGroupBars; ++s) {
      mbar_init(bar(BAR_KV_FULL + s), 1);
      mbar_init(bar(BAR_KV_EMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(BAR_S_FULL + t), 1);
      mbar_init(bar(BAR_P_FULL + t), (t == 0 && C::kWatch) ? 5 : 4);  // tile 0: + the K/V watcher
      mbar_init(bar(BAR_O_FINAL + t), 1);
    }
    mbar_init(bar(BAR_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    const uint32_t qbytes = (valid_t[0] ? C::kTileBytes : 0) + (valid_t[1] ? C::kTileBytes : 0);
    if (!sparse && qbytes != 0 && max(n_t[0], n_t[1]) > 0) {
      mbar_arrive_expect_tx(bar(BAR_Q), qbytes);
      for (int t = 0; t < 2; ++t) {
        if (!valid_t[t]) continue;
        const int row = (2 * mblk + t) * kRows;
        for (int s = 0; s < C::kSub; ++s) {
          const uint32_t dst = sbase + C::kOffQ + t * C::kTileBytes + s * C::kSubBytes;
          if (packed)
            tma_load_3d(dst, &tmQ, bar(BAR_Q), s * 64, head, tok0 + row);
          else
            tma_load_3d(dst, &tmQ, bar(BAR_Q), s * 64, row, bh);
        }
      }
    }
    if (early_k) {  // K of key tile 0 into ring slot 0: group 0 of the producer's stream
      mbar_arrive_expect_tx(bar(BAR_KV_FULL + 0), C::kTileBytes);
      for (int s = 0; s < C::kSub; ++s) {
        const uint32_t dst = sbase + C::kOffKV + s * C::kSubBytes;
        if (packed)
          tma_load_3d(dst, &tmK, bar(BAR_KV_FULL + 0), s * 64, head, tok0);
        else
          tma_load_3d(dst, &tmK, bar(BAR_KV_FULL + 0), s * 64, 0, bh);
      }
    }
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (sparse) {
    n_t[0] = mcount[0];
    n_t[1] = mcount[1];
  }
  const int nmax = max(n_t[0], n_t[1]);
  const uint32_t tmem = *tmem_slot;
#ifdef FA_DEBUG
  const WaitCtx wc{abort_flag, args.status, args.dbg_timeout_ns != 0 ? args.dbg_timeout_ns : kWaitTimeoutNs};
#else
  const WaitCtx wc{abort_flag, args.status};
#endif

  if (warp >= 8) {
   regs_dealloc<kRegsOther>();
   if (warp == 8) {
    // ------------------------------------------------------------ producer
    // TMA coordinates of 128 rows starting at `row`: dense maps are (d, N, B*H),
    // packed maps are (d, H, total)
    auto load_rows = [&](uint32_t dst, const CUtensorMap* tm, uint32_t mb, int x, int row) {
      if (packed)
        tma_load_3d(dst, tm, mb, x, head, tok0 + row);
      else
        tma_load_3d(dst, tm, mb, x, row, bh);
    };
    uint32_t qbytes = 0;
    for (int t = 0; t < 2; ++t)
      if (valid_t[t]) qbytes += C::kTileBytes;
    if (lane == 0 && sparse && qbytes != 0 && nmax > 0) {  // (dense: issued in the set-up)
      mbar_arrive_expect_tx(bar(BAR_Q), qbytes);
      for (int t = 0; t < 2; ++t) {
        if (!valid_t[t]) continue;
        for (int s = 0; s < C::kSub; ++s)
          load_rows(sbase + C::kOffQ + t * C::kTileBytes + s * C::kSubBytes, &tmQ, bar(BAR_Q), s * 64,
                    (2 * mblk + t) * kRows);
      }
    }
    // Paged K/V: a 128-key tile is gathered as `boxes` boxes of box_rows cache
    // rows, each inside one physical block (one block-table entry), and lane r
    // issues box r.  The warp keeps the block-table row in registers, 32
    // entries (one per lane) at a time: the window of the current tile and,
    // loaded one window ahead, the next, so no table read sits on the issue
    // path.  A tile's entries never straddle two windows (128 / block_size
    // divides 32, or one entry per tile).  A box past kv_len, or whose entry is
    // outside [0, num_blocks), reads the zero fill past the last cache row, so
    // masked keys and values stay finite; a bad entry is also recorded in the
    // status word.
    const int32_t* trow = paged ? args.block_table + static_cast<size_t>(b) * args.max_blocks : nullptr;
    const int n_entries = paged ? (kv_len + args.block_size - 1) / args.block_size : 0;
    const int boxes = paged ? kKeys / args.box_rows : 0;
    auto table_window = [&](int w) -> int {
      const int e = 32 * w + lane;
      return (e < n_entries && FA_IN_BOUNDS(static_cast<long long>(b) * args.max_blocks + e,
                                            static_cast<long long>(args.dbg_nb) * args.max_blocks, args.status))
                 ? trow[e]
                 : -1;
    };
    int win = 0, cur = -1, nxt = -1;
    if (paged) {
      cur = table_window(0);
      nxt = table_window(1);
    }
    int crow = args.num_rows;  // cache row of this lane's box in the newest key tile
    int crow_v = args.num_rows;  // ... and in the key tile whose V is loaded next
    bool bad_table = false;
    int groups = 0;  // groups issued
    int kt = -1, kt_v = -1;  // key tiles of the newest K and of the next V
    for (int p = 0; p <= nmax; ++p) {
      const bool has_v = p > 0, has_k = p < nmax;
      const int gb = p % C::kGroupBars;
      int ok = 1;
      if (lane == 0 && p >= C::kAhead) {
        const int pe = p - C::kAhead;  // the group whose slots this one reuses
        ok = mbar_wait(bar(BAR_KV_EMPTY + pe % C::kGroupBars), static_cast<uint32_t>(pe / C::kGroupBars) & 1u, wc)
                 ? 1 : 0;
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      kt_v = kt;
      crow_v = crow;
      if (has_k) {
        kt = sparse ? next_kt(kt + 1) : p;
        if (paged) {  // K and V of a key tile share its boxes
          const int key0 = kt * kKeys;
          const int e0 = key0 / args.block_size;
          if ((e0 >> 5) != win) {
            cur = ((e0 >> 5) == win + 1) ? nxt : table_window(e0 >> 5);
            win = e0 >> 5;
            nxt = table_window(win + 1);
          }
          const int entry = __shfl_sync(0xffffffffu, cur, ((e0 & 31) + lane) & 31);
          crow = args.num_rows;
          const int key = key0 + lane * args.box_rows;
          if (lane < boxes && key < kv_len) {
            if (entry >= 0 && entry < args.num_blocks)
              crow = entry * args.block_size + key % args.block_size;
            else
              bad_table = true;
          }
        }
      }
      if (p == 0 && early_k) {  // group 0 was issued in the set-up
        groups = 1;
        continue;
      }
      const uint32_t fb = bar(BAR_KV_FULL + gb);
      if (lane == 0) mbar_arrive_expect_tx(fb, (has_v ? C::kTileBytes : 0) + (has_k ? C::kTileBytes : 0));
      __syncwarp();  // the transaction count is armed before any copy lands
      for (int part = 0; part < 2; ++part) {  // V_{p-1}, then K_p
        if (part == 0 ? !has_v : !has_k) continue;
        const int u = part == 0 ? 2 * p - 1 : 2 * p;
        const uint32_t dst = sbase + C::kOffKV + (u % C::kSlots) * C::kTileBytes;
        const CUtensorMap* tm = part == 0 ? &tmV : &tmK;
        if (paged) {
          if (lane < boxes) {
            const int cr = part == 0 ? crow_v : crow;
            for (int s = 0; s < C::kSub; ++s)
              tma_load_3d(dst + s * C::kSubBytes + lane * args.box_rows * 128, tm, fb, s * 64, kv_head, cr);
          }
        } else if (lane == 0) {
          const int ktile = part == 0 ? kt_v : kt;
          for (int s = 0; s < C::kSub; ++s) load_rows(dst + s * C::kSubBytes, tm, fb, s * 64, ktile * kKeys);
        }
      }
      groups = p + 1;
    }
    if (__any_sync(0xffffffffu, bad_table) && lane == 0) atomicOr(args.status, kStatusBadTableBit);
    if (lane == 0) {
      // let every issued copy land before the CTA can exit
      if (qbytes != 0 && nmax > 0) drain_wait(bar(BAR_Q), 0);
      for (int g = 0; g < C::kGroupBars && g < groups; ++g) {
        const int p_last = g + C::kGroupBars * ((groups - 1 - g) / C::kGroupBars);
        drain_wait(bar(BAR_KV_FULL + g), static_cast<uint32_t>(p_last / C::kGroupBars) & 1u);
      }
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nmax > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idPV = idesc_bf16_f32(128, D, false, true);
      // Descriptors are built once per operand tile and advanced by immediates,
      // so the single issuing thread keeps the tensor pipe fed.
      const uint64_t dQ0 = sdesc_sw128(sbase + C::kOffQ, 16, 1024);
      const uint64_t dKV0 = sdesc_sw128(sbase + C::kOffKV, 16, 1024);            // K-major view of slot 0
      const uint64_t dV0 = sdesc_sw128(sbase + C::kOffKV, C::kSubBytes, 1024);  // MN-major view of slot 0
      auto issue_S = [&](int t, int slot) {
        const uint64_t da = sdesc_advance(dQ0, t * C::kTileBytes);
        const uint64_t db = sdesc_advance(dKV0, slot * C::kTileBytes);
        const uint32_t dcol = tmem + C::col_s(t);
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * C::kSubBytes + (k & 3) * 32;
          mma_ss(dcol, sdesc_advance(da, off), sdesc_advance(db, off), idS, k > 0 ? 1u : 0u);
        }
      };
      // A = P in TMEM: row = lane, 16 keys per MMA = 8 columns of packed bf16 pairs
      auto issue_PV = [&](int t, int slot, bool acc) {
        const uint64_t db = sdesc_advance(dV0, slot * C::kTileBytes);
        const uint32_t dcol = tmem + C::col_o(t), acol = tmem + C::col_s(t);
#pragma unroll
        for (int k = 0; k < kKeys / 16; ++k)
          mma_ts(dcol, acol + 8 * k, sdesc_advance(db, k * 16 * 128), idPV, (acc || k > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(bar(BAR_Q), 0, wc);
#ifdef FA_DEBUG
      const long long cta = blockIdx.x + static_cast<long long>(gridDim.x) *
                                             (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z);
      if (cta == args.dbg_stall_cta) ok = false;  // injected stall: this warp issues nothing
#endif
      if (ok) ok = mbar_wait(bar(BAR_KV_FULL + 0), 0, wc);  // group 0: K_0
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) {
            issue_S(t, 0);
            mma_commit(bar(BAR_S_FULL + t));
          }
        mma_commit(bar(BAR_KV_EMPTY + 0));
      }
      for (int j = 0; ok && j < nmax; ++j) {
        const int g = j + 1;  // group of V_j and K_{j+1}
        const int gb = g % C::kGroupBars;
        const int sV = (2 * j + 1) % C::kSlots, sK = (2 * j + 2) % C::kSlots;
        // d = 128: while query tile 0 has key tiles, the P(0, j) barrier
        // completes only after the watcher has seen group g land
        if ((!C::kWatch || j >= n_t[0]) &&
            !mbar_wait(bar(BAR_KV_FULL + gb), static_cast<uint32_t>(g / C::kGroupBars) & 1u, wc))
          break;
        tc_fence_after();
        for (int t = 0; t < 2; ++t) {
          if (j < n_t[t]) {
            if (!mbar_wait(bar(BAR_P_FULL + t), static_cast<uint32_t>(j) & 1u, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_PV(t, sV, j > 0);
            if (j == n_t[t] - 1) mma_commit(bar(BAR_O_FINAL + t));
          }
          if (j + 1 < n_t[t]) {
            issue_S(t, sK);
            mma_commit(bar(BAR_S_FULL + t));
          }
        }
        if (!ok) break;
        mma_commit(bar(BAR_KV_EMPTY + gb));
      }
      // every MMA issued above completes before the CTA releases TMEM
      mma_commit(bar(BAR_DRAIN));
      drain_wait(bar(BAR_DRAIN), 0);
    }
   } else if (warp == 10 && C::kWatch) {
    // ------------------------------------------------------------ K/V watcher
    // One arrival per phase of P(0, .): the watcher arrives for key tile j
    // only once phase j - 1 has completed, so it never runs ahead into a
    // phase whose softmax arrivals are still missing.
    if (lane == 0) {
      for (int j = 0; j < n_t[0]; ++j) {
        const int g = j + 1;  // group of V_j and K_{j+1}
        if (j > 0 && !mbar_wait(bar(BAR_P_FULL + 0), static_cast<uint32_t>(j - 1) & 1u, wc)) break;
        if (!mbar_wait(bar(BAR_KV_FULL + g % C::kGroupBars), static_cast<uint32_t>(g / C::kGroupBars) & 1u, wc)) break;
        mbar_arrive(bar(BAR_P_FULL + 0));
      }
    }
   }
  } else {
    regs_alloc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax / epilogue
    const int t = warp >> 2;
    const int q4 = warp & 3;
    const int r_in_tile = q4 * 32 + lane;
    const int row = (2 * mblk + t) * kRows + r_in_tile;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::col_s(t);
    const uint32_t tO = tmem + lane_off + C::col_o(t);
    const float sl2 = args.scale_log2;
    int last_key = kv_len - 1;
    if (args.causal) last_key = min(last_key, qoff + row);

    float m_ref = -INFINITY;
    float l_sum = 0.f;
    bool aborted = false;
    const int n = (t == 0) ? n_t[0] : n_t[1];  // selects, not a runtime-indexed (stack) array
    const uint32_t* rowbits = mwords + (1 + t) * kMaskWords;
    int kt = -1;  // key tile of the current stream step
    const bool valid = (t == 0) ? valid_t[0] : valid_t[1];
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait(bar(BAR_S_FULL + t), static_cast<uint32_t>(j) & 1u, wc)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      float s[kKeys];
      tmem_ld128f(tS, s);
      kt = sparse ? next_kt(kt + 1) : j;
      const bool kept = !sparse || ((rowbits[kt >> 5] >> (kt & 31)) & 1u);
      const int lim = kept ? last_key - kt * kKeys : -1;  // last visible key index within this tile
      if (lim < kKeys - 1) {
#pragma unroll
        for (int i = 0; i < kKeys; ++i)
          if (i > lim) s[i] = -INFINITY;
      }
      float mx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) mx[i] = s[i];
#pragma unroll
      for (int i = 4; i < kKeys; i += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) mx[k] = fmax3f(mx[k], s[i + k], s[i + 4 + k < kKeys ? i + 4 + k : i + k]);
      }
      const float tile_max = fmax3f(fmaxf(mx[0], mx[1]), mx[2], mx[3]);
      const float x_max = tile_max * sl2;
      const bool resc = x_max > m_ref + kRescaleLog2;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_ref - x_max);  // 0 when m_ref = -inf
        m_ref = x_max;
        l_sum *= alpha;
      }
      if (j > 0 && __any_sync(0xffffffffu, resc)) {
        // O <- alpha * O for this warp's 32 rows (alpha = 1 in rows that keep their reference)
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(tO + c0, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tO + c0, r);
        }
        tmem_st_wait();
      }
      const float neg_ref = (m_ref == -INFINITY) ? 0.f : -m_ref;
      const float2 sl2v = make_float2(sl2, sl2), negv = make_float2(neg_ref, neg_ref);
      float2 part[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
      uint32_t pk[kKeys / 2];  // P row as packed bf16 pairs, key 2i in the low half
#pragma unroll
      for (int i = 0; i < kKeys / 2; ++i) {
        const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), sl2v, negv);
        const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
        part[i & 1] = fadd2(part[i & 1], p);
        pk[i] = pack_bf16x2(p.x, p.y);
      }
      l_sum += (part[0].x + part[0].y) + (part[1].x + part[1].y);
      tmem_st64(tS, pk);  // P overwrites the S columns this thread has read
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P_FULL + t));
    }

    if (valid && !aborted) {
      bool have_o = n > 0;
      if (have_o) {
        have_o = mbar_wait(bar(BAR_O_FINAL + t), 0, wc);
        if (!have_o) aborted = true;
      }
      if (!aborted) {
        tc_fence_after();
        const bool empty = !(l_sum > 0.f);
        const float inv = empty ? 0.f : 1.f / l_sum;
        const bool in_range = row < Lq;
        const size_t orow_idx = packed ? static_cast<size_t>(tok0 + row) * args.H + head
                                       : static_cast<size_t>(bh) * N + row;
        uint8_t* orow = static_cast<uint8_t*>(args.O) + orow_idx * (D * 2);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t r[32];
          if (have_o) {
            tmem_ld32(tO + c0, r);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            w[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
          if (in_range && FA_IN_BOUNDS(static_cast<long long>(orow_idx), args.dbg_o_rows, args.status)) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 2);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          }
        }
        if (in_range) {
          const float lse = empty ? -INFINITY : (m_ref + lg2_approx(l_sum)) * 0.69314718055994531f;
          const size_t lidx = packed ? static_cast<size_t>(head) * args.total + tok0 + row
                                     : static_cast<size_t>(bh) * N + row;
          if (FA_IN_BOUNDS(static_cast<long long>(lidx), args.dbg_lse_len, args.status)) args.LSE[lidx] = lse;
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

// Heads per grid group for the dense forward: all H heads of a batch entry
// while their K and V (2 N d bf16 each per head) fit in kL2KVBudget bytes
// together, else the largest divisor of H whose heads do (at least one).
// In-flight CTAs then stream K/V that L2 still holds instead of re-reading it
// from DRAM once per CTA.  The grid's z extent (B x groups) stays <= 65535.
constexpr double kL2KVBudget = 64.0 * 1024 * 1024;
inline int dense_head_group(int B, int H, int N, int D) {
  const double kv_head = 4.0 * static_cast<double>(N) * D;  // K and V of one head, bf16
  int best = H;  // every head: the grid's z extent is then B <= 65535
  for (int g = H; g >= 1; --g) {
    if (H % g != 0 || static_cast<long long>(B) * (H / g) > 65535) continue;
    best = g;
    if (g * kv_head <= kL2KVBudget) return g;
  }
  return best;
}

template <int D>
fa_status fwd_launch_d(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N,
                       int causal, float scale, const int32_t* kv_lens, const uint8_t* block_mask,
                       long long mask_stride, cudaStream_t stream) {
  using C = FwdCfg<D>;
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(N), static_cast<uint64_t>(B) * H};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(N) * D * 2};
  const uint32_t box[3] = {64, kRows, 1};
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_tmap(&tq, Q, 3, dims, strides, box) || !encode_bf16_tmap(&tk, K, 3, dims, strides, box) ||
      !encode_bf16_tmap(&tv, V, 3, dims, strides, box))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&fwd_kernel<D>), C::kSmemBytes)) return FA_ERR_CUDA;
  unsigned* status = device_status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  FwdArgs a{};  // zero: no paged K/V
  a.O = O;
  a.LSE = LSE;
  a.kv_lens = kv_lens;
  a.cu_seqlens = nullptr;
  a.total = 0;
  a.H = H;
  a.N = N;
  a.block_mask = block_mask;
  a.mask_stride = mask_stride;
  a.nkb = ceil_div(N, kKeys);
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.head_group = dense_head_group(B, H, N, D);
#ifdef FA_DEBUG
  a.dbg_nb = B;
  a.dbg_o_rows = a.dbg_lse_len = static_cast<long long>(B) * H * N;
  a.dbg_mask_bytes = block_mask == nullptr ? 0 : (mask_stride != 0 ? static_cast<long long>(B) * H * mask_stride
                                                                     : static_cast<long long>(a.nkb) * a.nkb);
  take_forward_stall(a);
#endif
  dim3 grid(a.head_group, ceil_div(N, 2 * kRows), B * ceil_div(H, a.head_group));
  fwd_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, a);
  return launch_status();
}

template <int D>
fa_status fwd_varlen_launch_d(const void* Q, const void* K, const void* V, void* O, float* LSE,
                              const int32_t* cu_seqlens, int num_seqs, int total, int max_seqlen, int H, int causal,
                              float scale, cudaStream_t stream) {
  using C = FwdCfg<D>;
  // packed [total, H, D]: TMA dims (D, H, total), a box of 128 consecutive tokens of one head
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(H), static_cast<uint64_t>(total)};
  const uint64_t strides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(H) * D * 2};
  const uint32_t box[3] = {64, 1, kRows};
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_tmap(&tq, Q, 3, dims, strides, box) || !encode_bf16_tmap(&tk, K, 3, dims, strides, box) ||
      !encode_bf16_tmap(&tv, V, 3, dims, strides, box))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&fwd_kernel<D>), C::kSmemBytes)) return FA_ERR_CUDA;
  unsigned* status = device_status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  FwdArgs a{};  // zero: no paged K/V
  a.O = O;
  a.LSE = LSE;
  a.kv_lens = nullptr;
  a.cu_seqlens = cu_seqlens;
  a.total = total;
  a.H = H;
  a.N = max_seqlen;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  // a sequence's heads run side by side, grouped like the dense layout's by
  // the K/V of the longest sequence (which bounds every sequence's)
  a.head_group = dense_head_group(num_seqs, H, max_seqlen, D);
#ifdef FA_DEBUG
  a.dbg_nb = num_seqs;
  a.dbg_o_rows = a.dbg_lse_len = static_cast<long long>(total) * H;
  a.dbg_mask_bytes = 0;
  take_forward_stall(a);
#endif
  dim3 grid(a.head_group, ceil_div(max_seqlen, 2 * kRows), num_seqs * ceil_div(H, a.head_group));
  fwd_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, a);
  return launch_status();
}

template <int D>
fa_status fwd_paged_launch_d(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                             const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o, float* lse,
                             int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int num_blocks,
                             int block_size, int max_blocks, int causal, float scale, cudaStream_t stream) {
  using C = FwdCfg<D>;
  // queries packed [total_q, Hq, D] as in the ragged forward; the caches
  // [num_blocks, block_size, Hkv, D] as TMA dims (D, Hkv, num_blocks * block_size),
  // boxes of min(block_size, 128) rows of one KV head
  const int box_rows = block_size < kKeys ? block_size : kKeys;
  const uint64_t qdims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hq), static_cast<uint64_t>(total_q)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Hq) * D * 2};
  const uint32_t qbox[3] = {64, 1, kRows};
  const int num_rows = num_blocks * block_size;
  const uint64_t kdims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv), static_cast<uint64_t>(num_rows)};
  const uint64_t kstrides[2] = {static_cast<uint64_t>(D) * 2, static_cast<uint64_t>(Hkv) * D * 2};
  const uint32_t kbox[3] = {64, 1, static_cast<uint32_t>(box_rows)};
  CUtensorMap tq, tk, tv;
  if (!encode_bf16_tmap(&tq, q, 3, qdims, qstrides, qbox) || !encode_bf16_tmap(&tk, k_cache, 3, kdims, kstrides, kbox) ||
      !encode_bf16_tmap(&tv, v_cache, 3, kdims, kstrides, kbox))
    return FA_ERR_CUDA;
  if (!set_smem_limit(reinterpret_cast<const void*>(&fwd_kernel<D>), C::kSmemBytes)) return FA_ERR_CUDA;
  unsigned* status = device_status_ptr();
  if (status == nullptr) return FA_ERR_CUDA;
  FwdArgs a{};
  a.O = o;
  a.LSE = lse;
  a.kv_lens = seq_lens_k;
  a.cu_seqlens = cu_seqlens_q;
  a.total = total_q;
  a.H = Hq;
  a.N = max_seqlen_q;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.status = status;
  a.block_table = block_table;
  a.max_blocks = max_blocks;
  a.block_size = block_size;
  a.box_rows = box_rows;
  a.num_rows = num_rows;
  a.num_blocks = num_blocks;
  a.group = Hq / Hkv;
  a.head_group = Hq;
#ifdef FA_DEBUG
  a.dbg_nb = num_seqs;
  a.dbg_o_rows = a.dbg_lse_len = static_cast<long long>(total_q) * Hq;
  a.dbg_mask_bytes = 0;
  take_forward_stall(a);
#endif
  dim3 grid(Hq, ceil_div(max_seqlen_q, 2 * kRows), num_seqs);
  fwd_kernel<D><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, a);
  return launch_status();
}

}  // namespace

bool arm_forward_stall(long long cta, unsigned long long timeout_ns) {
#ifdef FA_DEBUG
  g_fwd_stall_cta = cta;
  g_fwd_stall_timeout_ns = timeout_ns;
  return true;
#else
  (void)cta;
  (void)timeout_ns;
  return false;
#endif
}

fa_status fwd_paged_launch(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                           const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o, float* lse,
                           int num_seqs, int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int num_blocks,
                           int block_size, int max_blocks, int causal, float scale, cudaStream_t stream) {
  if (d == 64)
    return fwd_paged_launch_d<64>(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, o, lse, num_seqs,
                                  total_q, max_seqlen_q, Hq, Hkv, num_blocks, block_size, max_blocks, causal, scale,
                                  stream);
  if (d == 128)
    return fwd_paged_launch_d<128>(q, k_cache, v_cache, block_table, cu_seqlens_q, seq_lens_k, o, lse, num_seqs,
                                   total_q, max_seqlen_q, Hq, Hkv, num_blocks, block_size, max_blocks, causal, scale,
                                   stream);
  return FA_ERR_UNSUPPORTED;
}

fa_status fwd_varlen_launch(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            const int32_t* cu_seqlens, int num_seqs, int total, int max_seqlen, int H, int d,
                            int causal, float scale, cudaStream_t stream) {
  if (d == 64)
    return fwd_varlen_launch_d<64>(Q, K, V, O, LSE, cu_seqlens, num_seqs, total, max_seqlen, H, causal, scale, stream);
  if (d == 128)
    return fwd_varlen_launch_d<128>(Q, K, V, O, LSE, cu_seqlens, num_seqs, total, max_seqlen, H, causal, scale, stream);
  return FA_ERR_UNSUPPORTED;
}

fa_status fwd_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                     int causal, float scale, const int32_t* kv_lens, const uint8_t* block_mask,
                     long long mask_stride, cudaStream_t stream) {
  if (d == 64)
    return fwd_launch_d<64>(Q, K, V, O, LSE, B, H, N, causal, scale, kv_lens, block_mask, mask_stride, stream);
  if (d == 128)
    return fwd_launch_d<128>(Q, K, V, O, LSE, B, H, N, causal, scale, kv_lens, block_mask, mask_stride, stream);
  return FA_ERR_UNSUPPORTED;
}

}  // namespace fa
