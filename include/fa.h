/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact IO-aware attention library.
 *
 * The library computes exact softmax attention without writing the N x N
 * score matrix to device memory, following the FlashAttention method as the
 * study notes "精读笔记 08：FlashAttention" describe it (§2.1 standard
 * attention, §3.1 online softmax, §3.2 tiling, §3.3 recomputation, §3.4
 * fusion) and the paged / split-KV decode of the tutorial chapter
 * "S12 FlashAttention" ("实现", flash-decoding, grouped-query heads).
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers unless stated; the caller owns every
 *     buffer (inputs, outputs, workspaces).  No entry point allocates device
 *     memory.
 *   - bf16 tensors are IEEE bfloat16 stored as 16-bit words; "bf16*" below is
 *     written as void*.  Layout [B, H, N, d] is row-major and contiguous
 *     (d fastest).  Base addresses must be 16-byte aligned.
 *   - d (head dimension) must be 64 or 128, else FA_ERR_UNSUPPORTED.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Every call
 *     is asynchronous: the returned status covers argument validation and
 *     launch errors only.  Errors the GPU detects (a timed-out pipeline wait,
 *     an out-of-range block-table entry) are latched in a device status word
 *     and returned by fa_get_device_status().
 *   - Scores are s_ij = scale * <q_i, k_j>; LSE_i = ln sum_j exp(s_ij) over
 *     the visible keys (natural log).  A query row with no visible key gets
 *     O_i = 0 and LSE_i = -inf; no NaN is produced for finite inputs.
 *   - Return values are fa_status codes (as int).
 */
#ifndef FA_GB300_H_
#define FA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fa_status {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,     /* null pointer, negative size, bad combination */
  FA_ERR_UNSUPPORTED = 2,     /* valid request outside what the kernels cover (e.g. d = 96) */
  FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call or launch failed */
  FA_ERR_TIMEOUT = 4,         /* device: a bounded pipeline wait gave up */
  FA_ERR_BAD_BLOCK_TABLE = 5, /* device: a block-table entry was outside [0, num_blocks) */
  FA_ERR_OUT_OF_BOUNDS = 6    /* device, debug builds only: a kernel computed an index outside one of
                                 its buffers; the access was skipped (see fa_debug_build) */
} fa_status;

/* Human-readable name of a status code; never NULL. */
const char* fa_status_string(int status);

/* ABI version of this header (major * 100 + minor). */
int fa_version(void);

/*
 * Forward attention (the tiled, fused forward of the notes' §3.2 / §3.4 with
 * the online-softmax recurrence of §3.1).
 *   Q, K, V : [B, H, N, d] bf16, read only.
 *   O       : [B, H, N, d] bf16, written: O = softmax(scale Q K^T) V per (b, h).
 *   LSE     : [B, H, N] fp32, written: per-row log-sum-exp (the row statistic
 *             that replaces the notes' (m, l) pair, §3.3).
 *   causal  : non-zero masks key j > query i (top-left aligned, square).
 *   scale   : logit scale, typically 1/sqrt(d); must be finite and > 0.
 * B, H >= 1, N >= 0 (N = 0 is a no-op); B <= 65535.  Errors: FA_ERR_INVALID_ARG,
 * FA_ERR_UNSUPPORTED, FA_ERR_CUDA.
 */
int fa_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d, int causal,
           float scale, void* stream);

/*
 * fa_fwd with a key-padding mask: kv_lens (device int32 [B], may be NULL)
 * gives the number of valid keys L_b of each batch entry; keys j >= L_b are
 * masked for every query row (values are clamped to [0, N]).  All N query
 * rows are still computed and written.
 */
int fa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
              int causal, float scale, const int32_t* kv_lens, void* stream);

/*
 * Block-sparse forward attention ("精读笔记 08：FlashAttention" §4.4): the
 * scores are cut into 128 x 128 blocks (query block qb = i / 128, key block
 * kb = j / 128) and a 0/1 block mask keeps or drops each block; dropped
 * blocks are masked like causal ones, and key tiles no query tile of a CTA
 * keeps are never loaded or multiplied.  The result is exact attention under
 * that mask (the approximation is the mask itself).
 *   Q, K, V, O, LSE, causal, scale, kv_lens : as fa_fwd_ex (masks combine by AND).
 *   block_mask : device uint8, nb = ceil(N / 128); [nb, nb] shared by every
 *                (batch, head) when mask_per_head = 0, else [B, H, nb, nb].
 *                Non-zero keeps the block.
 * A row whose blocks are all dropped gets O = 0, LSE = -inf.
 * N <= 262144 (else FA_ERR_UNSUPPORTED); B <= 65535.  Errors as fa_fwd.
 */
int fa_fwd_block_sparse(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int H, int N, int d,
                        int causal, float scale, const int32_t* kv_lens, const uint8_t* block_mask,
                        int mask_per_head, void* stream);

/*
 * Forward attention over a packed ragged batch: num_seqs sequences of
 * different lengths laid end to end, each attending only to itself (with
 * per-sequence causal masking).  This is the irregular-batch case of the
 * S12 chapter's "exp(-inf - -inf) is NaN" passage, where whole key tiles
 * are masked, and the no-padding form of fa_fwd_ex's key-padding mask.
 *   Q, K, V    : [total, H, d] bf16, read only; token t of every head is row t.
 *   O          : [total, H, d] bf16, written for every token of every sequence.
 *   LSE        : [H, total] fp32, written (natural log, as fa_fwd).
 *   cu_seqlens : device int32 [num_seqs + 1]; sequence s owns tokens
 *                cu_seqlens[s] .. cu_seqlens[s+1]-1.  It must start at 0,
 *                be non-decreasing and end at total.  Empty sequences are
 *                allowed.  Query i and key j of a sequence are positions
 *                within that sequence; causal masks j > i (square, top-left).
 *   max_seqlen : an upper bound of the longest sequence (it sizes the grid).
 * num_seqs in [1, 65535], H >= 1, total >= 0 (total = 0 is a no-op).
 * Errors: FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_CUDA for the
 * host-visible arguments.  cu_seqlens lives on the device, so a sequence with
 * bad offsets or longer than max_seqlen is found there: nothing is written for
 * it and fa_get_device_status() then returns FA_ERR_INVALID_ARG.
 */
int fa_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE, const int32_t* cu_seqlens,
                  int num_seqs, int total, int max_seqlen, int H, int d, int causal, float scale, void* stream);

/*
 * Paged (chunked) prefill: a packed batch of query chunks, each attending to
 * its sequence's keys and values in a paged KV cache.  This is the tiled
 * forward with its key tiles fetched through the block table, as the S12
 * chapter's "除了快，它还解锁了什么" (PagedAttention bullet) and "实现"
 * describe, with grouped-query heads.
 *   q            : [total_q, Hq, d] bf16; chunk s is rows cu_seqlens_q[s] ..
 *                  cu_seqlens_q[s+1]-1 (offsets as in fa_fwd_varlen).
 *   k_cache,
 *   v_cache      : [num_blocks, block_size, Hkv, d] bf16 (the decode layout).
 *                  Cache rows of a sequence's blocks past seq_lens_k are read
 *                  and masked, so they must hold finite values.
 *   block_table  : [num_seqs, max_blocks] int32; entries past
 *                  ceil(seq_lens_k[s] / block_size) are never read.  An entry
 *                  outside [0, num_blocks) reads as zero keys and values and
 *                  latches FA_ERR_BAD_BLOCK_TABLE (that sequence's results are
 *                  then meaningless).
 *   seq_lens_k   : [num_seqs] int32 context length kv_len of each sequence:
 *                  its cached prefix plus the chunk, 0 <= kv_len <=
 *                  max_blocks * block_size.  The chunk is the LAST q_len tokens
 *                  of the context: query i sits at position kv_len - q_len + i
 *                  and, when causal, sees keys j <= kv_len - q_len + i
 *                  (bottom-right alignment; q_len = kv_len is fa_fwd_varlen's
 *                  square mask, q_len = 1 is decode).  Rows that see no key
 *                  (q_len > kv_len) get O = 0 and LSE = -inf.
 *   o            : [total_q, Hq, d] bf16, written.   lse: [Hq, total_q] fp32.
 *   Query head h reads KV head h / (Hq / Hkv); Hq % Hkv must be 0.
 *   block_size   : a multiple of 8 that divides 128 or is a multiple of 128,
 *                  else FA_ERR_UNSUPPORTED.
 *   max_seqlen_q : an upper bound of the longest chunk (it sizes the grid).
 * num_seqs in [1, 65535].  Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED,
 * FA_ERR_CUDA; a chunk with bad offsets, longer than max_seqlen_q or with
 * kv_len outside its table row is skipped on the device and
 * fa_get_device_status() returns FA_ERR_INVALID_ARG.
 */
int fa_paged_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                     const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, void* o, float* lse, int num_seqs,
                     int total_q, int max_seqlen_q, int Hq, int Hkv, int d, int num_blocks, int block_size,
                     int max_blocks, int causal, float scale, void* stream);

/*
 * Bytes of device workspace fa_bwd needs: two fp32 [B, H, Npad] row buffers
 * (D = rowsum(dO * O) and LSE in log2 units; Npad = N rounded up to 128), an
 * fp32 [B, H, N, d] dQ accumulator, each rounded up to 256 bytes, and 256
 * bytes for the main kernel's work-item counter.  0 on invalid sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward attention by recomputation (notes §3.3: keep O and the row
 * statistics, rebuild the score tiles on chip).  Gradients of
 * sum(dO * O) for O = fa_fwd(Q, K, V):
 *   dV = P^T dO,  dP = dO V^T,  D = rowsum(dO * O),  dS = P * (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q,   with P = exp(scale Q K^T - LSE).
 *   Q, K, V, O, dO : [B, H, N, d] bf16 (O and LSE from fa_fwd/fa_fwd_ex with
 *                    the same causal, scale and kv_lens).
 *   LSE            : [B, H, N] fp32.
 *   dQ, dK, dV     : [B, H, N, d] bf16, written.  Padded keys get dK = dV = 0.
 *   kv_lens        : as in fa_fwd_ex, may be NULL.
 *   workspace      : device buffer of at least fa_bwd_workspace_size() bytes,
 *                    256-byte aligned; contents on entry are ignored.  Two
 *                    calls that overlap on the GPU must not share it.
 * Errors: FA_ERR_INVALID_ARG (including ws_bytes too small),
 * FA_ERR_UNSUPPORTED, FA_ERR_CUDA.
 */
int fa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE, void* dQ,
           void* dK, void* dV, int B, int H, int N, int d, int causal, float scale, const int32_t* kv_lens,
           void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of device workspace fa_bwd_varlen needs: two fp32 row buffers of
 * num_sequences x H x Npad (Npad = max_seqlen rounded up to 128), an fp32
 * [total, H, d] dQ accumulator, each rounded up to 256 bytes, and 256 bytes for
 * the main kernel's work-item counter.  0 on invalid sizes.
 */
size_t fa_bwd_varlen_workspace_size(int num_seqs, int total, int max_seqlen, int H, int d);

/*
 * Backward of fa_fwd_varlen (the packed ragged batch): the same gradients as
 * fa_bwd, computed per sequence.
 *   Q, K, V, O, dO : [total, H, d] bf16 (O and LSE from fa_fwd_varlen with the
 *                    same cu_seqlens, causal and scale).
 *   LSE            : [H, total] fp32.
 *   dQ, dK, dV     : [total, H, d] bf16, written.
 *   cu_seqlens     : device int32 [num_seqs + 1]; here it must start at 0 and
 *                    end at total (every token belongs to a sequence), be
 *                    non-decreasing, and no sequence may exceed max_seqlen.
 *                    Offsets breaking this are found on the device:
 *                    fa_get_device_status() then returns FA_ERR_INVALID_ARG
 *                    and the gradients are undefined.
 *   workspace      : at least fa_bwd_varlen_workspace_size() bytes, 256-byte
 *                    aligned; contents on entry are ignored.
 * Errors: FA_ERR_INVALID_ARG (including ws_bytes too small), FA_ERR_UNSUPPORTED,
 * FA_ERR_CUDA.
 */
int fa_bwd_varlen(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                  void* dQ, void* dK, void* dV, const int32_t* cu_seqlens, int num_seqs, int total, int max_seqlen,
                  int H, int d, int causal, float scale, void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of device workspace fa_paged_decode needs for `num_splits` partial
 * (m, l, o) states per (batch, query head): fp32 o [B, Hq, num_splits, d] and
 * fp32 (m, l) [B, Hq, num_splits, 2], each rounded up to 256 bytes.
 * num_splits = 0 means the automatic choice (16).  num_splits = 1 needs none
 * (returns 0): a single split writes o and lse itself, in one launch.
 */
size_t fa_paged_decode_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * Paged, split-KV, grouped-query decode (S12 "实现" paged loop, flash-decoding
 * split + (m, l, o) merge, GQA head sharing).
 *   q           : [B, Hq, d] bf16, one query token per sequence (d = 64 or 128).
 *   k_cache,
 *   v_cache     : [num_blocks, block_size, Hkv, d] bf16; key t of sequence b
 *                 and KV head g is k_cache[block_table[b][t / block_size],
 *                 t % block_size, g, :].
 *   block_table : [B, max_blocks] int32; entries past ceil(L_b / block_size)
 *                 are never read.  An entry outside [0, num_blocks) is skipped
 *                 (its keys are treated as masked) and latches
 *                 FA_ERR_BAD_BLOCK_TABLE in the device status word.
 *   seq_lens    : [B] int32 context lengths L_b, 0 <= L_b <= max_blocks *
 *                 block_size (larger values are clamped to that bound).
 *   o           : [B, Hq, d] bf16, written.  lse: [B, Hq] fp32 or NULL.
 *   Query head h reads KV head h / (Hq / Hkv); Hq % Hkv must be 0.
 *   block_size  : a multiple of 16 (16, 32, 64, ...).
 *   num_splits  : 1..16, or 0 for automatic (16).
 *   workspace   : at least fa_paged_decode_workspace_size(B, Hq, d,
 *                 num_splits) bytes, 256-byte aligned; may be NULL when
 *                 num_splits = 1 (one fused launch, the short-context and
 *                 small-batch choice).
 * Errors: FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA.
 */
int fa_paged_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                    const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d, int block_size,
                    int max_blocks, int num_blocks, int num_splits, float scale, void* workspace, size_t ws_bytes,
                    void* stream);

/*
 * A decode step replayed as one CUDA graph (the launch-overhead remark that
 * closes the S12 chapter: at small batch the GPU waits on the host between
 * kernel launches).  fa_decode_graph_create records num_calls paged decodes
 * -- typically one per layer -- into a graph; each call i has its own q[i],
 * k_cache[i], v_cache[i], o[i] and lse[i] (HOST arrays of device pointers;
 * lse itself may be NULL for no LSE output), and all share block_table,
 * seq_lens, the sizes, num_splits, scale and the workspace exactly as in
 * fa_paged_decode (whose validation applies to every call).  Nothing runs at
 * creation.  fa_decode_graph_launch replays the step on `stream`; the graph
 * keeps the device pointers it was built with, so between launches the caller
 * updates the buffers' contents (new queries, new cache rows, longer seq_lens
 * and table rows), never their addresses.  The caller owns every buffer and
 * must keep them alive while the graph exists; launches on one stream run in
 * order and share the workspace, launches on different streams must not
 * overlap.  Create and destroy are host calls that must not run inside
 * another stream capture.
 * Errors: FA_ERR_INVALID_ARG (including a NULL graph handle), any error of
 * fa_paged_decode for a call, FA_ERR_CUDA.
 */
typedef struct fa_decode_graph fa_decode_graph;
int fa_decode_graph_create(fa_decode_graph** graph, int num_calls, const void* const* q, const void* const* k_cache,
                           const void* const* v_cache, void* const* o, float* const* lse,
                           const int32_t* block_table, const int32_t* seq_lens, int B, int Hq, int Hkv, int d,
                           int block_size, int max_blocks, int num_blocks, int num_splits, float scale,
                           void* workspace, size_t ws_bytes);
int fa_decode_graph_launch(fa_decode_graph* graph, void* stream);
/* Number of kernel launches one fa_decode_graph_launch replays (0 for NULL). */
int fa_decode_graph_kernel_count(const fa_decode_graph* graph);
void fa_decode_graph_destroy(fa_decode_graph* graph);

/*
 * fa_paged_decode without a caller workspace.  (The pages have no counterpart
 * to this entry point; it exists for callers of this library.)
 *
 * Some callers cannot allocate device memory where they decode: an
 * inference-engine plugin whose device memory is assigned by the engine ahead
 * of time and which may not allocate while it enqueues work, or a serving loop
 * that avoids cudaMalloc/cudaFree because they can synchronise the device.
 * This entry point takes the same arguments as fa_paged_decode minus the
 * workspace, and calls no allocating routine: the split partials live in a
 * fixed device array inside the library.
 *   Limit: B * Hq * num_splits (num_splits = 0 counts as 16) must be at most
 *   32768, else FA_ERR_UNSUPPORTED is returned and nothing is launched.  The
 *   array (16.25 MiB) is held on every device that loads the library until
 *   the process exits.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  A first call made while `stream` is being captured does not
 *   look the address up: it returns FA_ERR_CUDA, launches nothing and leaves
 *   the capture as it was.  The address is kept for the life of the process;
 *   after cudaDeviceReset on a device, do not call this entry point on that
 *   device again in the same process.
 *   All calls on a device share the array and it keeps the last call's
 *   contents (nothing in it needs clearing between calls).  Calls that overlap
 *   on the GPU -- on different streams, or from host threads without ordering
 *   between them -- race on the array and give undefined results.
 * Other errors as fa_paged_decode.
 */
int fa_paged_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_table,
                            const int32_t* seq_lens, void* o, float* lse, int B, int Hq, int Hkv, int d,
                            int block_size, int max_blocks, int num_blocks, int num_splits, float scale,
                            void* stream);

/*
 * Self-test of the library's failure detection: launches one CTA that waits on
 * a pipeline barrier nothing ever completes.  The bounded wait used by every
 * kernel gives up after `timeout_us` microseconds (1 .. 1,000,000), latches
 * FA_ERR_TIMEOUT in the device status word and the kernel ends normally; the
 * CUDA context stays usable.  Read the result with fa_get_device_status().
 * (Not an operation of the pages; it checks this library's error path.)
 */
int fa_selftest_wait_timeout(unsigned timeout_us, void* stream);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device: FA_OK, or the most severe condition latched since the
 * last call -- FA_ERR_OUT_OF_BOUNDS (debug builds), FA_ERR_CUDA (a kernel could
 * not set up its shared memory, or the query itself failed),
 * FA_ERR_INVALID_ARG (device-side offsets check), FA_ERR_TIMEOUT,
 * FA_ERR_BAD_BLOCK_TABLE.
 */
int fa_get_device_status(void* stream);

/*
 * 1 if this library was built with device bounds checks (FA_DEBUG), else 0.
 * In such a build every global load or store a kernel's threads issue is
 * checked against the extent of its buffer; an index outside it skips the
 * access and latches FA_ERR_OUT_OF_BOUNDS (read with fa_get_device_status).
 * TMA copies clip at the tensor edges by themselves.  The checks stand in for
 * a memory checker; release builds carry none of them.
 * (Not an operation of the pages; it checks this library.)
 */
int fa_debug_build(void);

/*
 * Self-test of the bounds checks: one thread asks the device guard about an
 * index past the end of a 3-element extent, without touching memory.  In a
 * debug build the status word then reads FA_ERR_OUT_OF_BOUNDS; in a release
 * build FA_OK.  (Not an operation of the pages.)
 */
int fa_selftest_bounds(void* stream);

/*
 * Failure injection for the backward pass (debug builds only): the next
 * launch of the backward's main kernel (fa_bwd or fa_bwd_varlen, any stream)
 * runs with every bounded pipeline wait limited to `timeout_us` microseconds
 * (1 .. 1,000,000), and the tensor-core issuing warp of the CTA that takes
 * work item `item` (>= 0; item 0 is always taken) stops issuing there, as if
 * it hung.  The waits that depend on it give up, FA_ERR_TIMEOUT is latched in
 * the device status word, every CTA ends normally and the context stays
 * usable; that call's gradients are undefined.  One-shot: the launch after it
 * runs normally.  Host-side state, not thread-safe.
 * Returns FA_OK once armed, FA_ERR_INVALID_ARG for arguments out of range,
 * FA_ERR_UNSUPPORTED in a release build (nothing armed).
 * (Not an operation of the pages; it tests this library's failure path.)
 */
int fa_debug_stall_backward(int item, unsigned timeout_us);

/*
 * Failure injection for the forward pass (debug builds only): the next
 * forward launch (fa_fwd, fa_fwd_ex, fa_fwd_block_sparse, fa_fwd_varlen or
 * fa_paged_prefill, any stream) runs with every bounded pipeline wait limited
 * to `timeout_us` microseconds (1 .. 1,000,000), and the tensor-core issuing
 * warp of the CTA with linear block index `cta` (blockIdx.x + gridDim.x *
 * (blockIdx.y + gridDim.y * blockIdx.z); CTA 0 holds the first head's longest
 * query-tile pair, or the first sequence's last one) issues nothing, as if it
 * hung.  The waits that depend on it give up, FA_ERR_TIMEOUT is latched in the
 * device status word, every CTA ends normally and the context stays usable;
 * that call's outputs are undefined.  One-shot; host-side state, not
 * thread-safe.  Returns FA_OK once armed, FA_ERR_INVALID_ARG for arguments out
 * of range, FA_ERR_UNSUPPORTED in a release build (nothing armed).
 * (Not an operation of the pages; it tests this library's failure path.)
 */
int fa_debug_stall_forward(int cta, unsigned timeout_us);

/*
 * Failure injection for paged decode (debug builds only): the next decode
 * launch (fa_paged_decode or fa_paged_decode_noalloc, any stream; a decode
 * graph created next captures it) runs with every bounded pipeline wait
 * limited to `timeout_us` microseconds (1 .. 1,000,000), and the TMA warp of
 * the split kernel's CTA with linear block index `cta` (split + splits *
 * (KV head + Hkv * sequence); CTA 0 is the first sequence's first split)
 * loads nothing, as if it hung.  Its consumers' waits give up,
 * FA_ERR_TIMEOUT is latched in the device status word, every CTA ends
 * normally and the context stays usable; that call's output is undefined.
 * One-shot; host-side state, not thread-safe.  Returns FA_OK once armed,
 * FA_ERR_INVALID_ARG for arguments out of range, FA_ERR_UNSUPPORTED in a
 * release build (nothing armed).
 * (Not an operation of the pages; it tests this library's failure path.)
 */
int fa_debug_stall_decode(int cta, unsigned timeout_us);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H_ */
