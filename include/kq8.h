/*
 * kq8.h -- C ABI of libkq8: q8-KV single-query decode attention on NVIDIA GB300
 * (sm_103a).
 *
 * Method sources (the three web pages the method is described on):
 *   [9-2]  article 9-2, "flash_attn_single_q_q8_neon -- single q, one pass over
 *          all KV": §1 one-pass online softmax; §2 the kernel's signature and
 *          its segments 1 (Q quantisation), 2 (int8 scores + online softmax),
 *          3 (final divide); §3 the two-pass alternative.
 *   [9-3]  article 9-3, "q8 KV precision comparison": §2 the write-path
 *          quantisation rule (kv_quantize_per_head).
 *   [10-1] article 10-1, "why long context must be sparse": §1 block probe +
 *          top-k + bounded exact attention; §2 the knobs and the gate.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is DEVICE memory owned by the caller, except the
 *     kq8_cache_t itself (a host struct read during the call) and the
 *     host-side outputs that are documented as such.  The library allocates
 *     nothing and keeps no state between calls.
 *   - Calls enqueue work on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and return without waiting for it.  Stream order holds as for
 *     ordinary launches.  The decode kernels and the appends are programmatic
 *     launches (cudaLaunchAttributeProgrammaticStreamSerialization): one of
 *     them may be scheduled while the kernel just before it on the stream
 *     finishes (this library's, or any code's that signals its dependents
 *     early).  Until that kernel has completed (griddepcontrol.wait) it writes
 *     no global memory and reads no cache, workspace or output; the exact
 *     decode may read its query, lengths and page ids early, but only as a
 *     guess that it uses once the same values, read again after the wait,
 *     agree (else it starts over from those).  In stream capture these
 *     launches become programmatic graph edges.
 *   - Return value: KQ8_OK (0) or a negative KQ8_ERR_* code.  On an error
 *     nothing was enqueued.  kq8_strerror() names a code.
 *   - Device-resident metadata (sequence lengths, page tables, write slots) is
 *     not visible to the host: kernels check it and, on a bad value, skip the
 *     affected work and OR a KQ8_STATUS_* bit into a status word (the first
 *     word of the workspace, or the `status` argument of kq8_append_kv).
 *     kq8_read_status() fetches and clears it.
 */
#ifndef KQ8_H
#define KQ8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* An opaque CUDA stream (cudaStream_t). */
typedef struct CUstream_st* kq8_stream_t;

enum {
    KQ8_OK = 0,
    KQ8_ERR_INVALID_ARG = -1, /* null/misaligned pointer, negative size, ... */
    KQ8_ERR_UNSUPPORTED = -2, /* shape outside what the kernels implement   */
    KQ8_ERR_WORKSPACE = -3,   /* workspace missing, misaligned or too small  */
    KQ8_ERR_CUDA = -4         /* a CUDA runtime call or launch failed        */
};

/* Status bits written by kernels into the status word. */
#define KQ8_STATUS_BAD_PAGE 0x1u    /* a page id outside [0, num_pages)        */
#define KQ8_STATUS_BAD_SEQLEN 0x2u  /* seq_len < 0 or > max_seq_len / pages   */
#define KQ8_STATUS_BAD_SLOT 0x4u    /* a write slot outside the pool          */
#define KQ8_STATUS_TIMEOUT 0x8u     /* a bounded wait on a copy ran out       */

/*
 * The paged q8 KV cache of one layer.  A pool of `num_pages` pages; page p holds
 * kv_bs consecutive tokens of one sequence for all `num_kv_heads` KV heads.
 *   k      : int8 [num_pages][nkv][kv_bs/32][hd/32][32][32]
 *            page p, head h, token row r, element i lives at
 *            ((p*nkv + h)*kv_bs*hd) + (r/32)*32*hd + (i/32)*1024 + kpos*32 + i%32
 *            with kpos = (r%32 % 4)*8 + (r%32)/4: each token's 32-element
 *            block is 32 contiguous bytes, the same block of a 32-token
 *            sub-tile is 1 KB contiguous, and rows 0, 4, 8, ... of a sub-tile
 *            are adjacent (a block probe every 4 rows reads whole lines).
 *   v      : int8 [num_pages][nkv][kv_bs][hd], token rows contiguous.
 *   kscale : float [num_pages][nkv][kv_bs], the row's max |k| (the stored
 *            scale of [9-3] §2; readers multiply by 1/127 as on [9-2] §2).
 *   vscale : float [num_pages][nkv][kv_bs], likewise for V.
 * The codes are the [9-3] §2 rule: round(x / (max|x| * (1/127))) clamped to
 * [-127, 127].  All four arrays must be 16-byte aligned.  Supported: head_dim
 * 128, kv_bs a multiple of 32 up to 256.
 */
typedef struct {
    int8_t* k;
    int8_t* v;
    float* kscale;
    float* vscale;
    int32_t num_pages;
    int32_t kv_bs;
    int32_t num_kv_heads;
    int32_t head_dim;
} kq8_cache_t;

/*
 * Write path ([9-3] §2, kv_quantize_per_head): quantise T new tokens of K and V
 * into the cache.
 *   k, v   : float [T][nkv][hd] (device).
 *   slot   : int32 [T] (device); token t goes to page slot[t] / kv_bs, row
 *            slot[t] % kv_bs.  slot < 0 skips the token; slot >= num_pages *
 *            kv_bs skips it and sets KQ8_STATUS_BAD_SLOT.
 *   status : optional uint32 word (device) receiving status bits; may be NULL.
 * Per (token, head): m = max_i |x_i| is stored as the scale; codes are
 * round(x / (m * (1/127))) clamped to [-127, 127] (round half away from zero,
 * IEEE division); an all-zero row stores 0 and zero codes.
 */
int kq8_append_kv(const kq8_cache_t* cache, const float* k, const float* v, const int32_t* slot,
                  int32_t T, uint32_t* status, kq8_stream_t stream);

/*
 * Bytes of workspace kq8_decode_attn needs for these sizes on the current
 * device.  The first 256 bytes hold the status word, the next 64 KB the
 * per-(sequence, KV head) chunk counters of the in-kernel merge; both must be
 * zero before the first call (kq8_workspace_init) and every completed call
 * leaves the counters at zero.  Re-initialise a workspace after a failed call.
 */
size_t kq8_decode_workspace_bytes(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len);

/*
 * The split kq8_decode_attn uses for these sizes on the current device:
 * *chunk_tiles 32-token tiles per CTA (a multiple of 4) and *num_chunks chunks
 * for a sequence of max_seq_len tokens.  A sequence split over several chunks
 * has its partial results merged by the last of its CTAs to finish, or, when
 * B * nkv exceeds the 16384 ticket counters, by a merge kernel launched after
 * the attention kernel.  Host pointers.
 */
int kq8_decode_plan(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len, int32_t* chunk_tiles,
                    int32_t* num_chunks);

/*
 * Clears the status word and the chunk counters of a workspace (one memset of
 * up to 64 KB + 256 bytes on `stream`).  Call once after allocating a
 * workspace: an uninitialised workspace gives wrong results.
 */
int kq8_workspace_init(void* workspace, size_t workspace_bytes, kq8_stream_t stream);

/*
 * Exact decode attention ([9-2] §1-§2): for every sequence b and query head h,
 *   out[b][h] = sum_t softmax_t(s_t) * V'_t   over t < seq_lens[b]
 * with s_t the [9-2] §2 score: Q quantised once to int8 in 32-element
 * max-abs blocks (truncating, [9-2] segment 1), int32 block dots with the
 * int8 K row, s = ((sum_b dot_b * qsc_b) * (kscale_t/127)) * scale; V'_t the
 * dequantised V row (code * vscale_t/127).  The softmax is evaluated online
 * (running max and sum, rescaled when the max grows) over KV chunks that are
 * merged by their log-sum-exp, with one divide per output at the end.
 *   out        : float [B][nq][hd] (device), written.
 *   q          : float [B][nq][hd] (device).
 *   page_table : int32 [B][max_pages] (device); page of tokens
 *                [j*kv_bs, (j+1)*kv_bs) of sequence b is page_table[b][j].
 *   seq_lens   : int32 [B] (device), each in [0, max_seq_len]; seq_len counts
 *                the token appended this step.  seq_len 0 gives out = 0.
 *   max_seq_len: host bound on seq_lens, <= max_pages * kv_bs.
 *   nq         : query heads; nq % nkv == 0 and G = nq / nkv in 1..8; query
 *                head h reads KV head h / G.
 *   scale      : the softmax scale (1/sqrt(hd) on the pages).
 *   workspace  : device scratch of >= kq8_decode_workspace_bytes(...) bytes,
 *                256-byte aligned, initialised once by kq8_workspace_init.
 * Calls sharing a workspace must not overlap on the GPU.
 */
int kq8_decode_attn(float* out, const float* q, const kq8_cache_t* cache,
                    const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                    int32_t max_seq_len, int32_t B, int32_t nq, float scale, void* workspace,
                    size_t workspace_bytes, kq8_stream_t stream);

/*
 * Allocation-free variant of kq8_decode_attn, for callers that may not allocate
 * device memory: code running inside another runtime's allocator or launch path
 * (a cudaMalloc there can re-enter that runtime, and it may synchronise the
 * device and stall every other stream), or serving loops that forbid device
 * allocation after start-up.  The method's pages have no counterpart: this is a
 * deployment convenience.
 * Same arguments and result as kq8_decode_attn, without the workspace: the
 * partials go to a scratch array of KQ8_NOALLOC_SCRATCH_BYTES compiled into the
 * library, which every GPU that loads the library's code holds until the
 * process exits.  Returns KQ8_ERR_WORKSPACE when these sizes need more scratch
 * than that (see kq8_decode_workspace_bytes).  Calls no cudaMalloc, cudaFree or
 * other allocating routine.
 * First call on a device: under CUDA's default lazy module loading
 * (CUDA_MODULE_LOADING=LAZY) the array is reserved only when the library's
 * code is first used on a device, which for a caller of this entry point alone
 * is this first call; it also looks up the array's device address (with that
 * device current) and caches it.  So the first call on each device may take
 * the 32 MiB of device memory and synchronise: make it at start-up, before any
 * stream capture.  Later calls only enqueue the kernel.
 * Every call uses the same array: calls that overlap on the GPU (other streams,
 * other threads, the same device) race and corrupt each other's results.
 * Outputs are unchecked: device-side checks (bad page ids or lengths, a timed
 * out copy wait) leave their status bits in the array where nobody reads them.
 * A caller that needs them uses kq8_decode_attn and kq8_read_status.
 */
#define KQ8_NOALLOC_SCRATCH_BYTES (32u << 20)
int kq8_decode_attn_noalloc(float* out, const float* q, const kq8_cache_t* cache,
                            const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                            int32_t max_seq_len, int32_t B, int32_t nq, float scale,
                            kq8_stream_t stream);

/*
 * Bytes of workspace kq8_sparse_decode_attn needs (>= 256).
 */
size_t kq8_sparse_decode_workspace_bytes(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len,
                                         int32_t block, int32_t topk);

/*
 * The split kq8_sparse_decode_attn uses for its bounded attention (as
 * kq8_decode_plan, for lists of up to G * topk blocks): a list's entries are
 * dealt out to its num_chunks chunks in turn, at most chunk_tiles each.
 */
int kq8_sparse_decode_plan(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len, int32_t block,
                           int32_t topk, int32_t* chunk_tiles, int32_t* num_chunks);

/*
 * Block-sparse decode attention ([10-1] §1-§2).  Per sequence the gate of
 * [10-1] §2 applies: seq_len <= 2*block runs the exact kernel above.  Otherwise,
 * per query head: the sequence is cut into nblk = ceil(seq_len/block) blocks;
 * block j is probed at tokens j*block + p*(block/probe), p < probe, that are
 * < seq_len; its score is the max of the [9-2] scores there ("max-dot
 * fusion"); the topk highest blocks are kept (equal scores: lower block index
 * first; topk >= nblk keeps all) and exact one-pass attention runs over their
 * tokens in ascending block order.  These probe/selection details are this
 * library's reading: the page describing the probe is not available.
 *   block      : positions per block, a multiple of 32 (32 on the page).
 *   topk       : blocks kept per query head, >= 1 (32 on the page).
 *   probe      : probes per block, 1 <= probe <= block (8 on the page).
 *   sel_blocks : optional int32 [B][nq][topk] (device): kept block ids in
 *                ascending order, -1 padded; all -1 for gated sequences.
 * Other arguments as kq8_decode_attn; workspace from
 * kq8_sparse_decode_workspace_bytes.
 */
int kq8_sparse_decode_attn(float* out, const float* q, const kq8_cache_t* cache,
                           const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t B, int32_t nq, float scale, int32_t block,
                           int32_t topk, int32_t probe, int32_t* sel_blocks, void* workspace,
                           size_t workspace_bytes, kq8_stream_t stream);

/*
 * Streaming form ([9-2] §3: the one-pass kernel can compute while KV arrives
 * piece by piece).  A running state per (sequence, query head) is kept in
 * caller memory between calls: state_acc float [rows][hd] (16-byte aligned)
 * and state_ms float [rows][2] (8-byte aligned), rows = B * nq in the layout
 * of `out`.  Its contents are this library's unnormalised online-softmax state
 * (running max of the scores, running sum, accumulator);
 * treat them as opaque.
 *   kq8_state_reset        : makes every row empty.
 *   kq8_decode_attn_update : attends tokens [seq_begin[b], seq_end[b]) of each
 *                            sequence (seq_begin optional: NULL = 0; each in
 *                            [0, seq_end[b]], else KQ8_STATUS_BAD_SEQLEN and the
 *                            sequence is skipped) and folds the result into the
 *                            state by its log-sum-exp.  Other arguments as
 *                            kq8_decode_attn (workspace from
 *                            kq8_decode_workspace_bytes).  Feeding a sequence in
 *                            pieces gives the one-call result up to rounding.
 *                            max_range_len (host): an upper bound on
 *                            seq_end[b] - seq_begin[b], used to split the ranges
 *                            over enough CTAs; 0 = max_seq_len.  A range longer
 *                            than the bound sets KQ8_STATUS_BAD_SEQLEN and that
 *                            sequence is skipped.
 *   kq8_state_finalize     : out = acc / sum per row (0 for an empty row).
 */
int kq8_state_reset(float* state_acc, float* state_ms, int32_t rows, kq8_stream_t stream);
int kq8_decode_attn_update(float* state_acc, float* state_ms, const float* q,
                           const kq8_cache_t* cache, const int32_t* page_table, int32_t max_pages,
                           const int32_t* seq_begin, const int32_t* seq_end, int32_t max_seq_len,
                           int32_t max_range_len, int32_t B, int32_t nq, float scale,
                           void* workspace, size_t workspace_bytes, kq8_stream_t stream);
int kq8_state_finalize(float* out, const float* state_acc, const float* state_ms, int32_t rows,
                       kq8_stream_t stream);

/*
 * Merge of running states computed elsewhere ([9-2] §3: the one pass lets KV
 * arrive piece by piece; the pieces may as well be attended by different
 * devices or processes, each holding a range of one sequence's tokens).
 * Folds `parts` partial states into the running state (state_acc, state_ms,
 * as above), in order, by their log-sum-exp: with M the larger of the two
 * running maxima, both sums and accumulators are scaled by e^(their max - M)
 * and added.  Each partial is a state in this library's format, e.g. made by
 * kq8_state_reset + kq8_decode_attn_update over one token range and copied
 * from another device; an empty partial changes nothing.
 *   part_acc : float [parts][rows][hd] (device).
 *   part_ms  : float [parts][rows][2] (device, 8-byte aligned).
 * Merging the states of a split of a sequence's tokens gives the state of the
 * whole range up to rounding (the result does not depend on the split, as
 * for kq8_decode_attn_update pieces).  One block of hd threads per row.
 */
int kq8_state_merge(float* state_acc, float* state_ms, const float* part_acc,
                    const float* part_ms, int32_t parts, int32_t rows, kq8_stream_t stream);

/*
 * Block-sparse decode with one selection per KV head: the G query heads of a
 * KV head keep the same top-k blocks, so the bounded attention reads each kept
 * block once for all of them.  Not on the pages (their selection is per query
 * head, kq8_sparse_decode_attn); this library's reading: the group's score of a
 * block is the max over its G query heads of their block scores, one top-k on
 * that (ties to the lower block), then each head runs the one pass over those
 * blocks.  Arguments, gate, workspace (kq8_sparse_decode_workspace_bytes) and
 * status as kq8_sparse_decode_attn; sel_blocks repeats the group's selection
 * for each of its query heads.
 */
int kq8_sparse_decode_attn_shared(float* out, const float* q, const kq8_cache_t* cache,
                                  const int32_t* page_table, int32_t max_pages,
                                  const int32_t* seq_lens, int32_t max_seq_len, int32_t B,
                                  int32_t nq, float scale, int32_t block, int32_t topk,
                                  int32_t probe, int32_t* sel_blocks, void* workspace,
                                  size_t workspace_bytes, kq8_stream_t stream);

/*
 * Batched causal prefill attention over the q8 cache ([10-1] §1: a batch of nb
 * new tokens scores against the whole history, O(nb*n); §2: the exact batched
 * kernel of the prefill gate).  Reading (the page gives no formula for the
 * batched kernel): each new token is one decode query of [9-2] §2 over the
 * tokens up to and including itself.
 *   out, q      : float [total_q][nq][128] (device, 16-byte aligned); the new
 *                 tokens' queries packed by sequence: sequence b owns rows
 *                 q_offsets[b] .. q_offsets[b+1]-1.
 *   q_offsets   : int32 [B+1] (device), non-decreasing, q_offsets[B] <= total_q.
 *   seq_lens    : int32 [B] (device): tokens in the cache for sequence b,
 *                 INCLUDING its nb_b = q_offsets[b+1] - q_offsets[b] new ones
 *                 (append them with kq8_append_kv first).  New token i sits at
 *                 position seq_lens[b] - nb_b + i and attends tokens 0 .. that
 *                 position.
 *   max_seq_len, max_q_len : host bounds on seq_lens[b] and nb_b (grid size).
 *   cache, page_table, max_pages, scale : as kq8_decode_attn.
 *   workspace   : >= kq8_prefill_workspace_bytes(...) bytes, 256-byte aligned,
 *                 its status word cleared by kq8_workspace_init.
 * A sequence whose bounds are inconsistent (nb_b > seq_lens[b], seq_lens[b] >
 * max_seq_len, nb_b > max_q_len, rows outside total_q) sets
 * KQ8_STATUS_BAD_SEQLEN and is skipped (its outputs are not written); a page
 * id outside the pool sets KQ8_STATUS_BAD_PAGE and its 32-token sub-tiles are
 * left out.  Results match one kq8_decode_attn per new token to fp32
 * rounding.  Runs on the tcgen05 tensor cores: 128 (token, query head) rows
 * per CTA, exact integer block dots in fp32 TMEM accumulators.
 */
size_t kq8_prefill_workspace_bytes(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len,
                                   int32_t max_q_len);
int kq8_prefill_attn(float* out, const float* q, int32_t total_q, const kq8_cache_t* cache,
                     const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len, int32_t B,
                     int32_t nq, float scale, void* workspace, size_t workspace_bytes,
                     kq8_stream_t stream);

/*
 * Block-sparse batched prefill ([10-1] §1: the sparse prefill costs
 * O(nb*k*block) instead of O(nb*n); §2: the prefill gate).  Reading: each new
 * token is one block-sparse decode query (kq8_sparse_decode_attn) over the
 * tokens up to and including itself, the gate seq_len <= 2*block applied per
 * token to that prefix length; selection stays per query head.
 * Arguments as kq8_prefill_attn plus block, topk, probe and sel_blocks
 * (optional int32 [total_q][nq][topk], -1 padded) as kq8_sparse_decode_attn;
 * total_q <= 65535 rows per call.  Rows outside every sequence are written as
 * zeros; the rows of an inconsistent sequence set KQ8_STATUS_BAD_SEQLEN.
 * workspace: kq8_sparse_prefill_workspace_bytes(total_q, ...) bytes, status
 * word cleared by kq8_workspace_init.
 */
size_t kq8_sparse_prefill_workspace_bytes(int32_t total_q, int32_t nq, int32_t nkv,
                                          int32_t max_seq_len, int32_t block, int32_t topk);
int kq8_sparse_prefill_attn(float* out, const float* q, int32_t total_q, const kq8_cache_t* cache,
                            const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                            const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len,
                            int32_t B, int32_t nq, float scale, int32_t block, int32_t topk,
                            int32_t probe, int32_t* sel_blocks, void* workspace,
                            size_t workspace_bytes, kq8_stream_t stream);

/*
 * q4 KV cache ([10-1] §2 names the --kv-q4 switch and keeps it out of the
 * block-sparse path; no page gives the format).  Reading: the q8 write rule of
 * [9-3] §2 with 7 levels a side -- per (token, head) m = max|x| is stored,
 * codes round(x / (m * (1/7))) clamped to [-7, 7] -- and readers multiply the
 * stored max by 1/7; Q is quantised to int8 exactly as in kq8_decode_attn.
 * A q4 cache uses the same kq8_cache_t with half-size code arrays, per
 * (page, head): K kv_bs/32 sub-tiles of 2 KB = [4 blocks][32 positions (as
 * for q8)][16 B], V [kv_bs][64 B]; codes are 4-bit offset binary (code + 8),
 * and in every 4-byte word of a row byte i holds element i (low nibble) and
 * element i + 4 (high nibble).  k and v point to num_pages * nkv * kv_bs * 64
 * bytes each; kscale and vscale as for q8.
 *   kq8_append_kv_q4   : as kq8_append_kv, writing q4 codes.
 *   kq8_decode_attn_q4 : exact decode over a q4 cache, arguments, workspace
 *                        (kq8_decode_workspace_bytes) and status as
 *                        kq8_decode_attn.  There is no q4 block-sparse call.
 */
int kq8_append_kv_q4(const kq8_cache_t* cache, const float* k, const float* v,
                     const int32_t* slot, int32_t T, uint32_t* status, kq8_stream_t stream);
int kq8_decode_attn_q4(float* out, const float* q, const kq8_cache_t* cache,
                       const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                       int32_t max_seq_len, int32_t B, int32_t nq, float scale, void* workspace,
                       size_t workspace_bytes, kq8_stream_t stream);

/*
 * Copies the status word of `workspace` (or of a kq8_append_kv status word) to
 * *status (host), then clears it; synchronises `stream`.
 */
int kq8_read_status(void* status_word, uint32_t* status, kq8_stream_t stream);

/* Text for a KQ8_* return code. */
const char* kq8_strerror(int code);

/* Library version, major*10000 + minor*100 + patch. */
int kq8_version(void);

/* ---- test-only exports: the hot path's building blocks, for bit-exact checks ---- */

/* Q quantisation of [9-2] segment 1 for `rows` rows of hd floats:
 * qi int8 [rows][hd], qsc float [rows][hd/32] (device). */
int kq8_debug_quantize_q(int8_t* qi, float* qsc, const float* q, int32_t rows, int32_t hd,
                         kq8_stream_t stream);

/* int32 block dots of every token with every query head ([9-2] segment 2):
 * dots int32 [B][nq][max_seq_len][hd/32] (device); entries t >= seq_lens[b]
 * are left untouched. */
int kq8_debug_block_dots(int32_t* dots, const float* q, const kq8_cache_t* cache,
                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                         int32_t max_seq_len, int32_t B, int32_t nq, kq8_stream_t stream);

/* The sparse path's block scores float [B][nq][ceil(max_seq_len/block)] (device),
 * as the probe kernel computes them (entries of gated sequences and of blocks
 * >= nblk are left untouched). */
int kq8_debug_probe_scores(float* scores, const float* q, const kq8_cache_t* cache,
                           const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t B, int32_t nq, float scale, int32_t block,
                           int32_t probe, kq8_stream_t stream);

/* Failure-detection hook: kq8_prefill_attn with the bulk copy of raw
 * 32-token sub-tile `withhold_sub` (>= 0, counted from position 0 of each
 * CTA's walk) never issued, so the bounded wait on it runs out (2^28 SM clocks)
 * in every CTA that reaches it.  Such a CTA sets KQ8_STATUS_TIMEOUT, lets its
 * other copies and MMAs finish (bounded), frees its tensor memory and leaves
 * its rows unwritten; the context stays usable.  Returns as kq8_prefill_attn;
 * KQ8_ERR_INVALID_ARG for withhold_sub < 0. */
int kq8_debug_prefill_withhold(float* out, const float* q, int32_t total_q,
                               const kq8_cache_t* cache, const int32_t* page_table,
                               int32_t max_pages, const int32_t* seq_lens,
                               const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len,
                               int32_t B, int32_t nq, float scale, void* workspace,
                               size_t workspace_bytes, int32_t withhold_sub,
                               kq8_stream_t stream);

/* Failure-detection hook: kq8_decode_attn with the bulk copy of the tile at
 * index `withhold_tile` (>= 0) of every warp's walk never issued (each warp of
 * a CTA walks every fourth 32-token tile of its chunk; index 0 is its first).
 * The bounded wait on it runs out (2^28 SM clocks) in every warp whose walk is
 * that long; the warp lets its other copies land (bounded) and its CTA sets
 * KQ8_STATUS_TIMEOUT and writes no result, so the rows of every (sequence, KV
 * head) that had such a CTA are left as they were; the other rows are exact
 * and the context stays usable.  Arguments and workspace as kq8_decode_attn
 * (G = nq / nkv in {1, 2, 4, 8}); KQ8_ERR_INVALID_ARG for withhold_tile < 0. */
int kq8_debug_decode_withhold(float* out, const float* q, const kq8_cache_t* cache,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* seq_lens, int32_t max_seq_len, int32_t B, int32_t nq,
                              float scale, void* workspace, size_t workspace_bytes,
                              int32_t withhold_tile, kq8_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KQ8_H */
