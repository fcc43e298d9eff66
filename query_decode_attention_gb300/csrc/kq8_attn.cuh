// kq8_attn.cuh -- the split-KV one-pass attention kernel and the chunk merge.
//
// Work decomposition: CTA = (KV chunk, KV head h, sequence b), 4 warps.  A
// chunk is a run of `chunk_tiles` 32-token sub-tiles (a sparse list deals its
// entries out to the chunks in turn, see list_chunks); warp w of the CTA takes
// the chunk's tiles w, w+4, ...  All G query heads of KV head h are handled by
// the same warp, so each K/V byte is read from HBM once for the whole group.
//
// Per warp, a ring of ATTN_STAGES shared-memory stages is filled by bulk and
// tensor copies (one lane issues them; completion on an mbarrier per stage)
// while the warp computes on the previous stage.  The page ids of the warp's
// tiles are fetched once, one per lane, so issuing a copy never waits on
// memory.  The kernel is a programmatic launch: its prologue (Q quantisation,
// page ids, barriers) may overlap the kernel before it on the stream, and the
// first copy waits for that kernel's completion (griddepcontrol.wait).  Per
// tile:
//   score phase (lane = token): int32 block dots of the token's K row with
//     the G int8 query rows (dp4a), the fp32 score in the method's order on
//     pairs of heads (packed fp32 ops, each lane still rounded separately, so
//     every score is the method's fp32 score bit for bit); a warp vote checks
//     whether any weight e^(s - M) would exceed 2^RESCALE_SLACK and only then
//     reduces the tile max and rescales the warp's state (the online-softmax
//     rescale of article 9-2 §1, done lazily: between rescales the weights may
//     exceed 1 by at most 2^8, which fp32 absorbs); w = e^(s - M), the
//     difference taken before the move to base 2;
//   value phase on the tensor cores (mma.sync m16n8k16, fp16 in, fp32
//     accumulate): the tile's weights times the V step, as fp16 hi + lo rows
//     of an A operand (one head per row pair), times the V codes, converted
//     exactly to fp16 after a transposed ldmatrix of the tensor-copied,
//     swizzled V sub-tile (q8: 128-byte rows; q4: 64-byte rows of nibbles).
// The 4 warps' (M, S, acc) are merged in shared memory; a chunk that covers
// the whole sequence writes out = acc / S directly, others write an
// unnormalised partial (M, S, acc), and the last of a sequence's chunk CTAs to
// finish (an atomic ticket per (sequence, KV head)) combines them by their
// log-sum-exp -- the same algebra as the online rescale.  Without ticket
// counters (very large batches) kq8_merge_kernel does that step instead.
//
// Every wait on a copy is bounded and decided for the whole warp at once.  A
// CTA in which a wait ran out sets KQ8_STATUS_TIMEOUT and writes no result:
// a single-chunk row is left as it was, and a partial is marked failed
// (S = -1) so that the merge leaves the row as it was too.
#pragma once

#include "kq8_common.cuh"

namespace kq8 {

constexpr int ATTN_WARPS = 4;
constexpr int ATTN_THREADS = ATTN_WARPS * 32;
constexpr int ATTN_STAGES = 2;
constexpr int MAX_WARP_TILES = 32;     // tiles per warp per chunk, one per lane
constexpr int MAX_CHUNK_TILES = ATTN_WARPS * MAX_WARP_TILES;
constexpr float LOG2E = 1.4426950408889634f;
// Lazy rescale: between rescales a weight stays below 2^RESCALE_SLACK.
constexpr float RESCALE_SLACK = 8.0f;

struct AttnParams {
    // V sub-tiles as a 3-D tensor {row bytes, kv_bs rows, num_pages * nkv}, copied
    // into shared memory with the 128-byte (q8: 128-byte rows) or 64-byte (q4:
    // 64-byte rows) swizzle, so that the value phase's ldmatrix is conflict-free
    CUtensorMap vmap;
    float* out;
    const float* q;
    kq8_cache_t cache;
    const int32_t* page_table;
    int32_t max_pages;
    const int32_t* seq_lens;
    int32_t max_seq_len;
    int32_t B, nq;
    float scale;
    int32_t chunk_tiles;   // multiple of ATTN_WARPS, <= MAX_CHUNK_TILES
    int32_t num_chunks;    // grid.x
    float* part_acc;       // [B][nq][num_chunks][HD]
    float2* part_ms;       // [B][nq][num_chunks] (M in score units, S)
    uint32_t* status;
    uint32_t* counters;    // [B][nkv] chunk tickets, zero between calls; null: merge kernel
    // streaming form (exact mode only): attend tokens [seq_begin[b], seq_lens[b])
    // and fold the result into a caller-held running state instead of `out`
    const int32_t* seq_begin;  // optional [B]
    float* state_acc;          // optional [B][nq][HD] unnormalised accumulator
    float2* state_ms;          // optional [B][nq] (running max, running sum)
    // block-sparse tile lists (SPARSE only): entry = tile | head_mask << 24
    const int32_t* tile_list;  // [B][nkv][list_cap]
    const int32_t* list_len;   // [B][nkv]
    int32_t list_cap;
    // optional [B]: the page-table row of each row b (prefill: the query
    // token's sequence); null = row b
    const int32_t* row_seq;
    // failure-detection hook (WITHHOLD kernels only): the copy of the tile at
    // this index of every warp's walk is never issued, so its wait runs out
    int32_t withhold;
};

template <int G>
struct AttnShape {
    static constexpr int GP = (G + 1) / 2;       // head pairs
    static constexpr int MIN_CTAS = (G <= 4) ? 3 : 2;
};

template <int G>
struct AttnSmem {
    // per warp and stage: a V sub-tile (swizzled by the tensor copy, so
    // 1024-byte aligned; q4 uses its first 2 KB), a K sub-tile, the scales
    alignas(1024) uint8_t v[ATTN_WARPS][ATTN_STAGES][SUB_V_BYTES];
    alignas(128) uint8_t k[ATTN_WARPS][ATTN_STAGES][SUB_K_BYTES];
    alignas(16) float sc[ATTN_WARPS][ATTN_STAGES][2][TILE];  // kscale, vscale
    // the tile's weights as fp16 (hi, lo) pairs per (head, token slot sigma(t)),
    // rows padded to 36 words so the eight heads' fragment loads hit distinct banks
    alignas(16) uint32_t pw[ATTN_WARPS][G][TILE + 4];
    alignas(16) int8_t qi[G][HD];
    alignas(16) float qsc[G][NB];
    int qsum[G][NB];  // -8 x the sum of each 32-element block's Q codes (q4 cache only)
    alignas(8) uint64_t bar[ATTN_WARPS][ATTN_STAGES];
    int last;  // this CTA drew the last ticket of its (sequence, KV head)
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// e^(a - b) for two scores: the difference is taken first (exact whenever a and
// b are close, else rounded relative to it), and only then moved to base 2, so
// the result does not depend on how large the scores themselves are.
__device__ __forceinline__ float exp_diff(float a, float b) { return ex2((a - b) * LOG2E); }

// Four int8 codes in one word -> two float pairs, exactly: flip the sign bits
// (offset binary u = c + 128), drop each byte into the mantissa of 2^23 with a
// byte permute and subtract 2^23 + 128 with one packed add per pair.
__device__ __forceinline__ void i8x4_to_f2(uint32_t w, float2& a, float2& b) {
    const uint32_t u = w ^ 0x80808080u;
    const float2 bias = make_float2(-8388736.0f, -8388736.0f);
    a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7540)),
                               __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7541))),
                   bias);
    b = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7542)),
                               __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7543))),
                   bias);
}

// q4 word (8 offset-binary nibbles, elements 0-3 low, 4-7 high) -> four
// float pairs, exactly: each nibble u = c + 8 into the mantissa of 2^23, one
// packed subtract of 2^23 + 8 per pair.
__device__ __forceinline__ void u4x8_to_f2(uint32_t w, float2& a, float2& b, float2& c,
                                           float2& d) {
    const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
    const float2 bias = make_float2(-8388616.0f, -8388616.0f);
    a = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7540)),
                               __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7541))),
                   bias);
    b = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7542)),
                               __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7543))),
                   bias);
    c = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7540)),
                               __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7541))),
                   bias);
    d = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7542)),
                               __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7543))),
                   bias);
}
// Unsigned bytes of a times signed bytes of b, summed into c.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Two int32 dots (|d| < 2^22) -> a float pair, exactly.
__device__ __forceinline__ float2 i2f_pair(int d0, int d1) {
    return __fadd2_rn(make_float2(__int_as_float(0x4B400000 + d0), __int_as_float(0x4B400000 + d1)),
                      make_float2(-12582912.0f, -12582912.0f));
}

// The tokens of sequence b one call attends: [begin, n), as list entries
// (tiles) starting at tile first_tile; bad lengths/starts give an empty range.
struct SeqRange {
    int n, begin, first_tile, entries;
    bool bad;
};
template <bool SPARSE>
__device__ __forceinline__ SeqRange seq_range(const AttnParams& P, int b, int h, int raw_len,
                                              int raw_begin) {
    SeqRange r;
    // a sparse list's length is loaded with the sequence length, not after it
    const int list_len = SPARSE ? P.list_len[b * P.cache.num_kv_heads + h] : 0;
    r.n = (raw_len < 0 || raw_len > P.max_seq_len) ? -1 : raw_len;
    r.bad = r.n < 0;
    if (r.bad) r.n = 0;
    r.begin = 0;
    if (!SPARSE && P.seq_begin) {
        r.begin = raw_begin;
        if (r.begin < 0 || r.begin > r.n) {
            r.bad = true;
            r.begin = r.n;
        }
    }
    r.first_tile = r.begin / TILE;
    if (r.n == r.begin)
        r.entries = 0;
    else if (SPARSE)
        r.entries = list_len;
    else
        r.entries = (r.n + TILE - 1) / TILE - r.first_tile;
    if (r.entries > P.num_chunks * P.chunk_tiles) {  // longer than the plan's grid covers
        r.bad = true;
        r.entries = 0;
    }
    return r;
}
// The chunks of a list and their entries.  An exact walk's chunk c holds the
// run of chunk_tiles entries from c * chunk_tiles.  A sparse list's length is
// known only once the selection has run, so its entries are dealt out in turn:
// chunk c holds entries c, c + num_chunks, c + 2 num_chunks, ..., and every CTA
// the grid has for the list walks an even share of it.
template <bool SPARSE>
__device__ __forceinline__ int list_chunks(const AttnParams& P, int entries) {
    return SPARSE ? max(1, min(P.num_chunks, entries))
                  : max(1, (entries + P.chunk_tiles - 1) / P.chunk_tiles);
}
// list entry of the k-th entry of chunk c
template <bool SPARSE>
__device__ __forceinline__ int list_entry(const AttnParams& P, int c, int k) {
    return SPARSE ? c + P.num_chunks * k : c * P.chunk_tiles + k;
}
// entries of chunk c
template <bool SPARSE>
__device__ __forceinline__ int chunk_entries(const AttnParams& P, int c, int entries) {
    return SPARSE ? (entries > c ? (entries - c + P.num_chunks - 1) / P.num_chunks : 0)
                  : max(0, min(P.chunk_tiles, entries - c * P.chunk_tiles));
}
template <bool SPARSE>
__device__ __forceinline__ SeqRange seq_range(const AttnParams& P, int b, int h) {
    return seq_range<SPARSE>(P, b, h, P.seq_lens[b], (!SPARSE && P.seq_begin) ? P.seq_begin[b] : 0);
}

// Folds a result (m, s, a) into a running state (mo, so, ao), maxima in score
// units: M = max, then both sides are scaled by e^(their max - M) and added.
__device__ __forceinline__ void fold_state(float mo, float so, float m, float s, float& M,
                                           float& S, float& fo, float& fn) {
    M = fmaxf(mo, m);
    fo = exp_diff(mo, M);
    fn = exp_diff(m, M);
    S = so * fo + s * fn;
}

// WITHHOLD: the failure-detection test build (P.withhold honoured); the
// production instantiations compile the check out.
template <int G, bool SPARSE, bool Q4 = false, bool WITHHOLD = false>
__global__ void __launch_bounds__(ATTN_THREADS, AttnShape<G>::MIN_CTAS)
    kq8_attn_kernel(const __grid_constant__ AttnParams P) {
    using Sh = AttnShape<G>;
    constexpr int GP = Sh::GP;
    constexpr int NS = ATTN_STAGES;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // the swizzled tensor copies want 1024-byte aligned V tiles: the launch
    // adds 1 KB of slack to round the base up
    AttnSmem<G>& S = *reinterpret_cast<AttnSmem<G>*>(
        smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    const int subs = kv_bs / TILE;
    // a programmatic launch after this one (the next append, update or layer)
    // may be scheduled now: each of those waits for this grid's completion
    // before it reads or writes global memory
    griddep_launch_dependents();
    // fetch the V tensor map's descriptor while the prologue runs
    if (threadIdx.x == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.vmap))
                     : "memory");
    // Until griddep_wait() returns, the kernel before this one on the stream
    // (this library's or any other code's, when it signals its dependents
    // early) may still be writing anything this kernel reads -- Q, the
    // lengths, the page table, the KV, the tile lists.  So before it this CTA
    // sets up its barriers and, on the exact walk without a row map, reads its
    // inputs only as a guess: after the wait the same inputs are read again,
    // and the walk goes on from the guess only if every value is the same
    // (else it drops what it began and starts over from the values read after
    // the wait).
    if (lane == 0)
        for (int s = 0; s < NS; s++) mbar_init(&S.bar[warp][s], 1);
    fence_barrier_init();
    __syncthreads();

    // The exact walk's list entry e is tile first + e (first: the tile of the
    // streamed start, else 0), so its page ids need no list: they are part of
    // the guess, loaded at the guessed start; a sparse walk's entries are
    // loaded with the length after the wait (its page ids follow them).  A row
    // map (row_seq) keeps its loads after the wait.  Not at G = 4:
    // there the walk sits at the 168 registers of three CTAs per SM, and with
    // these loads (guessed or only early) the serving step measured 0.3 %
    // slower than with the length first and the rest after it.
    constexpr bool EARLY = G != 4;
    constexpr int QR = (G + ATTN_WARPS - 1) / ATTN_WARPS;  // query rows per warp
    const bool guess = EARLY && !SPARSE && P.row_seq == nullptr;
    const int e_spec = list_entry<SPARSE>(P, chunk, warp + ATTN_WARPS * lane);
    const bool in_chunk = warp + ATTN_WARPS * lane < P.chunk_tiles;
    // L2-only loads (ld.global.cg): a guess must not leave a line in this SM's
    // L1 that the check after the wait could hit
    auto load_inputs = [&](float4 (&qv)[QR], int32_t& len, int32_t& beg) {
#pragma unroll
        for (int k = 0; k < QR; k++) {
            const int g = warp + k * ATTN_WARPS;
            if (g < G)
                qv[k] = __ldcg(reinterpret_cast<const float4*>(
                                   P.q + ((size_t)b * P.nq + (size_t)h * G + g) * HD) +
                               lane);
        }
        len = __ldcg(P.seq_lens + b);
        beg = (!SPARSE && P.seq_begin) ? __ldcg(P.seq_begin + b) : 0;
    };
    // the page id of this lane's entry for a walk that starts at token beg
    auto page_at = [&](int32_t beg) -> int32_t {
        const int t = max(beg, 0) / TILE + e_spec;
        if (!in_chunk || t / subs >= P.max_pages) return -1;
        return __ldcg(P.page_table + (size_t)b * P.max_pages + t / subs);
    };
    float4 qx[QR];  // the query rows the walk quantises
    int32_t tl_spec = 0;

    // ---- prologue: quantise the G query heads once (article 9-2 §2 seg. 1)
    auto quantise_q = [&]() {
#pragma unroll
        for (int k = 0; k < QR; k++) {
            const int g = warp + k * ATTN_WARPS;
            if (g >= G) continue;
            float qs;
            const uint32_t codes = quantize_q_lane(qx[k], qs);
            reinterpret_cast<uint32_t*>(S.qi[g])[lane] = codes;
            if ((lane & 7) == 0) S.qsc[g][lane >> 3] = qs;
            if (Q4) {  // q4: dot = sum q * (u - 8) = dp4a(u, q) - 8 * sum q per block
                int qs4 = __dp4a((int)codes, 0x01010101, 0);
                qs4 += __shfl_xor_sync(0xffffffffu, qs4, 1);
                qs4 += __shfl_xor_sync(0xffffffffu, qs4, 2);
                qs4 += __shfl_xor_sync(0xffffffffu, qs4, 4);
                if ((lane & 7) == 0) S.qsum[g][lane >> 3] = -8 * qs4;  // the dots' start value
            }
        }
    };
    // ---- the walk's plan from a length (and, on the plain exact walk, a page
    // id): this chunk's entries and this warp's tiles, one per lane
    SeqRange rng;
    int nch = 1, mine = 0, my_tile = 0;
    uint32_t my_mask = 0;
    int32_t my_page = -1;
    bool bad_page = false;
    auto plan = [&](int32_t len, int32_t beg, int32_t pg_pre, bool use_pre) {
        rng = seq_range<SPARSE>(P, b, h, len, beg);
        nch = list_chunks<SPARSE>(P, rng.entries);
        const int ce = chunk < nch ? chunk_entries<SPARSE>(P, chunk, rng.entries) : 0;
        mine = ce > warp ? (ce - warp + ATTN_WARPS - 1) / ATTN_WARPS : 0;
        my_tile = 0;
        my_mask = 0;
        my_page = -1;
        bad_page = false;
        if (lane < mine) {
            const int e = e_spec;
            if (SPARSE) {
                const int32_t v =
                    EARLY ? tl_spec : P.tile_list[(size_t)(b * nkv + h) * P.list_cap + e];
                my_tile = v & 0xFFFFFF;
                my_mask = (uint32_t)v >> 24;
            } else {
                my_tile = rng.first_tile + e;
                my_mask = 0xFFu;
            }
            const int32_t pg =
                use_pre ? pg_pre
                        : P.page_table[(size_t)(P.row_seq ? P.row_seq[b] : b) * P.max_pages +
                                     my_tile / subs];
            if (pg >= 0 && pg < P.cache.num_pages)
                my_page = pg;
            else
                bad_page = true;
        }
    };

    // all lanes call this (it shuffles); lane 0 issues the stage's copies
    auto issue = [&](int i) {
        const int tile = __shfl_sync(0xffffffffu, my_tile, i);
        const int32_t pg = __shfl_sync(0xffffffffu, my_page, i);
        if (WITHHOLD && i == P.withhold) return;  // test hook: the phase never completes
        if (lane == 0) {
            uint64_t* bar = &S.bar[warp][i % NS];
            const uint64_t pol = l2_evict_first_policy();  // every KV byte is read once
            if (pg < 0) {
                mbar_arrive_expect_tx(bar, 0);  // completes the phase with no data
            } else {
                const int sub = tile % subs;
                const int s = i % NS;
                const size_t so = scale_sub_off(pg, h, nkv, kv_bs, sub);
                if (Q4) {  // half-size codes
                    const size_t kvo = kv4_sub_off(pg, h, nkv, kv_bs, sub);
                    mbar_arrive_expect_tx(bar, SUB_K4_BYTES + SUB_V4_BYTES + 2 * SUB_S_BYTES);
                    bulk_g2s(S.k[warp][s], P.cache.k + kvo, SUB_K4_BYTES, bar, pol);
                    tma_load_3d(S.v[warp][s], &P.vmap, 0, sub * TILE, (int)page_head(pg, h, nkv),
                                bar, pol);
                } else {
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    bulk_g2s(S.k[warp][s], P.cache.k + kv_sub_off(pg, h, nkv, kv_bs, sub),
                             SUB_K_BYTES, bar, pol);
                    tma_load_3d(S.v[warp][s], &P.vmap, 0, sub * TILE, (int)page_head(pg, h, nkv),
                                bar, pol);
                }
                bulk_g2s(S.sc[warp][s][0], P.cache.kscale + so, SUB_S_BYTES, bar, pol);
                bulk_g2s(S.sc[warp][s][1], P.cache.vscale + so, SUB_S_BYTES, bar, pol);
            }
        }
    };
    // the guess: inputs, plan and Q's codes before the wait (no global writes)
    int32_t len_g = 0, beg_g = 0, pg_g = -1;
    if (guess) {
        load_inputs(qx, len_g, beg_g);
        pg_g = page_at(beg_g);
        plan(len_g, beg_g, pg_g, true);
        quantise_q();
        __syncthreads();  // the guessed Q codes, for every warp
    }
    griddep_wait();
    float4 qv[QR];  // after the wait: the check of the guess, or the inputs
    int32_t len_v = 0, beg_v = 0, pg_v = -1;
    if (guess) {
        // the page id at the guessed start: if the start is confirmed, it is the
        // page id the walk needs.  The check compares these with the guess once
        // the first copies are out.
        load_inputs(qv, len_v, beg_v);
        pg_v = page_at(beg_g);
    } else {
        load_inputs(qx, len_v, beg_v);
        if (EARLY && SPARSE && in_chunk && e_spec < P.list_cap)
            tl_spec = P.tile_list[(size_t)(b * nkv + h) * P.list_cap + e_spec];
        plan(len_v, beg_v, -1, false);
    }
    for (int i = 0; i < NS && i < mine; i++) issue(i);
    if (!guess) {
        // Q's codes while the first copies are in flight; every warp reads all heads'
        quantise_q();
        __syncthreads();
    }
    bool failed = false;
    // the check of the guess: the same inputs read after the wait
    auto guess_holds = [&]() {
        bool same = len_g == len_v && beg_g == beg_v && pg_g == pg_v;
#pragma unroll
        for (int k = 0; k < QR; k++)
            if (warp + k * ATTN_WARPS < G)
                same = same && __float_as_uint(qx[k].x) == __float_as_uint(qv[k].x) &&
                       __float_as_uint(qx[k].y) == __float_as_uint(qv[k].y) &&
                       __float_as_uint(qx[k].z) == __float_as_uint(qv[k].z) &&
                       __float_as_uint(qx[k].w) == __float_as_uint(qv[k].w);
        return __syncthreads_and(same) != 0;
    };
    if (guess) {
        if (!guess_holds()) {
            // let the copies issued from the guess land, re-arm the barriers and
            // start over from the values read after the wait
            bool landed = true;
            for (int i = 0; i < NS && i < mine; i++)
                landed = __all_sync(0xffffffffu, mbar_wait_bounded(&S.bar[warp][i], 0)) && landed;
            if (landed) {
                if (lane == 0)
                    for (int s = 0; s < NS; s++) {
                        mbar_inval(&S.bar[warp][s]);
                        mbar_init(&S.bar[warp][s], 1);
                    }
                fence_barrier_init();
                __syncwarp();
            }
#pragma unroll
            for (int k = 0; k < QR; k++) qx[k] = qv[k];
            plan(len_v, beg_v, -1, false);  // page ids read afresh
            if (landed) {
                for (int i = 0; i < NS && i < mine; i++) issue(i);
            } else {
                failed = true;  // a copy never landed: this warp walks nothing
                mine = 0;
            }
            quantise_q();
            __syncthreads();  // the new Q codes, for every warp
        }
    }
    const int gq = lane >> 2, c4 = lane & 3;  // mma fragment coordinates
    // stored K max -> step (1/127); the softmax scale is applied after it
    const float kstep = Q4 ? inv7() : inv127();

    float M2[G], Sl[G];
    // The value phase runs on the tensor cores: 16 m16n8 accumulator tiles D[.][.]
    // of 4 fp32 per lane, rows 0..7 = head (weight hi), 8..15 = head (weight lo).
    // q8: D[cg][0] holds elements 16cg + 2j, D[cg][1] 16cg + 2j + 1 (column j);
    // lane (g, c) then holds head g's elements 16cg + 4c .. + 3.  q4: for the
    // 32-element chunk q, D[2q + k/2][k%2] holds elements 32q + 8(j/2) + 2(j%2) +
    // {0, 1, 4, 5}[k]; lane (g, c) holds head g's elements 32q + 8c .. + 7.
    float D[HD / 16][2][4];
    // the weights go to the tensor cores as fp16 scaled by 2^-ev (see below)
    int ev;
    {  // the walk
        ev = -149;
#pragma unroll
        for (int g = 0; g < G; g++) {
            M2[g] = M_INIT;
            Sl[g] = 0.0f;
        }
#pragma unroll
        for (int cg = 0; cg < HD / 16; cg++)
#pragma unroll
            for (int j = 0; j < 4; j++) D[cg][0][j] = D[cg][1][j] = 0.0f;
        float2 qsc2[GP][NB];  // block scales of head pairs (2gp, 2gp+1)
#pragma unroll
        for (int gp = 0; gp < GP; gp++)
#pragma unroll
            for (int bb = 0; bb < NB; bb++)
                qsc2[gp][bb] = make_float2(S.qsc[2 * gp][bb], S.qsc[min(2 * gp + 1, G - 1)][bb]);

        int i = 0;
        for (; i < mine; i++) {
            const int tile = __shfl_sync(0xffffffffu, my_tile, i);
            const uint32_t mask = __shfl_sync(0xffffffffu, my_mask, i);
            const int32_t pg = __shfl_sync(0xffffffffu, my_page, i);
            // every lane waits (each needs the barrier's acquire of the copied
            // bytes); the warp gives up only together, so no lane is left behind
            // in a shuffle
            if (!__all_sync(0xffffffffu,
                            mbar_wait_bounded(&S.bar[warp][i % NS], (i / NS) & 1))) {
                failed = true;
                break;
            }
            if (pg >= 0) {
                const int st = i % NS;
                const int8_t* kst = reinterpret_cast<const int8_t*>(S.k[warp][st]);
                const int8_t* vst = reinterpret_cast<const int8_t*>(S.v[warp][st]);
                const float* kss = S.sc[warp][st][0];
                const float* vss = S.sc[warp][st][1];

                // ---- score phase: lane q reads K position q, i.e. token row
                // t = krow(q) of the tile, and scores it for all G heads
                const int q = lane;
                const int t = krow(q);
                const bool live = tile * TILE + t < rng.n && tile * TILE + t >= rng.begin;
                int dot[G][NB];
                const int hs = Q4 ? 0 : (q >> 2) & 1;  // half order: conflict-free loads
#pragma unroll
                for (int bb = 0; bb < NB; bb++) {
                    uint4 kA, kB;
                    if (Q4) {  // 16 B = 32 nibbles -> offset-binary bytes in element order
                        const uint4 kp = *reinterpret_cast<const uint4*>(kst + bb * 512 + q * 16);
                        kA = make_uint4(kp.x & 0x0F0F0F0Fu, (kp.x >> 4) & 0x0F0F0F0Fu,
                                        kp.y & 0x0F0F0F0Fu, (kp.y >> 4) & 0x0F0F0F0Fu);
                        kB = make_uint4(kp.z & 0x0F0F0F0Fu, (kp.z >> 4) & 0x0F0F0F0Fu,
                                        kp.w & 0x0F0F0F0Fu, (kp.w >> 4) & 0x0F0F0F0Fu);
                    } else {
                        kA = *reinterpret_cast<const uint4*>(kst + bb * 1024 + q * 32 + hs * 16);
                        kB = *reinterpret_cast<const uint4*>(kst + bb * 1024 + q * 32 +
                                                             (hs ^ 1) * 16);
                    }
#pragma unroll
                    for (int g = 0; g < G; g++) {
                        const uint4 qA =
                            *reinterpret_cast<const uint4*>(S.qi[g] + bb * 32 + hs * 16);
                        const uint4 qB =
                            *reinterpret_cast<const uint4*>(S.qi[g] + bb * 32 + (hs ^ 1) * 16);
                        int d;
                        if (Q4) {
                            d = dp4a_us(kA.x, qA.x, S.qsum[g][bb]);
                            d = dp4a_us(kA.y, qA.y, d);
                            d = dp4a_us(kA.z, qA.z, d);
                            d = dp4a_us(kA.w, qA.w, d);
                            d = dp4a_us(kB.x, qB.x, d);
                            d = dp4a_us(kB.y, qB.y, d);
                            d = dp4a_us(kB.z, qB.z, d);
                            d = dp4a_us(kB.w, qB.w, d);
                        } else {
                            d = __dp4a((int)kA.x, (int)qA.x, 0);
                            d = __dp4a((int)kA.y, (int)qA.y, d);
                            d = __dp4a((int)kA.z, (int)qA.z, d);
                            d = __dp4a((int)kA.w, (int)qA.w, d);
                            d = __dp4a((int)kB.x, (int)qB.x, d);
                            d = __dp4a((int)kB.y, (int)qB.y, d);
                            d = __dp4a((int)kB.z, (int)qB.z, d);
                            d = __dp4a((int)kB.w, (int)qB.w, d);
                        }
                        dot[g][bb] = d;
                    }
                }
                // s = (s * ks) * scale with ks = kscale / 127, each product rounded
                // as the method writes it, so every score equals the oracle's
                const float ks = __fmul_rn(kss[t], kstep);
                const float vstep = __fmul_rn(vss[t], Q4 ? inv7() : inv127());
                float sv[2 * GP];
#pragma unroll
                for (int gp = 0; gp < GP; gp++) {
                    const int g1 = min(2 * gp + 1, G - 1);
                    // s = sum_b dot_b * qsc_b in block order (the first add, 0 + x, is exact);
                    // the int32 dots are < 2^22 in magnitude, so the conversions are exact
                    float2 s = __fmul2_rn(make_float2(__int2float_rn(dot[2 * gp][0]),
                                                      __int2float_rn(dot[g1][0])),
                                          qsc2[gp][0]);
#pragma unroll
                    for (int bb = 1; bb < NB; bb++)
                        s = __fadd2_rn(s, __fmul2_rn(make_float2(__int2float_rn(dot[2 * gp][bb]),
                                                                 __int2float_rn(dot[g1][bb])),
                                                     qsc2[gp][bb]));
                    s = __fmul2_rn(__fmul2_rn(s, make_float2(ks, ks)), make_float2(P.scale, P.scale));
                    sv[2 * gp] = s.x;
                    sv[2 * gp + 1] = s.y;
                }
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const bool on = live && ((mask >> g) & 1u);
                    sv[g] = on ? sv[g] : -INFINITY;
                }
                // (s - M) * log2(e): the difference first, then base 2 (masked: -inf)
                float dd[2 * GP];
                bool grow = false;
#pragma unroll
                for (int gp = 0; gp < GP; gp++) {
                    const int g1 = min(2 * gp + 1, G - 1);
                    const float2 x = __fmul2_rn(
                        __fadd2_rn(make_float2(sv[2 * gp], sv[g1]), make_float2(-M2[2 * gp], -M2[g1])),
                        make_float2(LOG2E, LOG2E));
                    dd[2 * gp] = x.x;
                    dd[2 * gp + 1] = x.y;
                    grow |= x.x > RESCALE_SLACK || x.y > RESCALE_SLACK;
                }
                if (__any_sync(0xffffffffu, grow)) {
                    // rare: some head's maximum grew by a wide margin -> rescale its state
                    float cl = 1.0f;  // the factor of this lane's accumulator head gq
#pragma unroll
                    for (int g = 0; g < G; g++) {
                        const float mn = fmaxf(M2[g], warp_max(sv[g]));
                        if (mn > M2[g]) {
                            const float c = exp_diff(M2[g], mn);
                            Sl[g] *= c;
                            cl = (g == gq) ? c : cl;
                            M2[g] = mn;
                            dd[g] = (sv[g] - mn) * LOG2E;
                        }
                    }
#pragma unroll
                    for (int cg = 0; cg < HD / 16; cg++)
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            D[cg][0][j] *= cl;
                            D[cg][1][j] *= cl;
                        }
                }
                float w[2 * GP];
#pragma unroll
                for (int g = 0; g < G; g++) {
                    w[g] = ex2(dd[g]);  // masked: ex2(-inf) = 0
                    Sl[g] += w[g];
                }
                if constexpr ((G & 1) != 0) w[G] = 0.0f;
                {
                    // weights for the tensor cores: P' = w * vstep * 2^-ev as fp16 hi + lo
                    // (22 significant bits).  ev keeps the tile's largest live V step
                    // times 2^-ev below 2^7, so with w <= 2^8 (the lazy rescale bound)
                    // P' < 2^15, inside the fp16 range; a tile that needs a larger ev
                    // first scales the accumulators by the exact power of two 2^(old - new)
                    const uint32_t vb = __reduce_max_sync(
                        0xffffffffu, (live && mask != 0u) ? __float_as_uint(vstep) : 0u);
                    const int ve = (int)(vb >> 23) - 127;
                    if (vb != 0u && ve > ev + 6) {  // warp-uniform, rare
                        const int en = ve - 6;
                        const float f = (ev - en >= -126) ? pow2i(ev - en) : 0.0f;
#pragma unroll
                        for (int cg = 0; cg < HD / 16; cg++)
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                D[cg][0][j] *= f;
                                D[cg][1][j] *= f;
                            }
                        ev = en;
                    }
                    const int k1 = min(max(-ev, -126), 127);
                    const float vsc = __fmul_rn(__fmul_rn(vstep, pow2i(k1)),
                                                pow2i(min(max(-ev - k1, -126), 127)));
                    // token t's slot: sigma(t) = 8c + 4ks + 2h + j for t = 16ks + 8h + 2c + j,
                    // so the 8 tokens an mma lane (., c) needs are contiguous
                    const int slot = ((t >> 1) & 3) * 8 + (t >> 4) * 4 + ((t >> 3) & 1) * 2 + (t & 1);
#pragma unroll
                    for (int gp = 0; gp < GP; gp++) {
                        float2 pp = __fmul2_rn(make_float2(w[2 * gp], w[2 * gp + 1]),
                                               make_float2(vsc, vsc));
                        // masked tokens have w = 0; their (possibly stale) scale must not leak in
                        pp.x = (w[2 * gp] != 0.0f) ? pp.x : 0.0f;
                        pp.y = (w[2 * gp + 1] != 0.0f) ? pp.y : 0.0f;
                        const uint32_t hi = f2_to_h2(pp.x, pp.y);
                        const float2 hf = h2_to_f2(hi);
                        const float2 r = __fadd2_rn(pp, make_float2(-hf.x, -hf.y));  // exact
                        const uint32_t lo = f2_to_h2(r.x, r.y);
                        S.pw[warp][2 * gp][slot] = __byte_perm(hi, lo, 0x5410);
                        if (2 * gp + 1 < G) S.pw[warp][2 * gp + 1][slot] = __byte_perm(hi, lo, 0x7632);
                    }
                }
                __syncwarp();

                {
                    // ---- value phase on the tensor cores: D += P' (rows: heads hi | lo,
                    // k: 32 tokens) x V (k: tokens, n: elements), two m16n8k16 k-steps per
                    // 8-element n-tile.  A (this lane's head gq; zero rows for gq >= G):
                    // tokens 2c, 2c+1, 2c+8, 2c+9 | +16, from slots 8c .. 8c+7.
                    uint32_t a0[4] = {0u, 0u, 0u, 0u}, a1[4] = {0u, 0u, 0u, 0u};
                    if (gq < G) {
                        const uint4 x0 = *reinterpret_cast<const uint4*>(&S.pw[warp][gq][8 * c4]);
                        const uint4 x1 = *reinterpret_cast<const uint4*>(&S.pw[warp][gq][8 * c4 + 4]);
                        a0[0] = __byte_perm(x0.x, x0.y, 0x5410);  // hi of tokens 2c, 2c+1
                        a0[1] = __byte_perm(x0.x, x0.y, 0x7632);  // lo
                        a0[2] = __byte_perm(x0.z, x0.w, 0x5410);  // hi of 2c+8, 2c+9
                        a0[3] = __byte_perm(x0.z, x0.w, 0x7632);
                        a1[0] = __byte_perm(x1.x, x1.y, 0x5410);  // k-step 1: tokens + 16
                        a1[1] = __byte_perm(x1.x, x1.y, 0x7632);
                        a1[2] = __byte_perm(x1.z, x1.w, 0x5410);
                        a1[3] = __byte_perm(x1.z, x1.w, 0x7632);
                    }
                    if (Q4) {
                        // B (q4): per 16-byte chunk cq of a 64-byte row (32 elements), one
                        // transposed ldmatrix of the four 8-token blocks as 16-bit words
                        // (64-byte swizzle: chunk cq of row t at cq ^ ((t / 2) % 4)).
                        // Register i holds for tokens 8i + 2c and + 1 the bytes 2(g%2),
                        // 2(g%2) + 1 of word 4cq + g/2: elements e0 = 32cq + 8(g/2) + 2(g%2),
                        // e0 + 1 (low nibbles) and e0 + 4, e0 + 5 (high nibbles).  A low
                        // nibble u = code + 8 masked into the mantissa of 1024 gives 1024 + u,
                        // minus 1032; a high one gives 1024 + 16u, times 1/16 minus 72 (one
                        // fma): both exact.
                        const uint32_t vrow = smem_u32(vst) + (uint32_t)lane * (HD / 2);
#pragma unroll
                        for (int cq = 0; cq < HD / 32; cq++) {
                            uint32_t r[4];
                            ldsm_x4_trans(vrow + ((uint32_t)(cq ^ ((lane >> 1) & 3)) << 4), r[0],
                                          r[1], r[2], r[3]);
                            uint32_t b[4][4];  // [n-tile: +0, +1, +4, +5][register]
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                const uint32_t r8 = r[j] >> 8;  // bytes 1, 3 -> 0, 2
                                b[0][j] = hsub2(and_or(r[j], 0x000F000Fu, 0x64006400u), 0x64086408u);
                                b[1][j] = hsub2(and_or(r8, 0x000F000Fu, 0x64006400u), 0x64086408u);
                                b[2][j] = hfma2(and_or(r[j], 0x00F000F0u, 0x64006400u), 0x2C002C00u,
                                                0xD480D480u);
                                b[3][j] = hfma2(and_or(r8, 0x00F000F0u, 0x64006400u), 0x2C002C00u,
                                                0xD480D480u);
                            }
#pragma unroll
                            for (int k = 0; k < 4; k++) {
                                mma_f16_16816(D[2 * cq + (k >> 1)][k & 1], a0, b[k][0], b[k][1]);
                                mma_f16_16816(D[2 * cq + (k >> 1)][k & 1], a1, b[k][2], b[k][3]);
                            }
                        }
                    } else {
                        // B: per 16-byte chunk cg, one transposed ldmatrix of the four 8-token
                        // blocks as 16-bit element pairs: register i holds, for tokens 8i + 2c
                        // and + 1, elements 16cg + 2g and + 1.  Lane L gives token row L's
                        // chunk, at its 128-byte-swizzled place.
                        const uint32_t vrow = smem_u32(vst) + (uint32_t)lane * HD;
#pragma unroll
                        for (int cg = 0; cg < HD / 16; cg++) {
                            uint32_t r[4];
                            ldsm_x4_trans(vrow + ((uint32_t)(cg ^ (lane & 7)) << 4), r[0], r[1], r[2], r[3]);
                            // int8 pair -> fp16 pair exactly: offset binary u = c + 128 into the
                            // mantissa of 1024 (0x64uu), minus 1152
                            uint32_t be[4], bo[4];
#pragma unroll
                            for (int j = 0; j < 4; j++) {
                                const uint32_t u = r[j] ^ 0x80808080u;
                                be[j] = hsub2(__byte_perm(u, 0x64646464u, 0x4240), 0x64806480u);
                                bo[j] = hsub2(__byte_perm(u, 0x64646464u, 0x4341), 0x64806480u);
                            }
                            mma_f16_16816(D[cg][0], a0, be[0], be[1]);
                            mma_f16_16816(D[cg][0], a1, be[2], be[3]);
                            mma_f16_16816(D[cg][1], a0, bo[0], bo[1]);
                            mma_f16_16816(D[cg][1], a1, bo[2], bo[3]);
                        }
                    }
                }
            }
            __syncwarp();
            if (i + NS < mine) issue(i + NS);
        }
        if (failed) {
            if (lane == 0) atomicOr(P.status, KQ8_STATUS_TIMEOUT);
            // let the copies this warp still has in flight land before leaving
            for (int j = i; j < mine && j < i + NS; j++)
                __all_sync(0xffffffffu,
                           mbar_wait_bounded(&S.bar[warp][j % NS], (j / NS) & 1));
#pragma unroll
            for (int g = 0; g < G; g++) {
                M2[g] = M_INIT;
                Sl[g] = 0.0f;
            }
#pragma unroll
            for (int cg = 0; cg < HD / 16; cg++)
#pragma unroll
                for (int j = 0; j < 4; j++) D[cg][0][j] = D[cg][1][j] = 0.0f;
        }
    }
    // the inputs are settled: report bad values
    if (rng.bad && threadIdx.x == 0 && chunk == 0 && h == 0) atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
    if (bad_page) atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
    if (chunk >= nch) return;

#pragma unroll
    for (int g = 0; g < G; g++) Sl[g] = warp_sum(Sl[g]);

    // ---- merge the 4 warps in shared memory (reuses the V buffers)
    const bool cta_failed = __syncthreads_or(failed ? 1 : 0) != 0;
    float* macc = reinterpret_cast<float*>(S.v);                          // [W][G][HD]
    float2* mms = reinterpret_cast<float2*>(macc + ATTN_WARPS * G * HD);  // [W][G]
    if (gq < G) {
        // head gq's elements: the hi and lo rows added, and the weights' 2^-ev
        // scale undone (an exact power of two, in two steps)
        const int k1 = min(max(ev, -126), 127);
        const float f = pow2i(k1), f2 = pow2i(min(max(ev - k1, -126), 127));
        auto sum = [&](int t, int n, int j) { return (D[t][n][j] + D[t][n][j + 2]) * f * f2; };
        float* row = &macc[(warp * G + gq) * HD];
#pragma unroll
        for (int q = 0; q < HD / 32; q++) {
            float4 lo, hi;  // elements base .. base + 3 and base + 4 .. base + 7
            int base;
            if (Q4) {  // n-tiles +0, +1, +4, +5 of chunk q
                base = 32 * q + 8 * c4;
                lo = make_float4(sum(2 * q, 0, 0), sum(2 * q, 1, 0), sum(2 * q, 0, 1),
                                 sum(2 * q, 1, 1));
                hi = make_float4(sum(2 * q + 1, 0, 0), sum(2 * q + 1, 1, 0),
                                 sum(2 * q + 1, 0, 1), sum(2 * q + 1, 1, 1));
                *reinterpret_cast<float4*>(row + base) = lo;
                *reinterpret_cast<float4*>(row + base + 4) = hi;
            } else {  // 16-element chunks 2q and 2q + 1
#pragma unroll
                for (int cg = 2 * q; cg < 2 * q + 2; cg++)
                    *reinterpret_cast<float4*>(row + 16 * cg + 4 * c4) =
                        make_float4(sum(cg, 0, 0), sum(cg, 1, 0), sum(cg, 0, 1), sum(cg, 1, 1));
            }
        }
    }
    if (lane == 0)
#pragma unroll
        for (int g = 0; g < G; g++) mms[warp * G + g] = make_float2(M2[g], Sl[g]);
    __syncthreads();

    const int d = threadIdx.x;  // output element
    for (int g = 0; g < G; g++) {
        float mx = M_INIT;
#pragma unroll
        for (int w = 0; w < ATTN_WARPS; w++) mx = fmaxf(mx, mms[w * G + g].x);
        float ssum = 0.0f, a = 0.0f;
#pragma unroll
        for (int w = 0; w < ATTN_WARPS; w++) {
            const float2 ms = mms[w * G + g];
            const float f = exp_diff(ms.x, mx);
            ssum += ms.y * f;
            a += macc[(w * G + g) * HD + d] * f;
        }
        const size_t row = (size_t)b * P.nq + (size_t)h * G + g;
        if (nch == 1 && cta_failed) {
            // a timed-out walk: the row (or its running state) stays as it was
        } else if (nch == 1 && P.state_acc) {
            const float2 old = P.state_ms[row];
            float M, Sn, fo, fn;
            fold_state(old.x, old.y, mx, ssum, M, Sn, fo, fn);
            const float an = P.state_acc[row * HD + d] * fo + a * fn;
            __syncthreads();  // every thread has read the old state row
            P.state_acc[row * HD + d] = an;
            if (d == 0) P.state_ms[row] = make_float2(M, Sn);
        } else if (nch == 1) {
            P.out[row * HD + d] = (ssum > 0.0f) ? a / ssum : 0.0f;
        } else {
            const size_t pr = row * P.num_chunks + chunk;
            P.part_acc[pr * HD + d] = a;
            if (d == 0) P.part_ms[pr] = make_float2(mx, cta_failed ? -1.0f : ssum);
        }
    }
    if (nch == 1 || P.counters == nullptr) return;

    // ---- the last CTA of this (sequence, KV head) to finish merges the chunks
    //   M = max_c m_c, out = sum_c acc_c e^(m_c - M) / sum_c S_c e^(m_c - M)
    __syncthreads();  // every partial of this CTA is written
    if (threadIdx.x == 0) {
        // one fence after the CTA barrier orders all of them before the ticket
        // (a fence is cumulative over the writes that happen before it)
        __threadfence();
        const unsigned ticket = atomicAdd(&P.counters[b * nkv + h], 1u);
        S.last = (ticket == (unsigned)(nch - 1));
    }
    __syncthreads();
    if (!S.last) return;
    __threadfence();
    // one warp per query head, 4 output elements per lane, one online pass over
    // the chunks with their loads issued in batches
    for (int g = warp; g < G; g += ATTN_WARPS) {
        const size_t base = ((size_t)b * P.nq + (size_t)h * G + g) * P.num_chunks;
        float mx = M_INIT, ssum = 0.0f;
        float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        bool chunk_failed = false;
#pragma unroll 8
        for (int c = 0; c < nch; c++) {
            const float2 ms = __ldcg(&P.part_ms[base + c]);
            chunk_failed |= ms.y < 0.0f;
            const float4 x = __ldcg(reinterpret_cast<const float4*>(P.part_acc + (base + c) * HD) + lane);
            const float mn = fmaxf(mx, ms.x);
            const float fo = exp_diff(mx, mn), fn = exp_diff(ms.x, mn);
            ssum = ssum * fo + ms.y * fn;
            a.x = a.x * fo + x.x * fn;
            a.y = a.y * fo + x.y * fn;
            a.z = a.z * fo + x.z * fn;
            a.w = a.w * fo + x.w * fn;
            mx = mn;
        }
        const size_t row = (size_t)b * P.nq + (size_t)h * G + g;
        if (chunk_failed) {
            // some chunk's walk timed out: the row (or its state) stays as it was
        } else if (P.state_acc) {  // fold into the caller's running state (this warp owns the row)
            const float2 old = P.state_ms[row];
            float M, Sn, fo, fn;
            fold_state(old.x, old.y, mx, ssum, M, Sn, fo, fn);
            float4* sa = reinterpret_cast<float4*>(P.state_acc + row * HD) + lane;
            const float4 ao = *sa;
            __syncwarp();
            *sa = make_float4(ao.x * fo + a.x * fn, ao.y * fo + a.y * fn, ao.z * fo + a.z * fn,
                              ao.w * fo + a.w * fn);
            if (lane == 0) P.state_ms[row] = make_float2(M, Sn);
        } else {
            float4 o = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (ssum > 0.0f) o = make_float4(a.x / ssum, a.y / ssum, a.z / ssum, a.w / ssum);
            reinterpret_cast<float4*>(P.out + row * HD)[lane] = o;
        }
    }
    if (threadIdx.x == 0) P.counters[b * nkv + h] = 0;  // ready for the next call
}

// Combine the partials of sequences split over several chunks:
//   M = max_c m_c, out = sum_c acc_c e^(m_c - M) / sum_c S_c e^(m_c - M).
template <bool SPARSE>
__global__ void __launch_bounds__(HD) kq8_merge_kernel(const AttnParams P) {
    const int row = blockIdx.x;  // b * nq + hq
    const int b = row / P.nq, hq = row % P.nq;
    const int G = P.nq / P.cache.num_kv_heads;
    const int h = hq / G;
    const int entries = seq_range<SPARSE>(P, b, h).entries;
    const int nch = entries > 0 ? list_chunks<SPARSE>(P, entries) : 0;
    if (nch <= 1) return;
    const size_t base = (size_t)row * P.num_chunks;
    float mx = M_INIT;
    for (int c = 0; c < nch; c++) {
        if (P.part_ms[base + c].y < 0.0f) return;  // a timed-out chunk: row left as it was
        mx = fmaxf(mx, P.part_ms[base + c].x);
    }
    float ssum = 0.0f, a = 0.0f;
    for (int c = 0; c < nch; c++) {
        const float2 ms = P.part_ms[base + c];
        const float f = exp_diff(ms.x, mx);
        ssum += ms.y * f;
        a += P.part_acc[(base + c) * HD + threadIdx.x] * f;
    }
    if (P.state_acc) {
        const float2 old = P.state_ms[row];
        float M, Sn, fo, fn;
        fold_state(old.x, old.y, mx, ssum, M, Sn, fo, fn);
        const float an = P.state_acc[(size_t)row * HD + threadIdx.x] * fo + a * fn;
        __syncthreads();  // every thread has read the old state row
        P.state_acc[(size_t)row * HD + threadIdx.x] = an;
        if (threadIdx.x == 0) P.state_ms[row] = make_float2(M, Sn);
    } else {
        P.out[(size_t)row * HD + threadIdx.x] = (ssum > 0.0f) ? a / ssum : 0.0f;
    }
}

}  // namespace kq8
