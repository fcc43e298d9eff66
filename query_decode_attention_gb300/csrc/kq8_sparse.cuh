// kq8_sparse.cuh -- block-sparse decode (article 10-1 §1-§2): probe kernel,
// top-k selection and the per-KV-head union tile lists that the attention
// kernel then walks in SPARSE mode.
//
// Readings taken where the pages are silent (the page that details the
// probe is not available): probe p of block j reads token
// j*block + p*(block/probe) if < seq_len; the block score is the max of the
// one-pass scores there; per query head the topk highest blocks are kept,
// equal scores going to the lower block index; topk >= nblk keeps all;
// attention runs over the kept blocks in ascending order.
#pragma once

#include "kq8_common.cuh"

namespace kq8 {

struct SparseParams {
    const float* q;
    kq8_cache_t cache;
    const int32_t* page_table;
    int32_t max_pages;
    const int32_t* seq_lens;
    int32_t max_seq_len;
    int32_t B, nq;
    float scale;
    int32_t block, topk, probe;
    int32_t max_nblk;        // ceil(max_seq_len / block)
    int32_t probe_bpc;       // probe blocks per CTA (its pages fit PROBE_MAX_PAGES)
    float* scores;           // [B][nq][max_nblk]
    uint32_t* masks;         // [B][nkv][max_nblk]: bit g = head g kept the block
    int32_t* tile_list;      // [B][nkv][list_cap]
    int32_t* list_len;       // [B][nkv]
    int32_t list_cap;
    int32_t* sel_blocks;     // optional [B][nq][topk]
    uint32_t* status;
    const int32_t* row_seq;  // optional [B]: page-table row of row b (null = b)
    int32_t shared_sel;      // 1: one selection per KV head (max of its heads' block scores)
    uint32_t* tickets;       // [B][nkv], zero between calls; null: one top-k CTA per KV head
};

__device__ __forceinline__ int sparse_seq_len(const SparseParams& P, int b) {
    int n = P.seq_lens[b];
    if (n < 0 || n > P.max_seq_len) return -1;
    return n;
}

// ---------------------------------------------------------------------------
// Selection (top-k per query head, ties to the lower block) and the per-KV-head
// union tile list, as device functions of a 256-thread CTA: run either by the
// last probe CTA of a (sequence, KV head) to finish (fused, the usual path) or
// by kq8_topk_kernel (batches with more (sequence, KV head) pairs than ticket
// counters).
// ---------------------------------------------------------------------------
constexpr int TOPK_THREADS = 256;

// Order-preserving map of a float to uint32 (larger float -> larger key);
// -0 and +0 map to the same key, so ties follow float equality.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t u = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of v over 256 threads; returns the prefix
// and writes the total.  Uses `tmp` (>= 8 ints).
__device__ __forceinline__ int block_excl_scan(int v, int* tmp, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) tmp[warp] = x;
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < TOPK_THREADS / 32; w++) {
        const int t = tmp[w];
        if (w < warp) base += t;
        tot += t;
    }
    __syncthreads();
    total = tot;
    return base + x - v;
}

struct SelectSmem {
    int hist[256];
    int scan_tmp[TOPK_THREADS / 32];
    uint32_t prefix;
    int kk, cnt;
    int last;
};

// sel_blocks rows of heads [g_first, g_end) of (b, h) := -1
template <int G>
__device__ void clear_selection(const SparseParams& P, int b, int h, int g_first, int g_end) {
    if (!P.sel_blocks) return;
    for (int g = g_first; g < g_end; g++) {
        int32_t* sel = P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + g) * P.topk;
        for (int i = threadIdx.x; i < P.topk; i += TOPK_THREADS) sel[i] = -1;
    }
}

// The exact path of the gate (article 10-1 §2): every tile, every head.
template <int G>
__device__ void gated_list(const SparseParams& P, int b, int h, int n) {
    const int ntiles = (n + TILE - 1) / TILE;
    int32_t* list = P.tile_list + (size_t)(b * P.cache.num_kv_heads + h) * P.list_cap;
    const int32_t all = (int32_t)(((1u << G) - 1u) << 24);
    for (int i = threadIdx.x; i < ntiles; i += TOPK_THREADS) list[i] = i | all;
    if (threadIdx.x == 0) P.list_len[b * P.cache.num_kv_heads + h] = ntiles;
}

// Shared selection: head 0's score row := the max over the group's G heads
// (in place; the scores are this call's).
template <int G>
__device__ void group_max_scores(const SparseParams& P, int b, int h, int nblk) {
    float* sc0 = P.scores + ((size_t)b * P.nq + (size_t)h * G) * P.max_nblk;
    for (int j = threadIdx.x; j < nblk; j += TOPK_THREADS) {
        float m = __ldcg(sc0 + j);
#pragma unroll
        for (int g = 1; g < G; g++) {
            const float v = __ldcg(P.scores + ((size_t)b * P.nq + (size_t)h * G + g) * P.max_nblk + j);
            m = v > m ? v : m;
        }
        sc0[j] = m;
    }
    __syncthreads();
}

// Top-k of score row g of (b, h): the k = min(topk, nblk) highest, equal
// scores going to the lower block.  Kept blocks OR `bits` into their masks and
// are written in ascending order to sel rows `sel_rows` (a group's rows for a
// shared selection).  Radix select of the k-th largest order-preserving key,
// 8 bits a pass from the top, stopping early once every key of the chosen
// bucket is kept; then keys above the threshold are kept, plus the first kk
// (by block index) equal to it.
template <int G>
__device__ void topk_row_global(const SparseParams& P, int b, int h, int g, int nblk,
                                uint32_t* masks, uint32_t bits, int sel_rows, SelectSmem& S) {
    const int tid = threadIdx.x;
    const float* sc = P.scores + ((size_t)b * P.nq + (size_t)h * G + g) * P.max_nblk;
    int32_t* sel = P.sel_blocks ? P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + g) * P.topk
                                : nullptr;
    const int k = min(P.topk, nblk);
    uint32_t thr = 0, tmask = 0xFFFFFFFFu;
    int kk = 0;
    if (k == nblk) {
        kk = nblk;  // keep everything (every key >= 0 = thr under an empty mask)
        tmask = 0u;
    } else {
        uint32_t prefix = 0, pmask = 0;
        int rem = k;
        for (int pass = 0; pass < 4; pass++) {
            const int shift = 24 - 8 * pass;
            S.hist[tid] = 0;
            __syncthreads();
            for (int j = tid; j < nblk; j += TOPK_THREADS) {
                const uint32_t u = order_key(__ldcg(sc + j));
                if ((u & pmask) == prefix) atomicAdd(&S.hist[(u >> shift) & 255], 1);
            }
            __syncthreads();
            // inclusive count from digit 255 downwards: thread t holds digit 255 - t
            const int cnt = S.hist[255 - tid];
            int tot;
            const int excl = block_excl_scan(cnt, S.scan_tmp, tot);
            if (excl < rem && excl + cnt >= rem) {
                S.prefix = prefix | ((uint32_t)(255 - tid) << shift);
                S.kk = rem - excl;
                S.cnt = cnt;
            }
            __syncthreads();
            prefix = S.prefix;
            rem = S.kk;
            pmask |= 0xFFu << shift;
            const bool all_kept = S.cnt == rem;
            __syncthreads();
            if (all_kept) break;
        }
        thr = prefix;
        tmask = pmask;
        kk = rem;
    }
    // mark: top bits > thr, or == thr among the first kk such keys by index
    int ties_before = 0, kept_before = 0;
    for (int base = 0; base < nblk; base += TOPK_THREADS) {
        const int j = base + tid;
        const bool in = j < nblk;
        const uint32_t u = in ? (order_key(__ldcg(sc + j)) & tmask) : 0u;
        const bool gt = in && u > thr;
        const bool eq = in && !gt && u == thr;
        int tie_tot;
        const int tie_rank = block_excl_scan(eq ? 1 : 0, S.scan_tmp, tie_tot) + ties_before;
        const bool keep = gt || (eq && tie_rank < kk);
        int keep_tot;
        const int pos = block_excl_scan(keep ? 1 : 0, S.scan_tmp, keep_tot) + kept_before;
        if (keep) {
            atomicOr(masks + j, bits);
            if (sel)
                for (int r = 0; r < sel_rows; r++) sel[(size_t)r * P.topk + pos] = j;
        }
        ties_before += tie_tot;
        kept_before += keep_tot;
    }
    __syncthreads();
}

// Union over the G heads of (b, h): the ascending tile list with per-entry
// head masks (entry = tile | mask << 24).
template <int G>
__device__ void build_union_global(const SparseParams& P, int b, int h, int n, int nblk,
                                   const uint32_t* masks, SelectSmem& S) {
    const int nkv = P.cache.num_kv_heads;
    const int ntiles = (n + TILE - 1) / TILE;
    const int m = P.block / TILE;  // tiles per block
    int32_t* list = P.tile_list + (size_t)(b * nkv + h) * P.list_cap;
    int written = 0;
    for (int base = 0; base < nblk; base += TOPK_THREADS) {
        const int j = base + threadIdx.x;
        const uint32_t mk = (j < nblk) ? __ldcg(masks + j) : 0u;
        const int cnt = mk ? min(m, ntiles - j * m) : 0;
        int tot;
        const int pos = block_excl_scan(cnt, S.scan_tmp, tot) + written;
        for (int s = 0; s < cnt; s++) list[pos + s] = (j * m + s) | (int32_t)(mk << 24);
        written += tot;
    }
    if (threadIdx.x == 0) P.list_len[b * nkv + h] = written;
}

// The same selection with each thread holding TOPK_KPT consecutive block
// scores in registers (rows of up to TOPK_THREADS * TOPK_KPT blocks): one read
// of the row, histogram updates aggregated per warp (one shared atomic per
// distinct digit), and the tie ranks and output positions from one block scan
// each -- thread t's blocks are t*KPT .. t*KPT+KPT-1, so a scan over threads of
// per-thread counts orders them by block index.
constexpr int TOPK_KPT = 8;

template <int G>
__device__ void topk_row(const SparseParams& P, int b, int h, int g, int nblk, uint32_t* masks,
                         uint32_t bits, int sel_rows, SelectSmem& S) {
    if (nblk > TOPK_THREADS * TOPK_KPT) {
        topk_row_global<G>(P, b, h, g, nblk, masks, bits, sel_rows, S);
        return;
    }
    const int tid = threadIdx.x, lane = tid & 31;
    const float* sc = P.scores + ((size_t)b * P.nq + (size_t)h * G + g) * P.max_nblk;
    int32_t* sel = P.sel_blocks ? P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + g) * P.topk
                                : nullptr;
    const int k = min(P.topk, nblk);
    const int j0 = tid * TOPK_KPT;
    // keys of real blocks are >= 1 (order_key(-inf) = 0x007FFFFF): 0 marks "no block"
    uint32_t key[TOPK_KPT];
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) key[i] = (j0 + i < nblk) ? order_key(__ldcg(sc + j0 + i)) : 0u;
    uint32_t thr = 0, tmask = 0;  // k == nblk: every block is kept
    int kk = nblk;
    if (k < nblk) {
        uint32_t prefix = 0, pmask = 0;
        int rem = k;
        for (int pass = 0; pass < 4; pass++) {
            const int shift = 24 - 8 * pass;
            S.hist[tid] = 0;
            __syncthreads();
#pragma unroll
            for (int i = 0; i < TOPK_KPT; i++) {
                const bool in = key[i] != 0u && (key[i] & pmask) == prefix;
                const uint32_t dig = (key[i] >> shift) & 255u;
                const uint32_t peers = __match_any_sync(0xffffffffu, in ? dig : 0x100u);
                if (in && (int)(__ffs(peers) - 1) == lane) atomicAdd(&S.hist[dig], __popc(peers));
            }
            __syncthreads();
            // inclusive count from digit 255 downwards: thread t holds digit 255 - t
            const int cnt = S.hist[255 - tid];
            int tot;
            const int excl = block_excl_scan(cnt, S.scan_tmp, tot);
            if (excl < rem && excl + cnt >= rem) {
                S.prefix = prefix | ((uint32_t)(255 - tid) << shift);
                S.kk = rem - excl;
                S.cnt = cnt;
            }
            __syncthreads();
            prefix = S.prefix;
            rem = S.kk;
            pmask |= 0xFFu << shift;
            const bool all_kept = S.cnt == rem;
            __syncthreads();
            if (all_kept) break;
        }
        thr = prefix;
        tmask = pmask;
        kk = rem;
    }
    // keep: top bits above thr, or equal to it among the first kk such blocks
    uint32_t gt = 0, eq = 0;
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) {
        const uint32_t u = key[i] & tmask;
        const bool valid = key[i] != 0u;
        gt |= (uint32_t)(valid && u > thr) << i;
        eq |= (uint32_t)(valid && u == thr && !(u > thr)) << i;
    }
    int tie_tot;
    int rank = block_excl_scan(__popc(eq), S.scan_tmp, tie_tot);
    uint32_t keep = gt;
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++)
        if ((eq >> i) & 1u) keep |= (uint32_t)(rank++ < kk) << i;
    int keep_tot;
    int pos = block_excl_scan(__popc(keep), S.scan_tmp, keep_tot);
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) {
        if (!((keep >> i) & 1u)) continue;
        atomicOr(masks + j0 + i, bits);
        if (sel)
            for (int r = 0; r < sel_rows; r++) sel[(size_t)r * P.topk + pos] = j0 + i;
        pos++;
    }
    __syncthreads();
}

// Union tile list from the masks, TOPK_KPT consecutive blocks per thread.
template <int G>
__device__ void build_union(const SparseParams& P, int b, int h, int n, int nblk,
                            const uint32_t* masks, SelectSmem& S) {
    if (nblk > TOPK_THREADS * TOPK_KPT) {
        build_union_global<G>(P, b, h, n, nblk, masks, S);
        return;
    }
    const int nkv = P.cache.num_kv_heads;
    const int ntiles = (n + TILE - 1) / TILE;
    const int m = P.block / TILE;  // tiles per block
    int32_t* list = P.tile_list + (size_t)(b * nkv + h) * P.list_cap;
    const int j0 = threadIdx.x * TOPK_KPT;
    uint32_t mk[TOPK_KPT];
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) {
        mk[i] = (j0 + i < nblk) ? __ldcg(masks + j0 + i) : 0u;
        cnt += mk[i] ? min(m, ntiles - (j0 + i) * m) : 0;
    }
    int tot;
    int pos = block_excl_scan(cnt, S.scan_tmp, tot);
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) {
        if (!mk[i]) continue;
        const int j = j0 + i, c = min(m, ntiles - j * m);
        for (int s2 = 0; s2 < c; s2++) list[pos + s2] = (j * m + s2) | (int32_t)(mk[i] << 24);
        pos += c;
    }
    if (threadIdx.x == 0) P.list_len[b * nkv + h] = tot;
}

// Every head of (b, h), or the group's one shared selection, then the union.
// Not inlined: its registers stay out of the probe loop's allocation.
template <int G>
__device__ __noinline__ void select_all(const SparseParams& P, int b, int h, int n, SelectSmem& S) {
    const int nblk = (n + P.block - 1) / P.block;
    uint32_t* masks = P.masks + (size_t)(b * P.cache.num_kv_heads + h) * P.max_nblk;
    clear_selection<G>(P, b, h, 0, G);
    __syncthreads();
    if (P.shared_sel) {
        group_max_scores<G>(P, b, h, nblk);
        topk_row<G>(P, b, h, 0, nblk, masks, (1u << G) - 1u, G, S);
    } else {
        for (int g = 0; g < G; g++) topk_row<G>(P, b, h, g, nblk, masks, 1u << g, 1, S);
    }
    build_union<G>(P, b, h, n, nblk, masks, S);
}

// ---------------------------------------------------------------------------
// Probe: grid (ceil(max_nblk / probe_bpc), nkv, B), 8 warps.  The CTA's page
// ids are read once into shared memory (no K load waits on a page-table load).
// The CTA's blocks form groups of 4; warp w owns groups w, w + 8, ... and walks
// units = (pass of 8 probe rows, group), loading the next unit before computing
// the current one so that loads stay in flight.  Lane (block gb = lane / 8 of
// the group, probe row pr = lane % 8 of the pass) loads its whole K row (the
// four 32-byte blocks of a row sit 1 KB apart in the sub-tile), forms the
// exact score in its own registers in the method's order, and the 8 lanes of a
// block take the maximum with three shuffles; block maxima collect in shared
// memory across passes.  With tickets (P.tickets), the last probe CTA of a
// (sequence, KV head) to finish runs the selection and builds the union tile
// list (select_all) in the same launch; CTA 0 of a gated sequence writes its
// full list.
// ---------------------------------------------------------------------------
constexpr int PROBE_WARPS = 8;
static_assert(PROBE_WARPS * 32 == TOPK_THREADS, "the probe CTA runs the selection");
// Blocks per CTA: long-lived CTAs (8 units of 4 blocks per warp at block 32)
// so that the prologue (page ids, Q quantisation, a CTA barrier) and the
// epilogue weigh little against the streaming.
constexpr int PROBE_MAX_BPC = 256;
constexpr int PROBE_MAX_PAGES = 512;   // page ids a CTA stages

struct ProbeRow {
    uint4 k[2 * NB];  // the row's 128 int8 codes, block by block
    float kst;        // its stored K maximum
    bool valid;
};

template <int G>
__global__ void __launch_bounds__(PROBE_WARPS * 32, 2) kq8_probe_kernel(const SparseParams P) {
    __shared__ __align__(16) int8_t qi[G][HD];
    __shared__ float qsc[G][NB];
    __shared__ int32_t pages[PROBE_MAX_PAGES];
    __shared__ float best[PROBE_MAX_BPC][G];
    __shared__ SelectSmem sel_smem;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    // the attention kernel after this one may become resident as soon as every
    // probe CTA has started; it waits for this grid's completion before it
    // reads the tile lists
    griddep_launch_dependents();
    int n = sparse_seq_len(P, b);
    if (n < 0 || n <= 2 * P.block) {  // gate: the exact path needs no probe
        if (P.tickets && blockIdx.x == 0) {
            if (n < 0 && threadIdx.x == 0 && h == 0 && P.status)
                atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
            n = max(n, 0);
            clear_selection<G>(P, b, h, 0, G);
            gated_list<G>(P, b, h, n);
        }
        return;
    }
    const int nblk = (n + P.block - 1) / P.block;
    const int j0 = blockIdx.x * P.probe_bpc;
    if (j0 >= nblk) return;
    const int j1 = min(j0 + P.probe_bpc, nblk);
    const int pg0 = (j0 * P.block) / kv_bs;
    const int pg1 = (min(j1 * P.block, n) - 1) / kv_bs;

    const size_t pt_row = (size_t)(P.row_seq ? P.row_seq[b] : b) * P.max_pages;
    for (int i = threadIdx.x; i <= pg1 - pg0; i += PROBE_WARPS * 32) {
        const int32_t pg = P.page_table[pt_row + pg0 + i];
        const bool ok = pg >= 0 && pg < P.cache.num_pages;
        if (!ok && P.status) atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
        pages[i] = ok ? pg : -1;
    }
    for (int i = threadIdx.x; i < (j1 - j0) * G; i += PROBE_WARPS * 32)
        best[i / G][i % G] = -INFINITY;
    // the top-k kernel ORs its heads' choices into these blocks' masks (a
    // probe-only call passes none)
    if (P.masks)
        for (int i = threadIdx.x; i < j1 - j0; i += PROBE_WARPS * 32)
            P.masks[(size_t)(b * nkv + h) * P.max_nblk + j0 + i] = 0u;
    for (int g = warp; g < G; g += PROBE_WARPS) {
        const float4 x =
            reinterpret_cast<const float4*>(P.q + ((size_t)b * P.nq + (size_t)h * G + g) * HD)[lane];
        float qs;
        const uint32_t codes = quantize_q_lane(x, qs);
        reinterpret_cast<uint32_t*>(qi[g])[lane] = codes;
        if ((lane & 7) == 0) qsc[g][lane >> 3] = qs;
    }
    __syncthreads();

    const int gb = lane >> 3, pr = lane & 7;
    const int stride = P.block / P.probe;
    float qs[G][NB];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int bb = 0; bb < NB; bb++) qs[g][bb] = qsc[g][bb];
    const float scale = P.scale;

    // this warp's units: (pass, group of 4 blocks)
    const int ngroups_cta = (j1 - j0 + 3) / 4;
    const int my_groups =
        (ngroups_cta > warp) ? (ngroups_cta - warp + PROBE_WARPS - 1) / PROBE_WARPS : 0;
    const int npass = (P.probe + 7) / 8;
    const int nunits = my_groups * npass;
    auto block_of = [&](int k) { return j0 + 4 * (warp + PROBE_WARPS * (k % my_groups)) + gb; };
    auto load = [&](ProbeRow& R, int k) {
        const int jj = block_of(k), p = (k / my_groups) * 8 + pr;
        const int t = jj * P.block + p * stride;
        R.valid = (jj < j1) && (p < P.probe) && (t < n);
#pragma unroll
        for (int i = 0; i < 2 * NB; i++) R.k[i] = make_uint4(0, 0, 0, 0);
        R.kst = 0.0f;
        if (R.valid) {
            const int32_t pg = pages[t / kv_bs - pg0];
            if (pg >= 0) {
                const int r = t % kv_bs;
                const int8_t* src =
                    P.cache.k + kv_sub_off(pg, h, nkv, kv_bs, r / TILE) + kpos(r % TILE) * 32;
#pragma unroll
                for (int bb = 0; bb < NB; bb++) {
                    R.k[2 * bb] = __ldg(reinterpret_cast<const uint4*>(src + bb * 1024));
                    R.k[2 * bb + 1] = __ldg(reinterpret_cast<const uint4*>(src + bb * 1024 + 16));
                }
                R.kst = __ldg(P.cache.kscale + scale_sub_off(pg, h, nkv, kv_bs, r / TILE) +
                              r % TILE);
            } else {
                R.valid = false;
            }
        }
    };
    auto compute = [&](const ProbeRow& R, int k) {
        const int jj = block_of(k);
#pragma unroll
        for (int g = 0; g < G; g++) {
            int d[NB];
#pragma unroll
            for (int bb = 0; bb < NB; bb++) {
                const uint4 qa = *reinterpret_cast<const uint4*>(qi[g] + bb * 32);
                const uint4 qb = *reinterpret_cast<const uint4*>(qi[g] + bb * 32 + 16);
                const uint4 ka = R.k[2 * bb], kb = R.k[2 * bb + 1];
                int x = __dp4a((int)ka.x, (int)qa.x, 0);
                x = __dp4a((int)ka.y, (int)qa.y, x);
                x = __dp4a((int)ka.z, (int)qa.z, x);
                x = __dp4a((int)ka.w, (int)qa.w, x);
                x = __dp4a((int)kb.x, (int)qb.x, x);
                x = __dp4a((int)kb.y, (int)qb.y, x);
                x = __dp4a((int)kb.z, (int)qb.z, x);
                d[bb] = __dp4a((int)kb.w, (int)qb.w, x);
            }
            float s = R.valid ? score_exact(d, qs[g], R.kst, scale) : -INFINITY;
            // max over the 8 probe rows of the block (lanes 8gb .. 8gb+7)
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 1));
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 2));
            s = fmaxf(s, __shfl_xor_sync(0xffffffffu, s, 4));
            if (pr == 0 && jj < j1) best[jj - j0][g] = fmaxf(best[jj - j0][g], s);
        }
    };
    ProbeRow A, Bu;
    if (nunits > 0) load(A, 0);
    for (int k = 0; k < nunits; k += 2) {
        if (k + 1 < nunits) load(Bu, k + 1);
        compute(A, k);
        if (k + 1 >= nunits) break;
        if (k + 2 < nunits) load(A, k + 2);
        compute(Bu, k + 1);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < (j1 - j0) * G; i += PROBE_WARPS * 32) {
        const int jj = j0 + i / G, g = i % G;
        P.scores[((size_t)b * P.nq + (size_t)h * G + g) * P.max_nblk + jj] = best[i / G][g];
    }
    if (!P.tickets) return;
    // the last of this (sequence, KV head)'s probe CTAs selects its blocks
    const unsigned nctas = (unsigned)((nblk + P.probe_bpc - 1) / P.probe_bpc);
    __syncthreads();  // this CTA's scores and cleared masks are written
    if (threadIdx.x == 0) {
        __threadfence();  // cumulative: orders them all before the ticket
        sel_smem.last = atomicAdd(P.tickets + b * nkv + h, 1u) == nctas - 1;
    }
    __syncthreads();
    if (!sel_smem.last) return;
    __threadfence();
    select_all<G>(P, b, h, n, sel_smem);
    if (threadIdx.x == 0) P.tickets[b * nkv + h] = 0u;  // ready for the next call
}

// ---------------------------------------------------------------------------
// Top-k + union as a kernel of its own, for batches with more (sequence, KV
// head) pairs than ticket counters: grid (KV head, sequence), one CTA of 256
// threads per KV head selecting its G heads in turn.
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(TOPK_THREADS) kq8_topk_kernel(const SparseParams P) {
    __shared__ SelectSmem S;
    const int h = blockIdx.x, b = blockIdx.y;
    griddep_launch_dependents();
    int n = sparse_seq_len(P, b);
    if (n < 0) {
        if (threadIdx.x == 0 && h == 0 && P.status) atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
        n = 0;
    }
    if (n <= 2 * P.block) {
        clear_selection<G>(P, b, h, 0, G);
        gated_list<G>(P, b, h, n);
        return;
    }
    select_all<G>(P, b, h, n, S);
}

}  // namespace kq8
