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
// Probe: grid (ceil(max_nblk / probe_bpc), nkv, B), 8 warps.  The CTA's page
// ids are read once into shared memory (no K load waits on a page-table load).
// The CTA's blocks form groups of 4; warp w owns groups w, w + 8, ... and walks
// units = (pass of 8 probe rows, group), loading the next unit before computing
// the current one so that loads stay in flight.  Lane (block gb = lane / 8 of
// the group, probe row pr = lane % 8 of the pass) loads its whole K row (the
// four 32-byte blocks of a row sit 1 KB apart in the sub-tile), forms the
// exact score in its own registers in the method's order, and the 8 lanes of a
// block take the maximum with three shuffles; block maxima collect in shared
// memory across passes.
// ---------------------------------------------------------------------------
constexpr int PROBE_WARPS = 8;
constexpr int PROBE_MAX_BPC = 128;     // blocks per CTA
constexpr int PROBE_MAX_PAGES = 256;   // page ids a CTA stages

struct ProbeRow {
    uint4 k[2 * NB];  // the row's 128 int8 codes, block by block
    float kst;        // its stored K maximum
    bool valid;
};

template <int G>
__global__ void __launch_bounds__(PROBE_WARPS * 32) kq8_probe_kernel(const SparseParams P) {
    __shared__ __align__(16) int8_t qi[G][HD];
    __shared__ float qsc[G][NB];
    __shared__ int32_t pages[PROBE_MAX_PAGES];
    __shared__ float best[PROBE_MAX_BPC][G];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    const int n = sparse_seq_len(P, b);
    if (n < 0 || n <= 2 * P.block) return;  // gate: the exact path needs no probe
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
}

// ---------------------------------------------------------------------------
// Top-k + union: grid (KV head, sequence, head g) with one CTA of 256
// threads per query head when tickets are available (a CTA selects head g's
// blocks and ORs bit g into the block masks, which the probe kernel cleared;
// the last of the G CTAs to finish builds the union), else one CTA per KV
// head that selects its G heads in turn.
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

template <int G>
__global__ void __launch_bounds__(TOPK_THREADS) kq8_topk_kernel(const SparseParams P) {
    __shared__ int hist[256];
    __shared__ int scan_tmp[TOPK_THREADS / 32];
    __shared__ uint32_t s_prefix;
    __shared__ int s_kk, s_cnt;
    __shared__ int s_last;
    const int h = blockIdx.x, b = blockIdx.y;
    const int nkv = P.cache.num_kv_heads;
    const int tid = threadIdx.x;
    int n = sparse_seq_len(P, b);
    if (n < 0) {
        if (tid == 0 && h == 0) atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
        n = 0;
    }
    const int ntiles = (n + TILE - 1) / TILE;
    const int m = P.block / TILE;  // tiles per block
    int32_t* list = P.tile_list + (size_t)(b * nkv + h) * P.list_cap;
    const bool gated = n <= 2 * P.block;

    const bool per_head = gridDim.z > 1;
    const int g_first = per_head ? (int)blockIdx.z : 0;
    const int g_end = per_head ? g_first + 1 : G;
    if (P.sel_blocks) {
        for (int g = g_first; g < g_end; g++) {
            int32_t* sel = P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + g) * P.topk;
            for (int i = tid; i < P.topk; i += TOPK_THREADS) sel[i] = -1;
        }
    }
    if (gated) {  // exact path: every tile, every head
        if (g_first != 0) return;
        const int32_t all = (int32_t)(((1u << G) - 1u) << 24);
        for (int i = tid; i < ntiles; i += TOPK_THREADS) list[i] = i | all;
        if (tid == 0) P.list_len[b * nkv + h] = ntiles;
        return;
    }
    const int nblk = (n + P.block - 1) / P.block;
    uint32_t* masks = P.masks + (size_t)(b * nkv + h) * P.max_nblk;
    if (P.shared_sel) {
        // one selection for the group: head 0's row becomes the max over the G
        // heads of their block scores (in place; the scores are this call's)
        float* sc0 = P.scores + ((size_t)b * P.nq + (size_t)h * G) * P.max_nblk;
        for (int j = tid; j < nblk; j += TOPK_THREADS) {
            float m = sc0[j];
#pragma unroll
            for (int g = 1; g < G; g++) {
                const float v = P.scores[((size_t)b * P.nq + (size_t)h * G + g) * P.max_nblk + j];
                m = v > m ? v : m;
            }
            sc0[j] = m;
        }
    }
    __syncthreads();

    const int nsel = P.shared_sel ? 1 : g_end;
    const uint32_t group_mask = (1u << G) - 1u;
    for (int g = g_first; g < nsel; g++) {
        const float* sc = P.scores + ((size_t)b * P.nq + (size_t)h * G + g) * P.max_nblk;
        int32_t* sel = P.sel_blocks ? P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + g) * P.topk
                                    : nullptr;
        const int k = min(P.topk, nblk);
        // keys whose top bits (tmask) exceed thr are kept, plus the first kk
        // whose top bits equal thr
        uint32_t thr = 0, tmask = 0xFFFFFFFFu;
        int kk = 0;
        if (k == nblk) {
            thr = 0;
            kk = nblk;  // every key >= 0: take all ties at key 0 too
        } else {
            // radix select of the k-th largest key, 8 bits at a time from the top;
            // it stops early once every key of the chosen bucket is kept (the
            // lower bits can then change nothing)
            uint32_t prefix = 0, pmask = 0;
            int rem = k;
            for (int pass = 0; pass < 4; pass++) {
                const int shift = 24 - 8 * pass;
                hist[tid] = 0;
                __syncthreads();
                for (int j = tid; j < nblk; j += TOPK_THREADS) {
                    const uint32_t u = order_key(sc[j]);
                    if ((u & pmask) == prefix) atomicAdd(&hist[(u >> shift) & 255], 1);
                }
                __syncthreads();
                // inclusive count from digit 255 downwards: thread t holds digit 255 - t
                const int cnt = hist[255 - tid];
                int tot;
                const int excl = block_excl_scan(cnt, scan_tmp, tot);
                if (excl < rem && excl + cnt >= rem) {
                    s_prefix = prefix | ((uint32_t)(255 - tid) << shift);
                    s_kk = rem - excl;
                    s_cnt = cnt;
                }
                __syncthreads();
                prefix = s_prefix;
                rem = s_kk;
                pmask |= 0xFFu << shift;
                const bool all_kept = s_cnt == rem;
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
            const uint32_t u = (j < nblk) ? (order_key(sc[j]) & tmask) : 0u;
            const bool in = j < nblk;
            const bool gt = in && (k == nblk || u > thr);
            const bool eq = in && !gt && u == thr;
            int tie_tot;
            const int tie_rank = block_excl_scan(eq ? 1 : 0, scan_tmp, tie_tot) + ties_before;
            const bool keep = gt || (eq && tie_rank < kk);
            int keep_tot;
            const int pos = block_excl_scan(keep ? 1 : 0, scan_tmp, keep_tot) + kept_before;
            if (keep) {
                atomicOr(masks + j, P.shared_sel ? group_mask : (1u << g));
                if (sel) {
                    if (P.shared_sel) {
                        for (int gg = 0; gg < G; gg++) sel[(size_t)gg * P.topk + pos] = j;
                    } else {
                        sel[pos] = j;
                    }
                }
            }
            ties_before += tie_tot;
            kept_before += keep_tot;
        }
        __syncthreads();
    }

    if (per_head) {
        // the last of the G CTAs of this (sequence, KV head) builds the union
        __threadfence();
        __syncthreads();
        if (tid == 0) s_last = atomicAdd(P.tickets + b * nkv + h, 1u) == (uint32_t)(G - 1);
        __syncthreads();
        if (!s_last) return;
        __threadfence();
    }
    // union over the G heads -> ascending tile list with per-entry head masks
    int written = 0;
    for (int base = 0; base < nblk; base += TOPK_THREADS) {
        const int j = base + tid;
        const uint32_t mk = (j < nblk) ? __ldcg(masks + j) : 0u;
        const int cnt = mk ? min(m, ntiles - j * m) : 0;
        int tot;
        const int pos = block_excl_scan(cnt, scan_tmp, tot) + written;
        for (int s = 0; s < cnt; s++) list[pos + s] = (j * m + s) | (int32_t)(mk << 24);
        written += tot;
    }
    if (tid == 0) {
        P.list_len[b * nkv + h] = written;
        if (per_head) P.tickets[b * nkv + h] = 0u;  // ready for the next call
    }
}

}  // namespace kq8
