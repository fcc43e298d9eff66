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
    // K sub-tiles as the 3-D tensor {1024 B (32 positions x 32 B), 4 element
    // blocks, num_pages * nkv * kv_bs / 32 sub-tiles}: the probe's tensor copies
    // of the first 8 positions of the 4 blocks (set when block = 4 * probe)
    CUtensorMap kmap;
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
    int32_t probe_tma;       // 1: kmap is set, the probe takes the tensor-copy form
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

// Rows (query heads) selected together by the in-register selection: they
// share every CTA barrier and scan.
constexpr int SEL_HG = 2;
constexpr int TOPK_KPT = 8;  // consecutive block scores per thread (in-register form)

constexpr int SEL_SMALL = 256;  // rows of up to this many blocks: one warp per head

struct SelectSmem {
    uint32_t keptw[8][SEL_SMALL / 32];  // short rows: bit l of word [r][i] = row r keeps block 32 i + l
    int hist[2][SEL_HG][256];  // double-buffered: a pass clears the next one's
    int scan_tmp[SEL_HG + 1][TOPK_THREADS / 32];
    uint32_t prefix[SEL_HG];
    int kk[SEL_HG], cnt[SEL_HG];
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
            S.hist[0][0][tid] = 0;
            __syncthreads();
            for (int j = tid; j < nblk; j += TOPK_THREADS) {
                const uint32_t u = order_key(__ldcg(sc + j));
                if ((u & pmask) == prefix) atomicAdd(&S.hist[0][0][(u >> shift) & 255], 1);
            }
            __syncthreads();
            // inclusive count from digit 255 downwards: thread t holds digit 255 - t
            const int cnt = S.hist[0][0][255 - tid];
            int tot;
            const int excl = block_excl_scan(cnt, S.scan_tmp[0], tot);
            if (excl < rem && excl + cnt >= rem) {
                S.prefix[0] = prefix | ((uint32_t)(255 - tid) << shift);
                S.kk[0] = rem - excl;
                S.cnt[0] = cnt;
            }
            __syncthreads();
            prefix = S.prefix[0];
            rem = S.kk[0];
            pmask |= 0xFFu << shift;
            const bool all_kept = S.cnt[0] == rem;
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
        const int tie_rank = block_excl_scan(eq ? 1 : 0, S.scan_tmp[0], tie_tot) + ties_before;
        const bool keep = gt || (eq && tie_rank < kk);
        int keep_tot;
        const int pos = block_excl_scan(keep ? 1 : 0, S.scan_tmp[0], keep_tot) + kept_before;
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
        const int pos = block_excl_scan(cnt, S.scan_tmp[0], tot) + written;
        for (int s = 0; s < cnt; s++) list[pos + s] = (j * m + s) | (int32_t)(mk << 24);
        written += tot;
    }
    if (threadIdx.x == 0) P.list_len[b * nkv + h] = written;
}

// Exclusive block-wide prefix sums of NV values at once (one set of barriers).
template <int NV>
__device__ __forceinline__ void block_excl_scan_v(const int (&v)[NV], int (&excl)[NV],
                                                  int (&total)[NV],
                                                  int (*tmp)[TOPK_THREADS / 32]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) x[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int y = __shfl_up_sync(0xffffffffu, x[i], o);
            if (lane >= o) x[i] += y;
        }
    if (lane == 31)
#pragma unroll
        for (int i = 0; i < NV; i++) tmp[i][warp] = x[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NV; i++) {
        int base = 0, tot = 0;
#pragma unroll
        for (int w = 0; w < TOPK_THREADS / 32; w++) {
            const int t = tmp[i][w];
            if (w < warp) base += t;
            tot += t;
        }
        excl[i] = base + x[i] - v[i];
        total[i] = tot;
    }
    __syncthreads();
}

// The selection and the union list for rows of up to TOPK_THREADS * TOPK_KPT
// blocks, in registers: thread t holds the order-preserving keys of blocks
// t*KPT .. t*KPT+KPT-1 of SEL_HG rows at a time (the G heads' rows, or one row
// of the heads' maxima for a shared selection).  Per row a radix select finds
// the k-th largest key 8 bits a pass from the top: every thread adds its keys
// to the row's digit histogram with shared atomics, then warp r alone scans
// row r's 256 counts and picks the digit -- two CTA barriers a pass; it
// stops once every key of the chosen bucket is kept.  Keys above the
// threshold are kept, plus the first kk equal to it by block index (a scan
// ranks the ties, only when some are left out); one scan over per-thread
// counts places the kept ids in ascending order (a thread's blocks are
// consecutive) and, with the kept head bits held by their threads, the
// entries of the union tile list.
template <int G, bool SHARED>
__device__ __forceinline__ void select_rows_smem(const SparseParams& P, int b, int h, int n,
                                                 int nblk, SelectSmem& S) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nkv = P.cache.num_kv_heads;
    const int j0 = tid * TOPK_KPT;
    constexpr int rows = SHARED ? 1 : G;
    const int k = min(P.topk, nblk);
    const int ntiles = (n + TILE - 1) / TILE;
    const int m = P.block / TILE;  // tiles per block
    const float* sc0 = P.scores + ((size_t)b * P.nq + (size_t)h * G) * P.max_nblk;
    uint8_t kept[TOPK_KPT];  // head bits of this thread's blocks
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) kept[i] = 0;
    // entries of the union list this thread writes (blocks are m tiles, the last one shorter)
    auto list_count = [&]() {
        int c = 0;
#pragma unroll
        for (int i = 0; i < TOPK_KPT; i++) c += kept[i] ? min(m, ntiles - (j0 + i) * m) : 0;
        return c;
    };
    int list_pos = -1, list_tot = 0;
#pragma unroll 1
    for (int r0 = 0; r0 < rows; r0 += SEL_HG) {
        const bool last_group = r0 + SEL_HG >= rows;
        // keys of real blocks are >= 1 (order_key(-inf) = 0x007FFFFF): 0 marks "no block"
        uint32_t key[SEL_HG][TOPK_KPT];
#pragma unroll
        for (int hh = 0; hh < SEL_HG; hh++)
#pragma unroll
            for (int i = 0; i < TOPK_KPT; i++) {
                const int j = j0 + i;
                const bool in = j < nblk && r0 + hh < rows;
                float v = -INFINITY;
                if (in) {
                    if (SHARED) {
                        v = __ldcg(sc0 + j);
#pragma unroll
                        for (int g = 1; g < G; g++) {
                            const float x = __ldcg(sc0 + (size_t)g * P.max_nblk + j);
                            v = x > v ? x : v;
                        }
                    } else {
                        v = __ldcg(sc0 + (size_t)(r0 + hh) * P.max_nblk + j);
                    }
                }
                key[hh][i] = in ? order_key(v) : 0u;
            }
        uint32_t prefix[SEL_HG], pmask[SEL_HG];
        int rem[SEL_HG];
        bool done[SEL_HG], exact[SEL_HG];  // exact: every key equal to the threshold is kept
#pragma unroll
        for (int hh = 0; hh < SEL_HG; hh++) {
            prefix[hh] = 0u;
            pmask[hh] = 0u;  // k == nblk: every block is kept (empty mask, threshold 0)
            rem[hh] = k;
            done[hh] = (k >= nblk) || (r0 + hh >= rows);
            exact[hh] = true;
            S.hist[0][hh][tid] = 0;
        }
        __syncthreads();
#pragma unroll 1
        for (int pass = 0; pass < 4; pass++) {
            bool all = true;
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) all = all && done[hh];
            if (all) break;  // uniform: every thread holds the same flags
            const int cur = pass & 1, shift = 24 - 8 * pass;
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) {
                S.hist[cur ^ 1][hh][tid] = 0;  // the next pass's buffer (read two barriers ago)
                if (done[hh]) continue;
#pragma unroll
                for (int i = 0; i < TOPK_KPT; i++) {
                    const bool in = key[hh][i] != 0u && (key[hh][i] & pmask[hh]) == prefix[hh];
                    if (in) atomicAdd(&S.hist[cur][hh][(key[hh][i] >> shift) & 255u], 1);
                }
            }
            __syncthreads();
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) {
                if (warp != hh || done[hh]) continue;
                // lane l: digits 255 - 8l .. 248 - 8l, counted from the top
                int c[8], sum = 0;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    c[i] = S.hist[cur][hh][255 - 8 * lane - i];
                    sum += c[i];
                }
                int incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                int excl = incl - sum;
                const int r = rem[hh];
                if (excl < r && incl >= r) {
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        if (excl + c[i] >= r) {
                            S.prefix[hh] = prefix[hh] | ((uint32_t)(255 - 8 * lane - i) << shift);
                            S.kk[hh] = r - excl;
                            S.cnt[hh] = c[i];
                            break;
                        }
                        excl += c[i];
                    }
                }
            }
            __syncthreads();
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) {
                if (done[hh]) continue;
                prefix[hh] = S.prefix[hh];
                rem[hh] = S.kk[hh];
                pmask[hh] |= 0xFFu << shift;
                done[hh] = S.cnt[hh] == rem[hh];
                exact[hh] = done[hh];
            }
            // S.prefix / kk / cnt are next written after another barrier
        }
        // keep: top bits above the threshold, or equal to it among the first kk
        uint32_t gt[SEL_HG], eq[SEL_HG];
        bool ranks = false;
#pragma unroll
        for (int hh = 0; hh < SEL_HG; hh++) {
            gt[hh] = eq[hh] = 0u;
#pragma unroll
            for (int i = 0; i < TOPK_KPT; i++) {
                const uint32_t u = key[hh][i] & pmask[hh];
                const bool valid = key[hh][i] != 0u;
                gt[hh] |= (uint32_t)(valid && u > prefix[hh]) << i;
                eq[hh] |= (uint32_t)(valid && u == prefix[hh]) << i;
            }
            ranks = ranks || !exact[hh];
        }
        uint32_t keep[SEL_HG];
        if (ranks) {  // uniform: some row keeps only part of its threshold bucket
            int ne[SEL_HG], rank[SEL_HG], tie_tot[SEL_HG];
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) ne[hh] = __popc(eq[hh]);
            block_excl_scan_v<SEL_HG>(ne, rank, tie_tot, S.scan_tmp);
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) {
                keep[hh] = gt[hh];
#pragma unroll
                for (int i = 0; i < TOPK_KPT; i++)
                    if ((eq[hh] >> i) & 1u) keep[hh] |= (uint32_t)(rank[hh]++ < rem[hh]) << i;
            }
        } else {
#pragma unroll
            for (int hh = 0; hh < SEL_HG; hh++) keep[hh] = gt[hh] | eq[hh];
        }
#pragma unroll
        for (int hh = 0; hh < SEL_HG; hh++) {
            if (r0 + hh >= rows) continue;
            const uint32_t bits = SHARED ? ((1u << G) - 1u) : (1u << (r0 + hh));
#pragma unroll
            for (int i = 0; i < TOPK_KPT; i++)
                if ((keep[hh] >> i) & 1u) kept[i] |= (uint8_t)bits;
        }
        // positions of the kept ids (and, in the last group, of the list entries)
        int cnt[SEL_HG + 1], pos[SEL_HG + 1], tot[SEL_HG + 1];
#pragma unroll
        for (int hh = 0; hh < SEL_HG; hh++) cnt[hh] = __popc(keep[hh]);
        cnt[SEL_HG] = last_group ? list_count() : 0;
        block_excl_scan_v<SEL_HG + 1>(cnt, pos, tot, S.scan_tmp);
        if (last_group) {
            list_pos = pos[SEL_HG];
            list_tot = tot[SEL_HG];
        }
#pragma unroll
        for (int hh = 0; hh < SEL_HG; hh++) {
            if (r0 + hh >= rows || !P.sel_blocks) continue;
            constexpr int sel_rows = SHARED ? G : 1;
            int32_t* sel = P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + r0 + hh) * P.topk;
            int p = pos[hh];
            for (uint32_t kb = keep[hh]; kb != 0u; kb &= kb - 1u, p++) {
                const int j = j0 + __ffs(kb) - 1;
#pragma unroll
                for (int r = 0; r < sel_rows; r++) sel[(size_t)r * P.topk + p] = j;
            }
            // fewer blocks than topk: the rest of the row is -1
            if (tid == 0)
                for (int r = 0; r < sel_rows; r++)
                    for (int i = k; i < P.topk; i++) sel[(size_t)r * P.topk + i] = -1;
        }
    }
    // the union tile list: ascending blocks, entry = tile | head mask << 24
    int32_t* list = P.tile_list + (size_t)(b * nkv + h) * P.list_cap;
    uint32_t any = 0;
#pragma unroll
    for (int i = 0; i < TOPK_KPT; i++) any |= (uint32_t)(kept[i] != 0) << i;
    for (; any != 0u; any &= any - 1u) {
        const int i = __ffs(any) - 1;
        uint32_t bitsi = 0;
#pragma unroll
        for (int x = 0; x < TOPK_KPT; x++) bitsi = (x == i) ? kept[x] : bitsi;
        const int c = min(m, ntiles - (j0 + i) * m);
        for (int s2 = 0; s2 < c; s2++)
            list[list_pos++] = ((j0 + i) * m + s2) | (int32_t)(bitsi << 24);
    }
    if (tid == 0) P.list_len[b * nkv + h] = list_tot;
}

// Short rows (at most SEL_SMALL blocks): one warp per row, no CTA barrier until
// the union.  Lane l holds the keys of blocks l + 32 i (i < KPL), so a ballot
// over slice i lists blocks 32 i .. 32 i + 31 in order.  The k-th largest key t
// comes from a bitwise binary search (the largest t with at least k keys >= t,
// counted with ballots); keys above t are kept, and of the keys equal to t the
// first ones by block index until k are kept.  Kept ids are written in
// ascending order from prefix counts of the slices' ballots.
template <int G, bool SHARED, int KPL>
__device__ __forceinline__ void select_rows_warp(const SparseParams& P, int b, int h, int n,
                                                 int nblk, SelectSmem& S) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nkv = P.cache.num_kv_heads;
    constexpr int rows = SHARED ? 1 : G;
    const int k = min(P.topk, nblk);
    if (warp < rows) {
        const float* sc0 = P.scores + ((size_t)b * P.nq + (size_t)h * G) * P.max_nblk;
        uint32_t key[KPL];  // 0 marks "no block" (real keys are >= 1)
#pragma unroll
        for (int i = 0; i < KPL; i++) {
            const int j = lane + 32 * i;
            float v = -INFINITY;
            if (j < nblk) {
                if (SHARED) {
                    v = __ldcg(sc0 + j);
#pragma unroll
                    for (int g = 1; g < G; g++) {
                        const float x = __ldcg(sc0 + (size_t)g * P.max_nblk + j);
                        v = x > v ? x : v;
                    }
                } else {
                    v = __ldcg(sc0 + (size_t)warp * P.max_nblk + j);
                }
            }
            key[i] = j < nblk ? order_key(v) : 0u;
        }
        // the k-th largest key (k <= the number of real keys)
        uint32_t t = 0u;
        for (int bit = 31; bit >= 0; bit--) {
            const uint32_t cand = t | (1u << bit);
            int cnt = 0;
#pragma unroll
            for (int i = 0; i < KPL; i++) cnt += __popc(__ballot_sync(0xffffffffu, key[i] >= cand));
            if (cnt >= k) t = cand;
        }
        int above = 0;
#pragma unroll
        for (int i = 0; i < KPL; i++) above += __popc(__ballot_sync(0xffffffffu, key[i] > t));
        int need = k - above;  // keys equal to t still to keep, lowest blocks first
        int32_t* sel = P.sel_blocks
                           ? P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + warp) * P.topk
                           : nullptr;
        constexpr int sel_rows = SHARED ? G : 1;
        const uint32_t lt = (1u << lane) - 1u;
        int base = 0;
#pragma unroll
        for (int i = 0; i < KPL; i++) {
            uint32_t eq = __ballot_sync(0xffffffffu, key[i] == t && key[i] != 0u);
            if (need <= 0) {
                eq = 0u;
            } else if (__popc(eq) > need) {  // a tie across the k-th place: lowest blocks
                uint32_t take = 0u, e = eq;
                for (int c = 0; c < need; c++) {
                    take |= e & (0u - e);  // lowest set bit
                    e &= e - 1u;
                }
                eq = take;
            }
            need -= __popc(eq);
            const uint32_t kept = __ballot_sync(0xffffffffu, key[i] > t) | eq;
            if (sel && ((kept >> lane) & 1u)) {
                const int pos = base + __popc(kept & lt);
#pragma unroll
                for (int r = 0; r < sel_rows; r++) sel[(size_t)r * P.topk + pos] = lane + 32 * i;
            }
            base += __popc(kept);
            if (lane == 0) S.keptw[warp][i] = kept;
        }
        if (sel)  // fewer blocks than topk: the rest of the row is -1
            for (int i = k + lane; i < P.topk; i += 32)
#pragma unroll
                for (int r = 0; r < sel_rows; r++) sel[(size_t)r * P.topk + i] = -1;
    }
    __syncthreads();
    // the union tile list (warp 0): ascending blocks, entry = tile | head mask << 24
    if (warp == 0) {
        const int ntiles = (n + TILE - 1) / TILE;
        const int m = P.block / TILE;  // tiles per block
        int32_t* list = P.tile_list + (size_t)(b * nkv + h) * P.list_cap;
        int written = 0;
#pragma unroll
        for (int i = 0; i < KPL; i++) {
            const int j = lane + 32 * i;
            uint32_t mk = 0u;
#pragma unroll
            for (int r = 0; r < rows; r++) mk |= ((S.keptw[r][i] >> lane) & 1u) << r;
            if (SHARED) mk = mk ? ((1u << G) - 1u) : 0u;
            const int c = mk ? min(m, ntiles - j * m) : 0;
            int incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            int pos = written + incl - c;
            for (int s2 = 0; s2 < c; s2++) list[pos++] = (j * m + s2) | (int32_t)(mk << 24);
            written += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) P.list_len[b * nkv + h] = written;
    }
}

template <int G>
__device__ __forceinline__ void select_all(const SparseParams& P, int b, int h, int n,
                                           SelectSmem& S) {
    const int nblk = (n + P.block - 1) / P.block;
    if (nblk <= SEL_SMALL / 2) {
        if (P.shared_sel)
            select_rows_warp<G, true, SEL_SMALL / 64>(P, b, h, n, nblk, S);
        else
            select_rows_warp<G, false, SEL_SMALL / 64>(P, b, h, n, nblk, S);
        return;
    }
    if (nblk <= SEL_SMALL) {
        if (P.shared_sel)
            select_rows_warp<G, true, SEL_SMALL / 32>(P, b, h, n, nblk, S);
        else
            select_rows_warp<G, false, SEL_SMALL / 32>(P, b, h, n, nblk, S);
        return;
    }
    if (nblk <= TOPK_THREADS * TOPK_KPT) {
        if (P.shared_sel)
            select_rows_smem<G, true>(P, b, h, n, nblk, S);
        else
            select_rows_smem<G, false>(P, b, h, n, nblk, S);
        return;
    }
    uint32_t* masks = P.masks + (size_t)(b * P.cache.num_kv_heads + h) * P.max_nblk;
    clear_selection<G>(P, b, h, 0, G);
    __syncthreads();
    if (P.shared_sel) {
        group_max_scores<G>(P, b, h, nblk);
        topk_row_global<G>(P, b, h, 0, nblk, masks, (1u << G) - 1u, G, S);
    } else {
        for (int g = 0; g < G; g++) topk_row_global<G>(P, b, h, g, nblk, masks, 1u << g, 1, S);
    }
    build_union_global<G>(P, b, h, n, nblk, masks, S);
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
// Tensor-copy form (block = 4 * probe): per warp a ring of PROBE_STAGES units,
// each the 4 sub-tiles' probe positions (4 x 1 KB), in dynamic shared memory.
constexpr int PROBE_STAGES = 3;
constexpr int PROBE_UNIT_BYTES = 4 * 1024;
constexpr size_t PROBE_RING_BYTES = (size_t)PROBE_WARPS * PROBE_STAGES * PROBE_UNIT_BYTES;

struct ProbeRow {
    uint4 k[2 * NB];  // the row's 128 int8 codes, block by block
    float kst;        // its stored K maximum
    bool valid;
};

// TMA: the probe rows come in by tensor copies into a per-warp ring of shared
// memory (more bytes in flight per SM than registers can hold); valid when
// block = 4 * probe, where pass q of a block reads positions 0..7 (tokens 0, 4,
// .., 28) of its sub-tile q -- 4 runs of 256 bytes, 1 KB apart, one box.
template <int G, bool TMA>
__global__ void __launch_bounds__(PROBE_WARPS * 32, 2)
    kq8_probe_kernel(const __grid_constant__ SparseParams P) {
    __shared__ __align__(16) int8_t qi[G][HD];
    __shared__ float qsc[G][NB];
    __shared__ int32_t pages[PROBE_MAX_PAGES];
    __shared__ float best[PROBE_MAX_BPC][G];
    __shared__ SelectSmem sel_smem;
    __shared__ __align__(8) uint64_t pbar[TMA ? PROBE_WARPS : 1][PROBE_STAGES];
    extern __shared__ __align__(1024) uint8_t probe_ring[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    // the attention kernel after this one may become resident as soon as every
    // probe CTA has started; it waits for this grid's completion before it
    // reads global memory
    griddep_launch_dependents();
    // A programmatic launch: until griddep_wait() returns, the kernel before
    // this one on the stream (this library's or any other code's, when it
    // signals its dependents early) may still be writing anything this kernel
    // reads -- Q, the lengths, the page table, the KV -- so before it only this
    // CTA's own barriers are set up.
    if (TMA) {
        if (lane == 0)
            for (int i = 0; i < PROBE_STAGES; i++) mbar_init(&pbar[warp][i], 1);
        if (threadIdx.x == 0)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&P.kmap))
                         : "memory");
        fence_barrier_init();
    }
    griddep_wait();
    // Loads that do not depend on the length go out with it: the Q rows and
    // (unless rows map to sequences through row_seq) the page ids this CTA's
    // blocks can span: pages pg0 .. pg0 + ceil(probe_bpc * block / kv_bs)
    static_assert(G <= PROBE_WARPS, "one Q row per warp");
    static_assert(PROBE_MAX_PAGES % (PROBE_WARPS * 32) == 0, "page ids per thread");
    constexpr int PPT = PROBE_MAX_PAGES / (PROBE_WARPS * 32);
    const int j0 = blockIdx.x * P.probe_bpc;
    const int pg0 = (j0 * P.block) / kv_bs;
    const bool pg_early = P.row_seq == nullptr;
    const int span = (P.probe_bpc * P.block + kv_bs - 1) / kv_bs;
    int32_t pspec[PPT];
#pragma unroll
    for (int k = 0; k < PPT; k++) {
        const int i = threadIdx.x + k * PROBE_WARPS * 32;
        pspec[k] = -1;
        if (pg_early && i <= span && pg0 + i < P.max_pages)
            pspec[k] = P.page_table[(size_t)b * P.max_pages + pg0 + i];
    }
    float4 qx = make_float4(0.f, 0.f, 0.f, 0.f);
    if (warp < G)
        qx = reinterpret_cast<const float4*>(
            P.q + ((size_t)b * P.nq + (size_t)h * G + warp) * HD)[lane];
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
    if (P.tickets && nblk <= P.topk) {
        // every block is kept whatever its score: the selection is blocks 0 ..
        // nblk - 1 in order for every head, the union every tile (no scores are
        // needed; with tickets nothing after this kernel reads them)
        if (blockIdx.x == 0) {
            if (P.sel_blocks)
                for (int g = 0; g < G; g++) {
                    int32_t* sel = P.sel_blocks + ((size_t)b * P.nq + (size_t)h * G + g) * P.topk;
                    for (int i = threadIdx.x; i < P.topk; i += PROBE_WARPS * 32)
                        sel[i] = i < nblk ? i : -1;
                }
            gated_list<G>(P, b, h, n);
        }
        return;
    }
    if (j0 >= nblk) return;
    const int j1 = min(j0 + P.probe_bpc, nblk);
    const int pg1 = (min(j1 * P.block, n) - 1) / kv_bs;

    const size_t pt_row = (size_t)(pg_early ? b : P.row_seq[b]) * P.max_pages;
#pragma unroll
    for (int k = 0; k < PPT; k++) {
        const int i = threadIdx.x + k * PROBE_WARPS * 32;
        if (i <= pg1 - pg0) {
            const int32_t pg = pg_early ? pspec[k] : P.page_table[pt_row + pg0 + i];
            const bool ok = pg >= 0 && pg < P.cache.num_pages;
            if (!ok && P.status) atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
            pages[i] = ok ? pg : -1;
        }
    }
    for (int i = threadIdx.x; i < (j1 - j0) * G; i += PROBE_WARPS * 32)
        best[i / G][i % G] = -INFINITY;
    if (warp < G) {
        float qs;
        const uint32_t codes = quantize_q_lane(qx, qs);
        reinterpret_cast<uint32_t*>(qi[warp])[lane] = codes;
        if ((lane & 7) == 0) qsc[warp][lane >> 3] = qs;
    }
    __syncthreads();
    // the selection ORs its heads' choices into these blocks' masks (rows of
    // more than 2048 blocks, or the separate top-k kernel; a probe-only call
    // passes none)
    if (P.masks)
        for (int i = threadIdx.x; i < j1 - j0; i += PROBE_WARPS * 32)
            P.masks[(size_t)(b * nkv + h) * P.max_nblk + j0 + i] = 0u;

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
    // R.k[2 bb] holds bytes 16 qh .. + 15 of block bb of the row, R.k[2 bb + 1] the
    // other half (the integer dot does not depend on the order)
    auto compute = [&](const ProbeRow& R, int k, int qh) {
        const int jj = block_of(k);
#pragma unroll
        for (int g = 0; g < G; g++) {
            int d[NB];
#pragma unroll
            for (int bb = 0; bb < NB; bb++) {
                const uint4 qa = *reinterpret_cast<const uint4*>(qi[g] + bb * 32 + qh * 16);
                const uint4 qb = *reinterpret_cast<const uint4*>(qi[g] + bb * 32 + (qh ^ 1) * 16);
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
    if constexpr (TMA) {
        constexpr int NS = PROBE_STAGES;
        uint8_t* ring = probe_ring + (size_t)warp * NS * PROBE_UNIT_BYTES;
        const int subs = kv_bs / TILE;
        const int hs = (pr >> 2) & 1;  // half order: conflict-free shared loads
        // this lane's probe row of unit k: token t, page pg; false if none
        auto row_of = [&](int k, int& t, int& pg) {
            const int jj = block_of(k), pass = k / my_groups;
            t = jj * P.block + (8 * pass + pr) * 4;
            pg = (jj < j1 && t < n) ? pages[t / kv_bs - pg0] : -1;
            return pg >= 0;
        };
        // all lanes: the row's stored maximum (returned); lane 0: the copies of
        // the unit's sub-tiles (lane 8gb's row is its sub-tile's first)
        auto issue = [&](int k, int s) -> float {
            int t, pg;
            const bool ok = row_of(k, t, pg);
            float kst = 0.0f;
            if (ok)
                kst = __ldg(P.cache.kscale +
                            scale_sub_off(pg, h, nkv, kv_bs, (t % kv_bs) / TILE) + t % TILE);
            const uint32_t copy = __ballot_sync(0xffffffffu, ok && pr == 0);
            int zc[4];
#pragma unroll
            for (int g4 = 0; g4 < 4; g4++) {
                const int tg = __shfl_sync(0xffffffffu, t, 8 * g4);
                const int pgg = __shfl_sync(0xffffffffu, pg, 8 * g4);
                zc[g4] = (int)page_head(pgg, h, nkv) * subs + (tg % kv_bs) / TILE;
            }
            if (lane == 0) {
                uint64_t* bar = &pbar[warp][s];
                mbar_arrive_expect_tx(bar, (uint32_t)__popc(copy) * 1024u);
                const uint64_t pol = l2_evict_first_policy();  // read once
#pragma unroll
                for (int g4 = 0; g4 < 4; g4++)
                    if (copy & (1u << (8 * g4)))
                        tma_load_3d(ring + s * PROBE_UNIT_BYTES + g4 * 1024, &P.kmap, 0, 0,
                                    zc[g4], bar, pol);
            }
            return kst;
        };
        float scr[NS];  // the rows' stored maxima of the units in flight
#pragma unroll
        for (int i = 0; i < NS; i++) scr[i] = (i < nunits) ? issue(i, i) : 0.0f;
        int k = 0;
        bool failed = false;
        for (; k < nunits; k++) {
            const int s = k % NS;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&pbar[warp][s], (k / NS) & 1))) {
                failed = true;
                break;
            }
            ProbeRow R;
            int t, pg;
            R.valid = row_of(k, t, pg);
            R.kst = scr[0];
            const uint8_t* row = ring + s * PROBE_UNIT_BYTES + gb * 1024 + pr * 32;
#pragma unroll
            for (int bb = 0; bb < NB; bb++) {
                R.k[2 * bb] = *reinterpret_cast<const uint4*>(row + bb * 256 + hs * 16);
                R.k[2 * bb + 1] = *reinterpret_cast<const uint4*>(row + bb * 256 + (hs ^ 1) * 16);
            }
            compute(R, k, hs);
#pragma unroll
            for (int i = 0; i + 1 < NS; i++) scr[i] = scr[i + 1];
            __syncwarp();
            if (k + NS < nunits) scr[NS - 1] = issue(k + NS, s);
        }
        if (failed) {
            if (lane == 0 && P.status) atomicOr(P.status, KQ8_STATUS_TIMEOUT);
            // let the copies still in flight land before the CTA leaves
            for (int j = k; j < nunits && j < k + NS; j++)
                __all_sync(0xffffffffu, mbar_wait_bounded(&pbar[warp][j % NS], (j / NS) & 1));
        }
    } else {
        ProbeRow A, Bu;
        if (nunits > 0) load(A, 0);
        for (int k = 0; k < nunits; k += 2) {
            if (k + 1 < nunits) load(Bu, k + 1);
            compute(A, k, 0);
            if (k + 1 >= nunits) break;
            if (k + 2 < nunits) load(A, k + 2);
            compute(Bu, k + 1, 0);
        }
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
__global__ void __launch_bounds__(TOPK_THREADS)
    kq8_topk_kernel(const __grid_constant__ SparseParams P) {
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
