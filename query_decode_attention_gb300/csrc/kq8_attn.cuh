// kq8_attn.cuh -- the split-KV one-pass attention kernel and the chunk merge.
//
// Work decomposition: CTA = (KV chunk, KV head h, sequence b), 4 warps.  A
// chunk is a run of `chunk_tiles` 32-token sub-tiles; warp w of the CTA takes
// the chunk's tiles w, w+4, ...  All G query heads of KV head h are handled by
// the same warp, so each K/V byte is read from HBM once for the whole group.
//
// Per warp, a ring of NS shared-memory stages is filled by bulk-async copies
// (one elected lane issues them, completion on an mbarrier per stage) while
// the warp computes on older stages.  Per tile:
//   score phase (lane = token): int32 block dots of the token's K row with
//     the G int8 query rows (dp4a), the fp32 score in the exact order of the
//     method, tile max across the warp, online-softmax rescale when the
//     running max grows, w = exp(s - M);
//   value phase (lane = 16 bytes of a V row, 4 rows per instruction): int8 ->
//     fp32 by byte permutes and a packed subtract, acc += v * (w * vs) with
//     packed FMAs.
// The 4 warps' (M, S, acc) are merged in shared memory; a chunk that covers
// the whole sequence writes out = acc / S directly, others write an
// unnormalised partial (M, S, acc) that kq8_merge_kernel combines by its
// log-sum-exp (the same algebra as the online rescale, article 9-2 §1).
#pragma once

#include "kq8_common.cuh"

namespace kq8 {

constexpr int ATTN_WARPS = 4;
constexpr int ATTN_THREADS = ATTN_WARPS * 32;

struct AttnParams {
    float* out;
    const float* q;
    kq8_cache_t cache;
    const int32_t* page_table;
    int32_t max_pages;
    const int32_t* seq_lens;
    int32_t max_seq_len;
    int32_t B, nq;
    float scale;
    int32_t chunk_tiles;   // multiple of ATTN_WARPS
    int32_t num_chunks;    // grid.x
    float* part_acc;       // [B][nq][num_chunks][HD]
    float2* part_ms;       // [B][nq][num_chunks] (M, S)
    uint32_t* status;
    // block-sparse tile lists (SPARSE only): entry = tile | head_mask << 24
    const int32_t* tile_list;  // [B][nkv][list_cap]
    const int32_t* list_len;   // [B][nkv]
    int32_t list_cap;
};

template <int G>
struct AttnShape {
    static constexpr int E = (G <= 4) ? 16 : 8;        // V elements per lane
    static constexpr int NC = HD / E;                   // lanes per V row
    static constexpr int TG = 32 / NC;                  // V rows per instruction
    static constexpr int GP = (G <= 4) ? 4 : 8;         // padded heads in p rows
};

template <int G, int NS>
struct AttnSmem {
    alignas(128) uint8_t stage[ATTN_WARPS][NS][STAGE_BYTES];
    alignas(16) float p[ATTN_WARPS][TILE][AttnShape<G>::GP];
    alignas(16) int8_t qi[G][HD];
    alignas(16) float qsc[G][NB];
    alignas(8) uint64_t bar[ATTN_WARPS][NS];
};

// Number of list entries (tiles) of sequence b / KV head h.
template <bool SPARSE>
__device__ __forceinline__ int attn_entries(const AttnParams& P, int b, int h, int n) {
    if (SPARSE) return P.list_len[b * P.cache.num_kv_heads + h];
    return (n + TILE - 1) / TILE;
}

__device__ __forceinline__ int valid_seq_len(const AttnParams& P, int b) {
    int n = P.seq_lens[b];
    if (n < 0 || n > P.max_seq_len) return -1;
    return n;
}

template <int G, int NS, bool SPARSE>
__global__ void __launch_bounds__(ATTN_THREADS, 2) kq8_attn_kernel(const AttnParams P) {
    using Sh = AttnShape<G>;
    constexpr int E = Sh::E, NC = Sh::NC, TG = Sh::TG, GP = Sh::GP;
    constexpr int EP = E / 2;  // float2 pairs per head per lane
    extern __shared__ __align__(128) uint8_t smem_raw[];
    AttnSmem<G, NS>& S = *reinterpret_cast<AttnSmem<G, NS>*>(smem_raw);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    const int subs = kv_bs / TILE;

    int n = valid_seq_len(P, b);
    if (n < 0) {
        if (threadIdx.x == 0 && chunk == 0 && h == 0) atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
        n = 0;
    }
    const int entries = (n == 0) ? 0 : attn_entries<SPARSE>(P, b, h, n);
    const int nch = max(1, (entries + P.chunk_tiles - 1) / P.chunk_tiles);
    if (chunk >= nch) return;
    const int e0 = chunk * P.chunk_tiles;
    const int e1 = min(e0 + P.chunk_tiles, entries);
    const int32_t* list = SPARSE ? P.tile_list + (size_t)(b * nkv + h) * P.list_cap : nullptr;

    // ---- prologue: quantise the G query heads once (article 9-2 §2 seg. 1)
    for (int g = warp; g < G; g += ATTN_WARPS) {
        const float4 x =
            reinterpret_cast<const float4*>(P.q + ((size_t)b * P.nq + (size_t)h * G + g) * HD)[lane];
        float qs;
        const uint32_t codes = quantize_q_lane(x, qs);
        reinterpret_cast<uint32_t*>(S.qi[g])[lane] = codes;
        if ((lane & 7) == 0) S.qsc[g][lane >> 3] = qs;
    }
    if (lane == 0)
        for (int s = 0; s < NS; s++) mbar_init(&S.bar[warp][s], 1);
    fence_barrier_init();
    __syncthreads();

    const int mine = (e1 - e0 > warp) ? (e1 - e0 - warp + ATTN_WARPS - 1) / ATTN_WARPS : 0;
    const uint64_t pol = l2_evict_first_policy();

    // entry i of this warp -> (tile, head mask, page); page < 0 when invalid
    auto entry_of = [&](int i, int& tile, uint32_t& mask) {
        const int e = e0 + warp + ATTN_WARPS * i;
        if (SPARSE) {
            const int32_t v = list[e];
            tile = v & 0xFFFFFF;
            mask = (uint32_t)v >> 24;
        } else {
            tile = e;
            mask = 0xFFu;
        }
    };
    auto page_of = [&](int tile) -> int32_t {
        const int32_t pg = P.page_table[(size_t)b * P.max_pages + tile / subs];
        return (pg >= 0 && pg < P.cache.num_pages) ? pg : -1;
    };
    auto issue = [&](int i) {  // lane 0 only
        int tile;
        uint32_t mask;
        entry_of(i, tile, mask);
        const int32_t pg = page_of(tile);
        uint64_t* bar = &S.bar[warp][i % NS];
        if (pg < 0) {
            atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
            mbar_arrive_expect_tx(bar, 0);  // completes the phase with no data
            return;
        }
        const int sub = tile % subs;
        uint8_t* st = S.stage[warp][i % NS];
        const size_t kvo = kv_sub_off(pg, h, nkv, kv_bs, sub);
        const size_t so = scale_sub_off(pg, h, nkv, kv_bs, sub);
        mbar_arrive_expect_tx(bar, STAGE_BYTES);
        bulk_g2s(st, P.cache.k + kvo, SUB_K_BYTES, bar, pol);
        bulk_g2s(st + SUB_K_BYTES, P.cache.v + kvo, SUB_V_BYTES, bar, pol);
        bulk_g2s(st + SUB_K_BYTES + SUB_V_BYTES, P.cache.kscale + so, SUB_S_BYTES, bar, pol);
        bulk_g2s(st + SUB_K_BYTES + SUB_V_BYTES + SUB_S_BYTES, P.cache.vscale + so, SUB_S_BYTES,
                 bar, pol);
    };

    if (lane == 0)
        for (int i = 0; i < NS && i < mine; i++) issue(i);

    float M[G], Sl[G];
    float2 acc[G][EP];
#pragma unroll
    for (int g = 0; g < G; g++) {
        M[g] = M_INIT;
        Sl[g] = 0.0f;
#pragma unroll
        for (int e = 0; e < EP; e++) acc[g][e] = make_float2(0.0f, 0.0f);
    }
    float qsc_r[G][NB];
#pragma unroll
    for (int g = 0; g < G; g++)
#pragma unroll
        for (int bb = 0; bb < NB; bb++) qsc_r[g][bb] = S.qsc[g][bb];

    const float scale = P.scale;
    bool failed = false;
    int i = 0;
    for (; i < mine; i++) {
        int tile;
        uint32_t mask;
        entry_of(i, tile, mask);
        const bool ok_page = page_of(tile) >= 0;
        if (!mbar_wait_bounded(&S.bar[warp][i % NS], (i / NS) & 1)) {
            failed = true;
            break;
        }
        if (ok_page) {
            const uint8_t* st = S.stage[warp][i % NS];
            const int8_t* kst = reinterpret_cast<const int8_t*>(st);
            const int8_t* vst = reinterpret_cast<const int8_t*>(st + SUB_K_BYTES);
            const float* kss = reinterpret_cast<const float*>(st + SUB_K_BYTES + SUB_V_BYTES);
            const float* vss = kss + TILE;

            // ---- score phase: lane t scores token tile*32 + t for all G heads
            const int t = lane;
            const bool live = tile * TILE + t < n;
            int dot[G][NB];
            const int hs = (t >> 2) & 1;  // half order that keeps the loads conflict-free
#pragma unroll
            for (int bb = 0; bb < NB; bb++) {
                const uint4 kA =
                    *reinterpret_cast<const uint4*>(kst + bb * 1024 + t * 32 + hs * 16);
                const uint4 kB =
                    *reinterpret_cast<const uint4*>(kst + bb * 1024 + t * 32 + (hs ^ 1) * 16);
#pragma unroll
                for (int g = 0; g < G; g++) {
                    const uint4 qA =
                        *reinterpret_cast<const uint4*>(S.qi[g] + bb * 32 + hs * 16);
                    const uint4 qB =
                        *reinterpret_cast<const uint4*>(S.qi[g] + bb * 32 + (hs ^ 1) * 16);
                    int d = __dp4a((int)kA.x, (int)qA.x, 0);
                    d = __dp4a((int)kA.y, (int)qA.y, d);
                    d = __dp4a((int)kA.z, (int)qA.z, d);
                    d = __dp4a((int)kA.w, (int)qA.w, d);
                    d = __dp4a((int)kB.x, (int)qB.x, d);
                    d = __dp4a((int)kB.y, (int)qB.y, d);
                    d = __dp4a((int)kB.z, (int)qB.z, d);
                    d = __dp4a((int)kB.w, (int)qB.w, d);
                    dot[g][bb] = d;
                }
            }
            const float ksv = kss[t];
            const float vstep = __fmul_rn(vss[t], inv127());
            float pw[GP];
#pragma unroll
            for (int g = 0; g < GP; g++) pw[g] = 0.0f;
#pragma unroll
            for (int g = 0; g < G; g++) {
                const bool on = live && ((mask >> g) & 1u);
                const float s = on ? score_exact(dot[g], qsc_r[g], ksv, scale) : -INFINITY;
                const float mt = warp_max(s);
                const float mn = fmaxf(M[g], mt);
                if (mn > M[g]) {  // warp-uniform: rescale what was accumulated
                    const float c = expf(M[g] - mn);
                    Sl[g] *= c;
#pragma unroll
                    for (int e = 0; e < EP; e++) fmul2(acc[g][e], c);
                    M[g] = mn;
                }
                const float w = on ? expf(s - mn) : 0.0f;
                Sl[g] += w;
                pw[g] = on ? w * vstep : 0.0f;
            }
            float* prow = S.p[warp][t];
#pragma unroll
            for (int g4 = 0; g4 < GP; g4 += 4)
                *reinterpret_cast<float4*>(prow + g4) =
                    make_float4(pw[g4], pw[g4 + 1], pw[g4 + 2], pw[g4 + 3]);
            __syncwarp();

            // ---- value phase: lane (tg, c) covers elements c*E.. of rows tg, tg+TG, ...
            const int tg = lane / NC, c = lane % NC;
#pragma unroll 2
            for (int r = tg; r < TILE; r += TG) {
                float f[E];
                if (E == 16) {
                    const uint4 vv = *reinterpret_cast<const uint4*>(vst + r * HD + c * 16);
                    i8x4_to_f32(vv.x, f[0], f[1], f[2], f[3]);
                    i8x4_to_f32(vv.y, f[4], f[5], f[6], f[7]);
                    i8x4_to_f32(vv.z, f[8], f[9], f[10], f[11]);
                    i8x4_to_f32(vv.w, f[12], f[13], f[14], f[15]);
                } else {
                    const uint2 vv = *reinterpret_cast<const uint2*>(vst + r * HD + c * 8);
                    i8x4_to_f32(vv.x, f[0], f[1], f[2], f[3]);
                    i8x4_to_f32(vv.y, f[4], f[5], f[6], f[7]);
                }
                float pr[GP];
#pragma unroll
                for (int g4 = 0; g4 < GP; g4 += 4) {
                    const float4 pp = *reinterpret_cast<const float4*>(&S.p[warp][r][g4]);
                    pr[g4] = pp.x;
                    pr[g4 + 1] = pp.y;
                    pr[g4 + 2] = pp.z;
                    pr[g4 + 3] = pp.w;
                }
#pragma unroll
                for (int g = 0; g < G; g++)
#pragma unroll
                    for (int e = 0; e < EP; e++) ffma2(acc[g][e], f[2 * e], f[2 * e + 1], pr[g]);
            }
        }
        __syncwarp();
        if (lane == 0 && i + NS < mine) issue(i + NS);
    }
    if (failed) {
        if (lane == 0) atomicOr(P.status, KQ8_STATUS_TIMEOUT);
        // let the copies this warp still has in flight land before leaving
        for (int j = i; j < mine && j < i + NS; j++) mbar_wait_bounded(&S.bar[warp][j % NS], (j / NS) & 1);
#pragma unroll
        for (int g = 0; g < G; g++) {
            M[g] = M_INIT;
            Sl[g] = 0.0f;
#pragma unroll
            for (int e = 0; e < EP; e++) acc[g][e] = make_float2(0.0f, 0.0f);
        }
    }

    // ---- reduce the lanes of a warp: V rows were split over TG lane groups
#pragma unroll
    for (int g = 0; g < G; g++) {
#pragma unroll
        for (int o = NC; o < 32; o <<= 1)
#pragma unroll
            for (int e = 0; e < EP; e++) {
                acc[g][e].x += __shfl_xor_sync(0xffffffffu, acc[g][e].x, o);
                acc[g][e].y += __shfl_xor_sync(0xffffffffu, acc[g][e].y, o);
            }
        Sl[g] = warp_sum(Sl[g]);
    }

    // ---- merge the 4 warps in shared memory (reuses the stage buffers)
    __syncthreads();
    float* macc = reinterpret_cast<float*>(S.stage);                  // [W][G][HD]
    float2* mms = reinterpret_cast<float2*>(macc + ATTN_WARPS * G * HD);  // [W][G]
    if (lane < NC) {
#pragma unroll
        for (int g = 0; g < G; g++)
#pragma unroll
            for (int e = 0; e < EP; e++)
                *reinterpret_cast<float2*>(&macc[(warp * G + g) * HD + lane * E + 2 * e]) =
                    acc[g][e];
    }
    if (lane == 0)
#pragma unroll
        for (int g = 0; g < G; g++) mms[warp * G + g] = make_float2(M[g], Sl[g]);
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
            const float f = expf(ms.x - mx);
            ssum += ms.y * f;
            a += macc[(w * G + g) * HD + d] * f;
        }
        const size_t row = (size_t)b * P.nq + (size_t)h * G + g;
        if (nch == 1) {
            P.out[row * HD + d] = (ssum > 0.0f) ? a / ssum : 0.0f;
        } else {
            const size_t pr = row * P.num_chunks + chunk;
            P.part_acc[pr * HD + d] = a;
            if (d == 0) P.part_ms[pr] = make_float2(mx, ssum);
        }
    }
}

// Combine the partials of sequences split over several chunks:
//   M = max_c m_c, out = sum_c acc_c e^(m_c - M) / sum_c S_c e^(m_c - M).
template <bool SPARSE>
__global__ void __launch_bounds__(HD) kq8_merge_kernel(const AttnParams P) {
    const int row = blockIdx.x;  // b * nq + hq
    const int b = row / P.nq, hq = row % P.nq;
    const int G = P.nq / P.cache.num_kv_heads;
    const int h = hq / G;
    const int n = valid_seq_len(P, b);
    if (n <= 0) return;
    const int entries = attn_entries<SPARSE>(P, b, h, n);
    const int nch = (entries + P.chunk_tiles - 1) / P.chunk_tiles;
    if (nch <= 1) return;
    const size_t base = (size_t)row * P.num_chunks;
    float mx = M_INIT;
    for (int c = 0; c < nch; c++) mx = fmaxf(mx, P.part_ms[base + c].x);
    float ssum = 0.0f, a = 0.0f;
    for (int c = 0; c < nch; c++) {
        const float2 ms = P.part_ms[base + c];
        const float f = expf(ms.x - mx);
        ssum += ms.y * f;
        a += P.part_acc[(base + c) * HD + threadIdx.x] * f;
    }
    P.out[(size_t)row * HD + threadIdx.x] = (ssum > 0.0f) ? a / ssum : 0.0f;
}

}  // namespace kq8
