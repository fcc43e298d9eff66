// kq8_prefill.cu -- batched causal prefill attention over the q8 cache on the
// 5th-generation tensor cores.
//
// Article 10-1 §1 ("why long context must be sparse"): a batch of nb new
// tokens scores against the whole history, an nb x n score matrix; §2 names
// the exact batched kernel the prefill gate falls back to.  Each query is
// computed like one decode query (article 9-2 §2): Q quantised once in
// 32-element max-abs blocks, score = ((sum_b dot_b * qsc_b) * ks) * scale with
// int32 block dots, one-pass online softmax, one divide at the end.  Query i
// of a sequence with nb new tokens and n cached tokens sits at position
// n - nb + i and sees tokens 0 .. n - nb + i.
//
// GB300 mapping.  A CTA takes 128 (token, query head) rows of one sequence and
// one KV head -- 128 / G consecutive new tokens x the G query heads sharing
// the KV head -- and walks the KV history in 32-token cache sub-tiles:
//   1. K and V codes are read once per CTA and widened exactly to 16-bit
//      (K -> fp16, V -> bf16; every int8 is exact in both) into the
//      tensor-core operand layout in shared memory.
//   2. S: four MMAs pairs (M = 128, N = 32, K = 16) per sub-tile, one per
//      32-element quantisation block, each into its own TMEM accumulator, so
//      every block dot is the exact integer (|sum| < 2^19 in fp32).
//   3. Each thread owns one row (one TMEM lane): it forms the scores from the
//      four block dots exactly as a decode query does, runs the online
//      softmax (rescaling its O row in TMEM only when the running max grows
//      by more than 2^8), and writes the weights w = p * vscale / 127 as a bf16
//      high part and a bf16 remainder (w = hi + lo to 2^-17 relative).
//   4. O += W_hi V + W_lo V: four MMAs (M = 128, N = 128, K = 16) into a
//      128-column TMEM accumulator that lives for the whole CTA.
// One thread issues every MMA; completion comes back through mbarriers.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kq8_internal.h"
#include "kq8_tc.cuh"

namespace kq8 {
namespace {

constexpr int PF_THREADS = 128;
constexpr int PF_ROWS = 128;             // MMA M: (token, head) rows per CTA
constexpr int PF_NT = TILE;              // KV tokens per step: one cache sub-tile
constexpr uint32_t PF_TMEM_COLS = 256;   // O (128 columns) + 4 block-dot accumulators (32 each)
constexpr uint32_t PF_COL_D = 128;       // first block-dot column

// Shared memory map (bytes).  Every operand is K-major without swizzle: 8-row
// x 16-byte core matrices, 128 B each, rows of a core matrix adjacent.  K, V,
// the weights and the per-token scales are double-buffered by sub-tile parity
// so that the tensor core works on one sub-tile while the CUDA cores prepare
// the next.
constexpr uint32_t SM_Q = 0;             // fp16 Q codes: 128 rows x 128 dims (32 KB)
constexpr uint32_t SM_K = 32768;         // 2 x fp16 K codes: 32 tokens x 128 dims (8 KB each)
constexpr uint32_t SM_V = 49152;         // 2 x bf16 V codes: 128 dims x 32 tokens (8 KB each)
constexpr uint32_t SM_W = 65536;         // 2 x (bf16 weights hi, lo): 128 rows x 32 tokens (16 KB)
constexpr uint32_t SM_SC = 98304;        // 2 x (32 score multipliers, 32 value steps) (256 B)
constexpr uint32_t SM_BAR = 98816;       // two mbarriers: S done, PV done
constexpr uint32_t SM_TMEM = 98832;      // TMEM base address written by the allocator
// 97 KB per CTA: two CTAs per SM, which is what two 256-column TMEM
// allocations allow (a third would wait in the allocator).
constexpr uint32_t PF_SMEM = 99328;

__device__ __forceinline__ uint32_t sm_k(int p) { return SM_K + 8192u * p; }
__device__ __forceinline__ uint32_t sm_v(int p) { return SM_V + 8192u * p; }
__device__ __forceinline__ uint32_t sm_whi(int p) { return SM_W + 16384u * p; }
__device__ __forceinline__ uint32_t sm_wlo(int p) { return SM_W + 16384u * p + 8192u; }
__device__ __forceinline__ uint32_t sm_km(int p) { return SM_SC + 256u * p; }
__device__ __forceinline__ uint32_t sm_vs(int p) { return SM_SC + 256u * p + 128u; }

constexpr size_t PF_STATUS_BYTES = 256;  // workspace: the status word (256-byte slot)

constexpr float PF_LOG2E = 1.4426950408889634f;
constexpr float PF_RESCALE_SLACK = 8.0f;  // log2 units: rescale O when the max grows > 2^8

// Byte offset of the 16-byte chunk holding elements 8*kc .. 8*kc+7 of row r in
// a K-major operand of R rows: core matrices adjacent along K are R*16 B apart
// (leading byte offset), along the rows 128 B apart (stride byte offset).
__device__ __forceinline__ uint32_t cm_off(int r, int kc, int R) {
    return (uint32_t)(kc * R * 16 + (r >> 3) * 128 + (r & 7) * 16);
}

__device__ __forceinline__ float pf_ex2(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two int8 codes (bytes 2*which, 2*which+1 of w) -> two exact fp16 values:
// offset-binary byte u = c + 128 in the mantissa of 1024, minus 1152.
__device__ __forceinline__ uint32_t i8x2_to_h2(uint32_t w, int which) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t x = __byte_perm(u, 0x64646464u, which ? 0x4342u : 0x4140u);
    __half2 hv = *reinterpret_cast<__half2*>(&x);
    hv = __hsub2(hv, __float2half2_rn(1152.0f));
    return *reinterpret_cast<uint32_t*>(&hv);
}

// Read-only global loads kept where they are written (volatile asm): the
// pipeline issues them a whole step before their data is needed, and a
// compiler under register pressure would otherwise sink them next to the use.
__device__ __forceinline__ uint4 ldg_pinned_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}
__device__ __forceinline__ uint32_t ldg_pinned_u32(const void* p) {
    uint32_t r;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(r) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t bf2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t h2_bits(int lo, int hi) {
    __half2 v = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
    return *reinterpret_cast<uint32_t*>(&v);
}

// One 32-token sub-tile of one KV head as this thread holds it in registers
// between the global loads and the shared-memory stores: the K half (with
// the page lookup and the scales) and the V half are loaded one sub-tile
// apart in the pipeline, so each has a whole step to arrive.
struct RawK {
    uint4 k0, k1;     // K codes of token `lane`, dims 32*warp .. 32*warp+31
    float sc;         // kscale (threads 0-31) or vscale (32-63) of token tid % 32
    int32_t pg;       // page id (-1 when out of range)
};
struct RawV {
    uint32_t v[8];    // V codes of tokens 8*warp .. +7, dims 4*lane .. +3
};

}  // namespace

struct PrefillParams {
    float* out;
    const float* q;
    kq8_cache_t cache;
    const int32_t* page_table;
    int32_t max_pages;
    const int32_t* seq_lens;
    const int32_t* q_off;
    int32_t total_q;
    int32_t max_seq_len;
    int32_t max_q_len;
    int32_t B;
    int32_t nq;
    float scale;
    uint32_t* status;
};

template <int G>
__global__ void __launch_bounds__(PF_THREADS, 2) kq8_prefill_kernel(const PrefillParams P) {
    constexpr int TQ = PF_ROWS / G;  // new tokens per CTA
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    const int qt = gridDim.x - 1 - blockIdx.x;  // the longest query tiles start first

    const int n = P.seq_lens[b];
    const int q0 = P.q_off[b];
    const int nb = P.q_off[b + 1] - q0;
    if (n < 0 || n > P.max_seq_len || nb < 0 || nb > n || nb > P.max_q_len || q0 < 0 ||
        (int64_t)q0 + nb > P.total_q) {
        if (tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
        return;
    }
    const int i0 = qt * TQ;
    if (i0 >= nb) return;
    const int ntok = min(TQ, nb - i0);
    const int tq = tid / G, g = tid % G;
    const bool valid = tid < TQ * G && tq < ntok;
    const int pos = valid ? n - nb + i0 + tq : -1;  // this row sees tokens 0 .. pos
    const int ntiles = (n - nb + i0 + ntok - 1) / PF_NT + 1;

    uint64_t* bar_s = reinterpret_cast<uint64_t*>(sm + SM_BAR);
    uint64_t* bar_pv = bar_s + 1;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SM_TMEM);
    if (warp == 0) {
        __syncwarp();
        tc::tmem_alloc(tslot, PF_TMEM_COLS);
    }
    if (tid == 0) {
        mbar_init(bar_s, 1);
        mbar_init(bar_pv, 1);
        fence_barrier_init();
    }

    // ---- Q: quantise this row once (article 9-2 §2 segment 1) -> fp16 codes
    float qsc[NB];
    {
        uint8_t* Qs = sm + SM_Q;
        const float4* src = reinterpret_cast<const float4*>(
            P.q + ((size_t)(q0 + i0 + tq) * P.nq + (size_t)h * G + g) * HD);
#pragma unroll
        for (int blk = 0; blk < NB; blk++) {
            float4 x[8];
#pragma unroll
            for (int i = 0; i < 8; i++) {
                if (valid)
                    x[i] = src[blk * 8 + i];
                else
                    x[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
            float m = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++)
                m = fmaxf(m, fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)),
                                   fmaxf(fabsf(x[i].z), fabsf(x[i].w))));
            if (m < 1e-6f) m = 1.0f;
            qsc[blk] = __fmul_rn(m, inv127());
            const float iq = __fdiv_rn(127.0f, m);
            auto code = [&](float v) -> int {
                float t = __fmul_rn(v, iq);
                t = fminf(fmaxf(t, -128.0f), 127.0f);
                return __float2int_rz(t);
            };
#pragma unroll
            for (int c = 0; c < 4; c++) {
                const float4 a = x[2 * c], e = x[2 * c + 1];
                const uint4 w = make_uint4(h2_bits(code(a.x), code(a.y)),
                                           h2_bits(code(a.z), code(a.w)),
                                           h2_bits(code(e.x), code(e.y)),
                                           h2_bits(code(e.z), code(e.w)));
                *reinterpret_cast<uint4*>(Qs + cm_off(tid, blk * 4 + c, PF_ROWS)) = w;
            }
        }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;
    const uint32_t t_lane = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lanes

    // ---- KV sub-tile loads (global -> registers)
    // per-token score multiplier kscale * (1/127) * scale * log2(e)
    const float kmul = inv127() * P.scale * PF_LOG2E;
    // page ids: lane l of every warp holds the page of sub-tile 32*w + l for
    // the current window w and the next one, so that a page id is a shuffle
    // away and its global load is a whole window ahead of its use
    auto load_window = [&](int w) -> int32_t {
        const int t = 32 * w + lane;
        if (t >= ntiles) return -1;
        const int32_t pg = P.page_table[(size_t)b * P.max_pages + (t * PF_NT) / kv_bs];
        return (pg >= 0 && pg < P.cache.num_pages) ? pg : -1;
    };
    int32_t pw_cur = load_window(0), pw_nxt = load_window(1);
    auto page_of = [&](int t) -> int32_t {  // t = 0, 1, 2, ... in order, warp-uniform
        if ((t & 31) == 0 && t > 0) {
            pw_cur = pw_nxt;
            pw_nxt = load_window((t >> 5) + 1);
        }
        return __shfl_sync(0xffffffffu, pw_cur, t & 31);
    };
    auto load_k = [&](int j, RawK& r) {
        const int t0 = j * PF_NT;
        const int32_t pg = page_of(j);
        r.sc = 0.0f;
        if (pg < 0) {
            r.pg = -1;
            r.k0 = r.k1 = make_uint4(0, 0, 0, 0);
            return;
        }
        r.pg = pg;
        const int sub = (t0 % kv_bs) / PF_NT;
        const size_t kvo = kv_sub_off(pg, h, nkv, kv_bs, sub);
        const uint4* kp =
            reinterpret_cast<const uint4*>(P.cache.k + kvo + warp * 1024 + kpos(lane) * 32);
        r.k0 = ldg_pinned_v4(kp);
        r.k1 = ldg_pinned_v4(kp + 1);
        if (tid < 64 && t0 + (tid & 31) < n) {
            const size_t so = scale_sub_off(pg, h, nkv, kv_bs, sub) + (tid & 31);
            r.sc = __uint_as_float(
                ldg_pinned_u32(tid < 32 ? (const void*)(P.cache.kscale + so)
                                        : (const void*)(P.cache.vscale + so)));
        }
    };
    auto load_v = [&](int j, int32_t pg, RawV& r) {
        if (pg < 0) {
#pragma unroll
            for (int tt = 0; tt < 8; tt++) r.v[tt] = 0;
            return;
        }
        const int t0 = j * PF_NT;
        const size_t kvo = kv_sub_off(pg, h, nkv, kv_bs, (t0 % kv_bs) / PF_NT);
        const uint32_t* vp =
            reinterpret_cast<const uint32_t*>(P.cache.v + kvo + (size_t)warp * 8 * HD) + lane;
#pragma unroll
        for (int tt = 0; tt < 8; tt++) r.v[tt] = ldg_pinned_u32(vp + tt * (HD / 4));
    };
    // registers -> 16-bit operands of buffer p in shared memory
    auto stage_k = [&](const RawK& r, int p) {
        uint8_t* Ks = sm + sm_k(p);
        const uint32_t kw[8] = {r.k0.x, r.k0.y, r.k0.z, r.k0.w, r.k1.x, r.k1.y, r.k1.z, r.k1.w};
#pragma unroll
        for (int c = 0; c < 4; c++)
            *reinterpret_cast<uint4*>(Ks + cm_off(lane, warp * 4 + c, PF_NT)) =
                make_uint4(i8x2_to_h2(kw[2 * c], 0), i8x2_to_h2(kw[2 * c], 1),
                           i8x2_to_h2(kw[2 * c + 1], 0), i8x2_to_h2(kw[2 * c + 1], 1));
        if (tid < 64)
            reinterpret_cast<float*>(sm + (tid < 32 ? sm_km(p) : sm_vs(p)))[tid & 31] =
                __fmul_rn(r.sc, tid < 32 ? kmul : inv127());
    };
    // V is stored transposed (dims as rows, tokens along K): one 16-byte chunk
    // = 8 tokens of one dim.  The dim order is rotated per lane pair so that
    // the eight lanes of each store phase hit eight bank groups.
    auto stage_v = [&](const RawV& r, int p) {
        uint8_t* Vs = sm + sm_v(p);
        uint32_t u[8];
#pragma unroll
        for (int tt = 0; tt < 8; tt++) u[tt] = r.v[tt] ^ 0x80808080u;
        const float2 bias = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
        for (int e = 0; e < 4; e++) {
            const int ee = (e + (lane >> 1)) & 3;
            const uint32_t sel = 0x7540u | (uint32_t)ee;
            float2 f[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; q2++)
                f[q2] = __fadd2_rn(
                    make_float2(__uint_as_float(__byte_perm(u[2 * q2], 0x4B000000u, sel)),
                                __uint_as_float(__byte_perm(u[2 * q2 + 1], 0x4B000000u, sel))),
                    bias);
            *reinterpret_cast<uint4*>(Vs + cm_off(4 * lane + ee, warp, PF_ROWS)) =
                make_uint4(bf2_bits(f[0].x, f[0].y), bf2_bits(f[1].x, f[1].y),
                           bf2_bits(f[2].x, f[2].y), bf2_bits(f[3].x, f[3].y));
        }
    };
    // one thread issues the MMAs of a step
    // Matrix descriptors of every operand buffer, built once; an MMA at K
    // chunk kc adds kc * leading-byte-offset / 16 to the start-address field.
    const uint64_t d_q = tc::sdesc(smem_u32(sm + SM_Q), PF_ROWS * 16, 128);
    const uint64_t d_k0 = tc::sdesc(smem_u32(sm + sm_k(0)), PF_NT * 16, 128);
    const uint64_t d_v0 = tc::sdesc(smem_u32(sm + sm_v(0)), PF_ROWS * 16, 128);
    const uint64_t d_w0 = tc::sdesc(smem_u32(sm + sm_whi(0)), PF_ROWS * 16, 128);
    auto issue_s = [&](int p) {  // D_blk = Q_blk K_blk^T, blk = 0..3 (exact block dots)
        const uint64_t dk = d_k0 + (uint64_t)p * (8192u >> 4);
        constexpr uint32_t ID = tc::IDesc<128, PF_NT, false>::value;
#pragma unroll
        for (int blk = 0; blk < NB; blk++)
#pragma unroll
            for (int kk = 0; kk < 2; kk++) {
                const int kc = blk * 4 + kk * 2;
                tc::mma_f16(tbase + PF_COL_D + 32 * blk, d_q + (uint64_t)(kc * PF_ROWS),
                            dk + (uint64_t)(kc * PF_NT), ID, kk > 0);
            }
        tc::mma_commit(bar_s);
    };
    auto issue_pv = [&](int p, bool accumulate) {  // O (+)= W_hi V + W_lo V
        const uint64_t dv = d_v0 + (uint64_t)p * (8192u >> 4);
        const uint64_t dh = d_w0 + (uint64_t)p * (16384u >> 4), dl = dh + (8192u >> 4);
        constexpr uint32_t ID = tc::IDesc<128, HD, true>::value;
#pragma unroll
        for (int kk = 0; kk < PF_NT / 16; kk++) {
            const uint64_t off = (uint64_t)(kk * 2 * PF_ROWS);  // 2 K chunks, in 16-byte units
            tc::mma_f16(tbase, dh + off, dv + off, ID, accumulate || kk > 0);
            tc::mma_f16(tbase, dl + off, dv + off, ID, true);
        }
        tc::mma_commit(bar_pv);
    };

    // ---- pipeline.  Step j (buffer cur = j & 1, nxt = cur ^ 1):
    //   0. K half of sub-tile j+1 -> buffer nxt (its last reader S(j-1) is done)
    //   1. wait S(j)
    //   2. softmax of sub-tile j -> weights in buffer cur (while PV(j-1) runs)
    //   3. wait PV(j-1); V half of sub-tile j+1 -> buffer nxt
    //   4. barrier; issue S(j+1), then PV(j)
    // Global loads run one step ahead of the stores that consume them.
    float M2 = M_INIT, Mhi = M_INIT + PF_RESCALE_SLACK;
    float2 S2 = make_float2(0.0f, 0.0f);  // running sum, even and odd tokens
    const int pos_first = n - nb + i0;    // position of the CTA's first new token
    bool alive = true;
    uint64_t* fail_bar = nullptr;
    uint32_t fail_par = 0;
    RawK rk;
    RawV rv;
    load_k(0, rk);
    load_v(0, rk.pg, rv);
    stage_k(rk, 0);
    stage_v(rv, 0);
    bool ok_cur = rk.pg >= 0, ok_nxt = false;
    if (ntiles > 1) {
        load_k(1, rk);
        load_v(1, rk.pg, rv);
    }
    tc::fence_smem_to_async();
    __syncthreads();
    if (tid == 0) {
        if (!ok_cur) atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
        tc::fence_after_sync();
        issue_s(0);
    }
    for (int j = 0; j < ntiles; j++) {
        const int cur = j & 1, nxt = cur ^ 1;
        const bool more = j + 1 < ntiles;
        // step 0
        int32_t pg_after = -1;
        if (more) {
            stage_k(rk, nxt);
            ok_nxt = rk.pg >= 0;
            if (j + 2 < ntiles) {
                load_k(j + 2, rk);
                pg_after = rk.pg;
            }
        }
        // step 1
        const bool ok_s = __all_sync(0xffffffffu, mbar_wait_bounded(bar_s, j & 1));
        bool ok_pv = true;
        if (ok_s) {
            tc::fence_after_sync();
            // ---- step 2: scores of this row against the sub-tile (article
            // 9-2 §2 seg. 2): s = sum_b dot_b * qsc_b, times the token's
            // kscale / 127 * scale, in log2 units for ex2
            float2 x[PF_NT / 2];
            {
                float d[PF_NT];
                tc::tmem_ld32(tbase + t_lane + PF_COL_D, d);
                const float2 c0 = make_float2(qsc[0], qsc[0]);
#pragma unroll
                for (int i = 0; i < PF_NT / 2; i++)
                    x[i] = __fmul2_rn(make_float2(d[2 * i], d[2 * i + 1]), c0);
#pragma unroll
                for (int blk = 1; blk < NB; blk++) {
                    tc::tmem_ld32(tbase + t_lane + PF_COL_D + 32 * blk, d);
                    const float2 cb = make_float2(qsc[blk], qsc[blk]);
#pragma unroll
                    for (int i = 0; i < PF_NT / 2; i++)
                        x[i] = __ffma2_rn(make_float2(d[2 * i], d[2 * i + 1]), cb, x[i]);
                }
            }
            const float2* km2 = reinterpret_cast<const float2*>(sm + sm_km(cur));
#pragma unroll
            for (int i = 0; i < PF_NT / 2; i++) x[i] = __fmul2_rn(x[i], km2[i]);
            const int t0 = j * PF_NT;
            // every row of the CTA sees every token of this sub-tile: no masking
            const bool full = ok_cur && t0 + PF_NT - 1 <= pos_first;
            if (!full) {
                const int nvis = ok_cur ? max(0, min(PF_NT, pos - t0 + 1)) : 0;
#pragma unroll
                for (int i = 0; i < PF_NT / 2; i++) {
                    if (2 * i >= nvis) x[i].x = -INFINITY;
                    if (2 * i + 1 >= nvis) x[i].y = -INFINITY;
                }
            }
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < PF_NT / 2; i++) mt = fmaxf(mt, fmaxf(x[i].x, x[i].y));
            // lazy rescale of S and of this row of O (online-softmax max);
            // O is read only after PV(j-1) has landed
            const bool need = mt > Mhi;
            float cf = 1.0f;
            if (need) {
                cf = pf_ex2(M2 - mt);
                S2 = __fmul2_rn(S2, make_float2(cf, cf));
                M2 = mt;
                Mhi = mt + PF_RESCALE_SLACK;
            }
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                ok_pv = __all_sync(0xffffffffu, mbar_wait_bounded(bar_pv, (j - 1) & 1));
                if (ok_pv) {
                    tc::fence_after_sync();
#pragma unroll 1
                    for (int c = 0; c < HD / 32; c++) {
                        float o[32];
                        tc::tmem_ld32(tbase + t_lane + 32 * c, o);
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] = __fmul_rn(o[i], cf);
                        tc::tmem_st32(tbase + t_lane + 32 * c, o);
                    }
                }
            }
            // weights w = p * vscale / 127 = hi + lo: hi is w cut to bf16 (its
            // top 16 bits), lo = w - hi (exact) rounded to bf16
            uint8_t* Wh = sm + sm_whi(cur);
            uint8_t* Wl = sm + sm_wlo(cur);
            const float2* vs2 = reinterpret_cast<const float2*>(sm + sm_vs(cur));
            const float2 negm = make_float2(-M2, -M2);
#pragma unroll
            for (int c = 0; c < PF_NT / 8; c++) {
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int u2 = 0; u2 < 4; u2++) {
                    const int i = 4 * c + u2;
                    const float2 y = __fadd2_rn(x[i], negm);  // -inf (masked) -> ex2 = 0
                    const float2 pr = make_float2(pf_ex2(y.x), pf_ex2(y.y));
                    S2 = __fadd2_rn(S2, pr);
                    const float2 w = __fmul2_rn(pr, vs2[i]);
                    const uint32_t wx = __float_as_uint(w.x), wy = __float_as_uint(w.y);
                    hi[u2] = __byte_perm(wx, wy, 0x7632);
                    const float2 r = __fadd2_rn(w, make_float2(-__uint_as_float(wx & 0xFFFF0000u),
                                                               -__uint_as_float(wy & 0xFFFF0000u)));
                    lo[u2] = bf2_bits(r.x, r.y);
                }
                *reinterpret_cast<uint4*>(Wh + cm_off(tid, c, PF_ROWS)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(Wl + cm_off(tid, c, PF_ROWS)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
        }
        // step 3
        if (ok_s && ok_pv && j > 0)
            ok_pv = __all_sync(0xffffffffu, mbar_wait_bounded(bar_pv, (j - 1) & 1));
        if (ok_s && ok_pv && more) {
            stage_v(rv, nxt);
            if (j + 2 < ntiles) load_v(j + 2, pg_after, rv);
        }
        // step 4
        tc::fence_before_sync();
        tc::fence_smem_to_async();
        if (!__syncthreads_and(ok_s && ok_pv)) {
            alive = false;
            fail_bar = ok_s ? bar_pv : bar_s;
            fail_par = ok_s ? (uint32_t)((j - 1) & 1) : (uint32_t)(j & 1);
            break;
        }
        if (tid == 0) {
            tc::fence_after_sync();
            if (more) {
                if (!ok_nxt) atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
                issue_s(nxt);
            }
            issue_pv(cur, j > 0);
        }
        ok_cur = ok_nxt;
    }

    if (alive) {
        const bool ok = mbar_wait_bounded(bar_pv, (ntiles - 1) & 1);
        if (!__syncthreads_and(ok)) {
            alive = false;
            fail_bar = bar_pv;
            fail_par = (ntiles - 1) & 1;
        }
    }
    if (alive) {
        tc::fence_after_sync();
        __syncwarp();
        const float S = S2.x + S2.y;
        const float inv_ok = S > 0.0f ? 1.0f : 0.0f;  // no visible token: 0 (pages' empty case)
        const float Sd = S > 0.0f ? S : 1.0f;
        float* dst = P.out + ((size_t)(q0 + i0 + tq) * P.nq + (size_t)h * G + g) * HD;
#pragma unroll 1
        for (int c = 0; c < HD / 32; c++) {
            float o[32];
            tc::tmem_ld32(tbase + t_lane + 32 * c, o);
            if (valid) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(dst + 32 * c + i) =
                        make_float4(__fdiv_rn(o[i], Sd) * inv_ok, __fdiv_rn(o[i + 1], Sd) * inv_ok,
                                    __fdiv_rn(o[i + 2], Sd) * inv_ok,
                                    __fdiv_rn(o[i + 3], Sd) * inv_ok);
            }
        }
    } else {
        // a completion never came: record it, give the tensor core one more
        // bounded wait, then release TMEM without touching the outputs
        if (tid == 0) atomicOr(P.status, KQ8_STATUS_TIMEOUT);
        if (fail_bar) mbar_wait_bounded(fail_bar, fail_par);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tbase, PF_TMEM_COLS);
    }
}

template <int G>
int launch_prefill_g(const PrefillParams& p, int nkv, cudaStream_t s) {
    constexpr int TQ = PF_ROWS / G;
    if (cudaFuncSetAttribute(kq8_prefill_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PF_SMEM) != cudaSuccess)
        return KQ8_ERR_CUDA;
    const dim3 grid((unsigned)((p.max_q_len + TQ - 1) / TQ), (unsigned)nkv, (unsigned)p.B);
    kq8_prefill_kernel<G><<<grid, PF_THREADS, PF_SMEM, s>>>(p);
    return cudaPeekAtLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

int launch_prefill(const PrefillParams& p, int G, int nkv, cudaStream_t s) {
    switch (G) {
        case 1: return launch_prefill_g<1>(p, nkv, s);
        case 2: return launch_prefill_g<2>(p, nkv, s);
        case 3: return launch_prefill_g<3>(p, nkv, s);
        case 4: return launch_prefill_g<4>(p, nkv, s);
        case 5: return launch_prefill_g<5>(p, nkv, s);
        case 6: return launch_prefill_g<6>(p, nkv, s);
        case 7: return launch_prefill_g<7>(p, nkv, s);
        case 8: return launch_prefill_g<8>(p, nkv, s);
        default: return KQ8_ERR_UNSUPPORTED;
    }
}

}  // namespace kq8

using namespace kq8;

extern "C" {

size_t kq8_prefill_workspace_bytes(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len,
                                   int32_t max_q_len) {
    (void)B, (void)nq, (void)nkv, (void)max_seq_len, (void)max_q_len;
    return PF_STATUS_BYTES;
}

int kq8_prefill_attn(float* out, const float* q, int32_t total_q, const kq8_cache_t* cache,
                     const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len, int32_t B,
                     int32_t nq, float scale, void* workspace, size_t workspace_bytes,
                     kq8_stream_t stream) {
    int rc = check_cache_args(cache);
    if (rc) return rc;
    if (B < 0 || nq < 1 || total_q < 0 || max_seq_len < 0 || max_q_len < 0 || max_pages < 0)
        return KQ8_ERR_INVALID_ARG;
    const int nkv = cache->num_kv_heads;
    if (nq % nkv != 0 || nq / nkv > MAX_G) return KQ8_ERR_UNSUPPORTED;
    if ((int64_t)max_seq_len > (int64_t)max_pages * cache->kv_bs) return KQ8_ERR_INVALID_ARG;
    if (max_q_len > max_seq_len) return KQ8_ERR_INVALID_ARG;
    if (max_seq_len >= (1 << 29) || B > 65535) return KQ8_ERR_UNSUPPORTED;
    if (!workspace || (uintptr_t)workspace % 256 != 0 ||
        workspace_bytes < kq8_prefill_workspace_bytes(B, nq, nkv, max_seq_len, max_q_len))
        return KQ8_ERR_WORKSPACE;
    if (B == 0 || max_q_len == 0) return KQ8_OK;
    if (!out || !q || !seq_lens || !q_offsets || !page_table) return KQ8_ERR_INVALID_ARG;
    if ((uintptr_t)out % 16 != 0 || (uintptr_t)q % 16 != 0) return KQ8_ERR_INVALID_ARG;
    PrefillParams p;
    p.out = out;
    p.q = q;
    p.cache = *cache;
    p.page_table = page_table;
    p.max_pages = max_pages;
    p.seq_lens = seq_lens;
    p.q_off = q_offsets;
    p.total_q = total_q;
    p.max_seq_len = max_seq_len;
    p.max_q_len = max_q_len;
    p.B = B;
    p.nq = nq;
    p.scale = scale;
    p.status = static_cast<uint32_t*>(workspace);
    return launch_prefill(p, nq / nkv, nkv, (cudaStream_t)stream);
}

}  // extern "C"
