// kq8_prefill.cu -- batched causal prefill attention over the q8 cache on the
// 5th-generation tensor cores, warp-specialised.
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
// GB300 mapping.  A CTA (one per SM: all 512 TMEM columns) takes two query
// tiles A and B of 128 (token, query head) rows each -- 128/G consecutive new
// tokens x the G query heads of one KV head -- and walks the KV history in
// 64-token steps, each filled from two 32-token cache sub-tiles.  Warps have
// fixed roles and meet only on mbarriers:
//   warp 11     copies raw sub-tiles (codes + scales as stored) into a
//               three-stage ring with bulk-async copies;
//   warps 8-9   widen them exactly to tensor-core operands: K to fp16, V to
//               bf16 (every int8 is exact in both), double-buffered by step,
//               K of a step before its V;
//   warp 10     one thread issues every MMA: S_t = Q_t K^T as four per-block
//               MMA pairs (N = 64) into four TMEM accumulators (each holds the
//               exact integer block dot), and O_t += W_hi V + W_lo V (N = 128);
//   warps 0-7   softmax of tile A (0-3) and B (4-7), one thread per row (TMEM
//               lane): the scores from the block dots in the method's order,
//               the online softmax with a lazy rescale of the TMEM O row, and
//               the weights w = p * vscale / 127 as bf16 hi + lo (2^-16).
// The two tiles take the block-dot accumulators in turn, and each PV is
// followed by the other tile's next S: the tiles run half a step apart, one
// scoring while the other computes.  An M = 128, K = 16 MMA costs the same
// issue time for N = 32, 64 or 128, so the 64-token step halves the S
// instructions per token against 32-token steps.  K and V buffers are
// released separately (K once both tiles have read the step's scores, V after
// the second PV), so the widening of the next step's K never waits for a PV.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kq8_internal.h"
#include "kq8_tc.cuh"

namespace kq8 {
namespace {

constexpr int PF_ROWS = 128;            // rows per query tile (MMA M, TMEM lanes)
constexpr int PF_NT = TILE;             // tokens per cache sub-tile (copy and widening unit)
constexpr int PF_STEP = 2 * TILE;       // tokens per pipeline step (S and PV unit)
constexpr int PF_RAW = 3;               // raw sub-tile ring stages
constexpr int PF_CV_WARP = 8;           // warps 8-9 widen K/V
constexpr int PF_CV_WARPS = 2;
constexpr int PF_MMA_WARP = 10;
constexpr int PF_LOAD_WARP = 11;
constexpr int PF_THREADS = 12 * 32;
// TMEM columns: O of tile t at 128 t; the block dots of the tile being scored
// (the two tiles take it in turn) at 256 + 64 b for block b.
constexpr uint32_t PF_TMEM_COLS = 512;
constexpr uint32_t PF_COL_D = 256;

// Shared memory map (bytes).  Tensor-core operands are K-major without
// swizzle: 8-row x 16-byte core matrices, 128 B each.  A 64-token step's K and
// V buffers are filled one 32-token cache sub-tile (one half) at a time.
constexpr uint32_t SM_Q = 0;            // 2 tiles x fp16 Q codes, 128 rows x 128 dims (32 KB)
constexpr uint32_t SM_K = 65536;        // 2 buffers x fp16 K codes, 64 tokens x 128 dims (16 KB)
constexpr uint32_t SM_V = 98304;        // 2 buffers x bf16 V codes, 128 dims x 64 tokens (16 KB)
constexpr uint32_t SM_W = 131072;       // 2 tiles x bf16 weights hi, lo: 128 x 64 (32 KB)
constexpr uint32_t SM_RAW = 196608;     // 3 stages x raw sub-tile (8448 B)
constexpr uint32_t SM_SC = 221952;      // 2 buffers x (64 score multipliers, 64 value steps)
constexpr uint32_t SM_OK = 222976;      // int: page valid per (buffer, half), then per raw stage
constexpr uint32_t SM_BAR = 223008;     // mbarriers (below)
constexpr uint32_t SM_TMEM = 223200;    // TMEM base address written by the allocator
constexpr uint32_t SM_ABORT = 223204;   // set when a bounded wait ran out
constexpr uint32_t PF_SMEM = 223232;

// mbarriers: index, arrivals per phase
constexpr int B_RAW_FULL = 0;   // [3] producer's expect-tx arrive + the copied bytes
constexpr int B_RAW_EMPTY = 3;  // [3] 2 widening warps
constexpr int B_K_FULL = 6;     // [2] 2 widening warps x the step's 2 sub-tiles (K, scales)
constexpr int B_V_FULL = 8;     // [2] the same for V and its scales
constexpr int B_K_EMPTY = 10;   // [2] commit once both tiles have read S of the step
constexpr int B_V_EMPTY = 12;   // [2] commit after the second tile's PV of the step
constexpr int B_S_FULL = 14;    // [tile] commit after S_t
constexpr int B_D_FREE = 16;    // [tile] 4 softmax warps have read S_t (and its multipliers)
constexpr int B_W_FULL = 18;    // [tile] 4 softmax warps wrote W_t (and rescaled O_t)
constexpr int B_PV_DONE = 20;   // [tile] commit after PV_t
constexpr int B_FINAL = 22;     // last commit of the MMA thread, waited on before TMEM is freed
constexpr int B_COUNT = 23;

constexpr size_t PF_STATUS_BYTES = 256;  // workspace: the status word (256-byte slot)

constexpr float PF_LOG2E = 1.4426950408889634f;
constexpr float PF_RESCALE_SLACK = 8.0f;  // log2 units: rescale O when the max grows > 2^8

__device__ __forceinline__ uint32_t sm_k(int p) { return SM_K + 16384u * p; }
__device__ __forceinline__ uint32_t sm_v(int p) { return SM_V + 16384u * p; }
__device__ __forceinline__ uint32_t sm_whi(int t) { return SM_W + 32768u * t; }
__device__ __forceinline__ uint32_t sm_raw(int s) { return SM_RAW + (uint32_t)STAGE_BYTES * s; }
__device__ __forceinline__ uint32_t sm_km(int p) { return SM_SC + 512u * p; }
__device__ __forceinline__ uint32_t sm_vs(int p) { return SM_SC + 512u * p + 256u; }

// Byte offset of the 16-byte chunk holding elements 8*kc .. 8*kc+7 of row r in
// a K-major operand of R rows: core matrices adjacent along K are R*16 B apart
// (leading byte offset), along the rows 128 B apart (stride byte offset).
__device__ __forceinline__ uint32_t cm_off(int r, int kc, int R) {
    return (uint32_t)(kc * R * 16 + (r >> 3) * 128 + (r & 7) * 16);
}

__device__ __forceinline__ float pf_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void pf_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
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

__device__ __forceinline__ uint32_t bf2_bits(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t h2_bits(int lo, int hi) {
    __half2 v = __halves2half2(__int2half_rn(lo), __int2half_rn(hi));
    return *reinterpret_cast<uint32_t*>(&v);
}

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
    int32_t withhold_sub;  // test hook: this raw sub-tile is never copied (-1: none)
};

template <int G>
__global__ void __launch_bounds__(PF_THREADS, 1) kq8_prefill_kernel(const PrefillParams P) {
    constexpr int TQ = PF_ROWS / G;  // new tokens per query tile
    extern __shared__ __align__(1024) uint8_t sm[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTAs start in linear order (x fastest): the linear index is read with the
    // (KV head, sequence) fastest and the query tile slowest, longest first, so
    // that every head's and sequence's longest tiles start in the first wave
    const unsigned lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    const unsigned hbn = gridDim.y * gridDim.z;
    const int h = (int)((lin % hbn) % gridDim.y), b = (int)((lin % hbn) / gridDim.y);
    const int nkv = P.cache.num_kv_heads, kv_bs = P.cache.kv_bs;
    const int qt = (int)gridDim.x - 1 - (int)(lin / hbn);

    const int n = P.seq_lens[b];
    const int q0 = P.q_off[b];
    const int nb = P.q_off[b + 1] - q0;
    if (n < 0 || n > P.max_seq_len || nb < 0 || nb > n || nb > P.max_q_len || q0 < 0 ||
        (int64_t)q0 + nb > P.total_q) {
        if (tid == 0 && qt == (int)gridDim.x - 1 && h == 0) atomicOr(P.status, KQ8_STATUS_BAD_SEQLEN);
        return;
    }
    const int i0 = qt * 2 * TQ;  // first new token of tile A; tile B follows
    if (i0 >= nb) return;
    const int ntok = min(2 * TQ, nb - i0);
    const int nsub = (n - nb + i0 + ntok - 1) / PF_NT + 1;  // cache sub-tiles the CTA reads
    const int nsteps = (nsub + 1) / 2;                       // 64-token steps
    const int pos_first = n - nb + i0;  // position of the CTA's first new token

    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + SM_BAR);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SM_TMEM);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + SM_ABORT);
    // page-valid flags: [0..3] per (buffer, half), [4..6] per raw stage
    volatile int* okv = reinterpret_cast<volatile int*>(sm + SM_OK);
    if (warp == 0) {
        __syncwarp();
        tc::tmem_alloc(tslot, PF_TMEM_COLS);
    }
    if (tid == 0) {
        for (int i = 0; i < B_COUNT; i++) {
            uint32_t cnt = 1;
            if (i >= B_D_FREE && i < B_PV_DONE) cnt = 4;
            if (i >= B_RAW_EMPTY && i < B_K_FULL) cnt = PF_CV_WARPS;
            if (i >= B_K_FULL && i < B_K_EMPTY) cnt = 2 * PF_CV_WARPS;
            mbar_init(bars + i, cnt);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // A wait that gives up after the bounded spin, records it and makes every
    // later wait of the CTA give up at once.
    auto wait = [&](int i, uint32_t parity) -> bool {
        if (*abort_flag) return false;
        if (mbar_wait_bounded(bars + i, parity)) return true;
        *abort_flag = 1;
        atomicOr(P.status, KQ8_STATUS_TIMEOUT);
        return false;
    };

    // ---- softmax rows: tile A = warps 0-3, tile B = warps 4-7; one row each
    const int qtile = (warp >> 2) & 1;
    const int row = (warp & 3) * 32 + lane;
    const int tq = qtile * TQ + row / G, g = row % G;
    const bool valid = warp < 8 && row < TQ * G && tq < ntok;
    const int pos = valid ? n - nb + i0 + tq : -1;  // this row sees tokens 0 .. pos
    float qsc[NB] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (warp < 8) {
        // quantise this row once (article 9-2 §2 segment 1) -> fp16 codes
        uint8_t* Qs = sm + SM_Q + 32768u * qtile;
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
                *reinterpret_cast<uint4*>(Qs + cm_off(row, blk * 4 + c, PF_ROWS)) =
                    make_uint4(h2_bits(code(a.x), code(a.y)), h2_bits(code(a.z), code(a.w)),
                               h2_bits(code(e.x), code(e.y)), h2_bits(code(e.z), code(e.w)));
            }
        }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tslot;

    if (warp == PF_LOAD_WARP) {
        // ---- producer: raw sub-tile t into ring stage t % 3 (page ids one per
        // lane for a 32-sub-tile window, fetched a window ahead).  A step's
        // second half past the last sub-tile is an empty sub-tile (no copy).
        auto load_window = [&](int w) -> int32_t {
            const int t = 32 * w + lane;
            if (t >= nsub) return -1;
            const int32_t pg = P.page_table[(size_t)b * P.max_pages + (t * PF_NT) / kv_bs];
            return (pg >= 0 && pg < P.cache.num_pages) ? pg : -2;
        };
        int32_t pw_cur = load_window(0), pw_nxt = load_window(1);
        int armed[PF_RAW] = {-1, -1, -1};  // last sub-tile whose copies went into each stage
        uint64_t pol;
        asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
        for (int t = 0; t < 2 * nsteps; t++) {
            const int s = t % PF_RAW;
            if (t >= PF_RAW &&
                !__all_sync(0xffffffffu, wait(B_RAW_EMPTY + s, ((t - PF_RAW) / PF_RAW) & 1)))
                break;
            if ((t & 31) == 0 && t > 0) {
                pw_cur = pw_nxt;
                pw_nxt = load_window((t >> 5) + 1);
            }
            const int32_t pg = __shfl_sync(0xffffffffu, pw_cur, t & 31);  // -1: none, -2: bad
            if (lane == 0 && t != P.withhold_sub) {
                armed[s] = t;
                uint64_t* bar = bars + B_RAW_FULL + s;
                uint8_t* st = sm + sm_raw(s);
                okv[4 + s] = pg >= 0;
                if (pg < 0) {
                    if (pg == -2) atomicOr(P.status, KQ8_STATUS_BAD_PAGE);
                    mbar_arrive_expect_tx(bar, 0);  // completes the phase with no data
                } else {
                    const int sub = ((t * PF_NT) % kv_bs) / PF_NT;
                    const size_t kvo = kv_sub_off(pg, h, nkv, kv_bs, sub);
                    const size_t so = scale_sub_off(pg, h, nkv, kv_bs, sub);
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    bulk_g2s(st, P.cache.k + kvo, SUB_K_BYTES, bar, pol);
                    bulk_g2s(st + SUB_K_BYTES, P.cache.v + kvo, SUB_V_BYTES, bar, pol);
                    bulk_g2s(st + SUB_K_BYTES + SUB_V_BYTES, P.cache.kscale + so, SUB_S_BYTES,
                             bar, pol);
                    bulk_g2s(st + SUB_K_BYTES + SUB_V_BYTES + SUB_S_BYTES, P.cache.vscale + so,
                             SUB_S_BYTES, bar, pol);
                }
            }
        }
        // an aborted CTA lets the copies it started land before shared memory
        // is given up (each stage's last armed phase, bounded)
        if (*abort_flag && lane == 0) {
            for (int s = 0; s < PF_RAW; s++)
                if (armed[s] >= 0)
                    mbar_wait_bounded(bars + B_RAW_FULL + s, (armed[s] / PF_RAW) & 1);
        }
    } else if (warp >= PF_CV_WARP && warp < PF_CV_WARP + PF_CV_WARPS) {
        // ---- widening, one step at a time: K of both raw sub-tiles (halves)
        // of step j into buffer j & 1, then V of both.  K and V are released
        // separately -- K once both tiles have scored the step, V after the
        // second tile's PV -- and the K of a step never waits behind the V of
        // an earlier one, so scoring runs a step ahead of PV.
        const float kmul = inv127() * P.scale * PF_LOG2E;  // score multiplier per kscale
        for (int j = 0; j < nsteps; j++) {
            const int p = j & 1;
            const uint32_t reuse = ((j - 2) >> 1) & 1;  // phase of the step that used buffer p
            bool ok = j < 2 || __all_sync(0xffffffffu, wait(B_K_EMPTY + p, reuse));
#pragma unroll 1
            for (int half = 0; ok && half < 2; half++) {
                const int t = 2 * j + half, s = t % PF_RAW;
                if (!(ok = __all_sync(0xffffffffu, wait(B_RAW_FULL + s, (t / PF_RAW) & 1)))) break;
                const uint8_t* st = sm + sm_raw(s);
                const bool tok = okv[4 + s] != 0;
                // K: cw = 32-element block (warp w takes w and w + 2), lane =
                // token row (stored at position kpos)
                uint8_t* Ks = sm + sm_k(p);
#pragma unroll 1
                for (int cw = warp - PF_CV_WARP; cw < 4; cw += PF_CV_WARPS) {
                    const uint4* kr =
                        reinterpret_cast<const uint4*>(st + cw * 1024 + kpos(lane) * 32);
                    const uint4 ka = kr[0], kb = kr[1];
                    const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        *reinterpret_cast<uint4*>(
                            Ks + cm_off(32 * half + lane, cw * 4 + c, PF_STEP)) =
                            make_uint4(i8x2_to_h2(kw[2 * c], 0), i8x2_to_h2(kw[2 * c], 1),
                                       i8x2_to_h2(kw[2 * c + 1], 0), i8x2_to_h2(kw[2 * c + 1], 1));
                }
                // score multipliers: 0 for a missing page, an empty half and past
                // the sequence end (masked tokens must carry finite values)
                if (warp == PF_CV_WARP) {
                    const float* rs =
                        reinterpret_cast<const float*>(st + SUB_K_BYTES + SUB_V_BYTES);
                    const bool live = tok && t * PF_NT + lane < n;
                    reinterpret_cast<float*>(sm + sm_km(p))[32 * half + lane] =
                        live ? __fmul_rn(rs[lane], kmul) : 0.0f;
                    if (lane == 0) okv[2 * p + half] = tok;
                }
                tc::fence_smem_to_async();
                __syncwarp();
                if (lane == 0) pf_arrive(bars + B_K_FULL + p);
            }
            if (ok && j >= 2) ok = __all_sync(0xffffffffu, wait(B_V_EMPTY + p, reuse));
#pragma unroll 1
            for (int half = 0; ok && half < 2; half++) {
                const int t = 2 * j + half, s = t % PF_RAW;
                const uint8_t* st = sm + sm_raw(s);
                const bool tok = okv[4 + s] != 0;
                // V transposed (dims as rows, tokens along K): tokens 8*cw .. +7
                // of this half, dims 4*lane .. +3; the dim order rotates per lane
                // pair so that the eight lanes of each 16-byte store phase hit
                // eight bank groups
                uint8_t* Vs = sm + sm_v(p);
#pragma unroll 1
                for (int cw = warp - PF_CV_WARP; cw < 4; cw += PF_CV_WARPS) {
                    const uint32_t* vr =
                        reinterpret_cast<const uint32_t*>(st + SUB_K_BYTES + cw * 8 * HD) + lane;
                    uint32_t u[8];
#pragma unroll
                    for (int tt = 0; tt < 8; tt++) u[tt] = vr[tt * (HD / 4)] ^ 0x80808080u;
                    const float2 bias = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
#pragma unroll
                    for (int e = 0; e < 4; e++) {
                        const int ee = (e + (lane >> 1)) & 3;
                        const uint32_t sel = 0x7540u | (uint32_t)ee;
                        float2 f[4];
#pragma unroll
                        for (int q2 = 0; q2 < 4; q2++)
                            f[q2] = __fadd2_rn(
                                make_float2(
                                    __uint_as_float(__byte_perm(u[2 * q2], 0x4B000000u, sel)),
                                    __uint_as_float(__byte_perm(u[2 * q2 + 1], 0x4B000000u, sel))),
                                bias);
                        *reinterpret_cast<uint4*>(
                            Vs + cm_off(4 * lane + ee, 4 * half + cw, PF_ROWS)) =
                            make_uint4(bf2_bits(f[0].x, f[0].y), bf2_bits(f[1].x, f[1].y),
                                       bf2_bits(f[2].x, f[2].y), bf2_bits(f[3].x, f[3].y));
                    }
                }
                if (warp == PF_CV_WARP + PF_CV_WARPS - 1) {
                    const float* rs =
                        reinterpret_cast<const float*>(st + SUB_K_BYTES + SUB_V_BYTES) + 32;
                    const bool live = tok && t * PF_NT + lane < n;
                    reinterpret_cast<float*>(sm + sm_vs(p))[32 * half + lane] =
                        live ? __fmul_rn(rs[lane], inv127()) : 0.0f;
                }
                tc::fence_smem_to_async();
                __syncwarp();
                if (lane == 0) {
                    pf_arrive(bars + B_RAW_EMPTY + s);
                    pf_arrive(bars + B_V_FULL + p);
                }
            }
            if (!ok) break;
        }
    } else if (warp == PF_MMA_WARP) {
        // ---- one thread issues every MMA; descriptors are built once and an
        // MMA at K chunk kc adds kc * leading-byte-offset / 16 to the address
        if (lane == 0) {
            const uint64_t d_q = tc::sdesc(smem_u32(sm + SM_Q), PF_ROWS * 16, 128);
            const uint64_t d_k = tc::sdesc(smem_u32(sm + SM_K), PF_STEP * 16, 128);
            const uint64_t d_v = tc::sdesc(smem_u32(sm + SM_V), PF_ROWS * 16, 128);
            const uint64_t d_w = tc::sdesc(smem_u32(sm + SM_W), PF_ROWS * 16, 128);
            auto issue_s = [&](int t, int p) {  // D_blk = Q_blk K_blk^T, blk = 0..3, 64 tokens
                const uint64_t dq = d_q + (uint64_t)t * (32768u >> 4);
                const uint64_t dk = d_k + (uint64_t)p * (16384u >> 4);
                constexpr uint32_t ID = tc::IDesc<128, PF_STEP, false>::value;
#pragma unroll
                for (int blk = 0; blk < NB; blk++)
#pragma unroll
                    for (int kk = 0; kk < 2; kk++) {
                        const int kc = blk * 4 + kk * 2;
                        tc::mma_f16(tbase + PF_COL_D + 64 * blk, dq + (uint64_t)(kc * PF_ROWS),
                                    dk + (uint64_t)(kc * PF_STEP), ID, kk > 0);
                    }
                tc::mma_commit(bars + B_S_FULL + t);
            };
            auto issue_pv = [&](int t, int p, bool accumulate) {  // O_t (+)= W_hi V + W_lo V
                const uint64_t dv = d_v + (uint64_t)p * (16384u >> 4);
                const uint64_t dh = d_w + (uint64_t)(sm_whi(t) - SM_W) / 16;
                const uint64_t dl = dh + (16384u >> 4);
                constexpr uint32_t ID = tc::IDesc<128, HD, true>::value;
#pragma unroll
                for (int kk = 0; kk < PF_STEP / 16; kk++) {
                    const uint64_t off = (uint64_t)(kk * 2 * PF_ROWS);
                    tc::mma_f16(tbase + 128 * t, dh + off, dv + off, ID, accumulate || kk > 0);
                    tc::mma_f16(tbase + 128 * t, dl + off, dv + off, ID, true);
                }
                tc::mma_commit(bars + B_PV_DONE + t);
            };
            // The tiles take the block dots in turn: S_A(j), (A has read them)
            // S_B(j), (B has read them) S_A(j+1), ...  Each PV is followed by
            // the other tile's next S, so a tile's next S waits for the other
            // tile, not for its own PV; the tiles settle half a step apart.
            // K buffer p is released once B has read S(j) and its multipliers,
            // V buffer p after PV_B(j); a release (a commit) is issued only
            // when a later step reuses the buffer (every commit must be waited
            // on before the CTA exits).
            bool ok = wait(B_K_FULL, 0);
            if (ok) {
                tc::fence_after_sync();
                issue_s(0, 0);
                ok = wait(B_D_FREE + 0, 0);
            }
            if (ok) {
                tc::fence_after_sync();
                issue_s(1, 0);
                ok = wait(B_D_FREE + 1, 0);
            }
            if (ok) {
                if (2 < nsteps) tc::mma_commit(bars + B_K_EMPTY + 0);
                if (nsteps > 1 && (ok = wait(B_K_FULL + 1, 0))) {
                    tc::fence_after_sync();
                    issue_s(0, 1);
                }
            }
            for (int j = 0; ok && j < nsteps; j++) {
                const int p = j & 1;
                if (!(ok = wait(B_W_FULL + 0, j & 1) && wait(B_V_FULL + p, (j >> 1) & 1))) break;
                tc::fence_after_sync();
                issue_pv(0, p, j > 0);
                if (j + 1 < nsteps) {
                    if (!(ok = wait(B_D_FREE + 0, (j + 1) & 1))) break;
                    tc::fence_after_sync();
                    issue_s(1, p ^ 1);
                }
                if (!(ok = wait(B_W_FULL + 1, j & 1))) break;
                tc::fence_after_sync();
                issue_pv(1, p, j > 0);
                if (j + 2 < nsteps) tc::mma_commit(bars + B_V_EMPTY + p);
                if (j + 1 < nsteps) {
                    if (!(ok = wait(B_D_FREE + 1, (j + 1) & 1))) break;
                    if (j + 3 < nsteps) tc::mma_commit(bars + B_K_EMPTY + (p ^ 1));
                    if (j + 2 < nsteps) {
                        if (!(ok = wait(B_K_FULL + p, ((j + 2) >> 1) & 1))) break;
                        tc::fence_after_sync();
                        issue_s(0, p);
                    }
                }
            }
            // completes once every MMA issued above has (bounded wait)
            tc::mma_commit(bars + B_FINAL);
            mbar_wait_bounded(bars + B_FINAL, 0);
        }
    } else if (warp < 8) {
        // ---- softmax of this row over every 64-token step
        const uint32_t t_row = (uint32_t)((warp & 3) * 32) << 16;  // this warp's TMEM lanes
        const uint32_t tO = tbase + 128 * qtile + t_row, tD = tbase + PF_COL_D + t_row;
        float M2 = M_INIT, Mhi = M_INIT + PF_RESCALE_SLACK;
        float2 S2 = make_float2(0.0f, 0.0f);  // running sum, even and odd tokens
        bool ok = true;
        for (int j = 0; j < nsteps; j++) {
            const int p = j & 1;
            ok = __all_sync(0xffffffffu, wait(B_S_FULL + qtile, j & 1));
            // the widening warps' scales and page flags of buffer p (long complete)
            if (ok) ok = __all_sync(0xffffffffu, wait(B_K_FULL + p, (j >> 1) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            // scores against the step's 64 tokens (article 9-2 §2 seg. 2): s =
            // sum_b dot_b * qsc_b, times the token's kscale / 127 * scale, base 2
            float2 x[PF_STEP / 2];
#pragma unroll
            for (int blk = 0; blk < NB; blk++) {
                const float2 cb = make_float2(qsc[blk], qsc[blk]);
#pragma unroll
                for (int q16 = 0; q16 < PF_STEP / 16; q16++) {
                    float d[16];
                    tc::tmem_ld16(tD + 64 * blk + 16 * q16, d);
#pragma unroll
                    for (int i = 0; i < 8; i++) {
                        const float2 dv = make_float2(d[2 * i], d[2 * i + 1]);
                        x[8 * q16 + i] =
                            blk == 0 ? __fmul2_rn(dv, cb) : __ffma2_rn(dv, cb, x[8 * q16 + i]);
                    }
                }
            }
            const float2* km2 = reinterpret_cast<const float2*>(sm + sm_km(p));
#pragma unroll
            for (int i = 0; i < PF_STEP / 2; i++) x[i] = __fmul2_rn(x[i], km2[i]);
            const bool ok0 = okv[2 * p] != 0, ok1 = okv[2 * p + 1] != 0;
            // the block dots may be overwritten, and (once both tiles are here)
            // K buffer p with its multipliers and page flags
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) pf_arrive(bars + B_D_FREE + qtile);
            const int t0 = j * PF_STEP;
            // every row of the CTA sees every token of this step: no masking
            const bool full = ok0 && ok1 && t0 + PF_STEP - 1 <= pos_first;
            if (!full) {
                const int nvis = max(0, min(PF_STEP, pos - t0 + 1));
#pragma unroll
                for (int i = 0; i < PF_STEP / 2; i++) {
                    const bool hok = (2 * i < PF_NT) ? ok0 : ok1;
                    if (!hok || 2 * i >= nvis) x[i].x = -INFINITY;
                    if (!hok || 2 * i + 1 >= nvis) x[i].y = -INFINITY;
                }
            }
            float mt = -INFINITY;
#pragma unroll
            for (int i = 0; i < PF_STEP / 2; i++) mt = fmaxf(mt, fmaxf(x[i].x, x[i].y));
            // lazy rescale of S and of this row of O (online-softmax max)
            const bool need = mt > Mhi;
            float cf = 1.0f;
            if (need) {
                cf = pf_ex2(M2 - mt);
                S2 = __fmul2_rn(S2, make_float2(cf, cf));
                M2 = mt;
                Mhi = mt + PF_RESCALE_SLACK;
            }
            // PV_t of the previous step has read W_t and written O_t
            if (j > 0 && !(ok = __all_sync(0xffffffffu, wait(B_PV_DONE + qtile, (j - 1) & 1))))
                break;
            if (j > 0 && __any_sync(0xffffffffu, need)) {
                tc::fence_after_sync();
#pragma unroll 1
                for (int c = 0; c < HD / 32; c++) {
                    float o[32];
                    tc::tmem_ld32(tO + 32 * c, o);
#pragma unroll
                    for (int i = 0; i < 32; i++) o[i] = __fmul_rn(o[i], cf);
                    tc::tmem_st32(tO + 32 * c, o);
                }
            }
            if (!(ok = __all_sync(0xffffffffu, wait(B_V_FULL + p, (j >> 1) & 1)))) break;
            // weights w = p * vscale / 127 = hi + lo: hi is w cut to bf16 (its
            // top 16 bits), lo = w - hi (exact) rounded to bf16
            uint8_t* Wh = sm + sm_whi(qtile);
            uint8_t* Wl = Wh + 16384;
            const float2* vs2 = reinterpret_cast<const float2*>(sm + sm_vs(p));
            const float2 negm = make_float2(-M2, -M2);
#pragma unroll
            for (int c = 0; c < PF_STEP / 8; c++) {
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
                *reinterpret_cast<uint4*>(Wh + cm_off(row, c, PF_ROWS)) =
                    make_uint4(hi[0], hi[1], hi[2], hi[3]);
                *reinterpret_cast<uint4*>(Wl + cm_off(row, c, PF_ROWS)) =
                    make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            tc::fence_smem_to_async();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) pf_arrive(bars + B_W_FULL + qtile);
        }
        // ---- output: acc / S after the last PV_t
        if (ok) ok = __all_sync(0xffffffffu, wait(B_PV_DONE + qtile, (nsteps - 1) & 1));
        if (ok) {
            tc::fence_after_sync();
            const float S = S2.x + S2.y;
            const float inv_ok = S > 0.0f ? 1.0f : 0.0f;  // no visible token: 0
            const float Sd = S > 0.0f ? S : 1.0f;
            float* dst = P.out + ((size_t)(q0 + i0 + tq) * P.nq + (size_t)h * G + g) * HD;
#pragma unroll 1
            for (int c = 0; c < HD / 32; c++) {
                float o[32];
                tc::tmem_ld32(tO + 32 * c, o);
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        *reinterpret_cast<float4*>(dst + 32 * c + i) =
                            make_float4(__fdiv_rn(o[i], Sd) * inv_ok,
                                        __fdiv_rn(o[i + 1], Sd) * inv_ok,
                                        __fdiv_rn(o[i + 2], Sd) * inv_ok,
                                        __fdiv_rn(o[i + 3], Sd) * inv_ok);
                }
            }
        }
    }
    // ---- teardown: every role has left its loop and the MMA thread has seen
    // its last commit complete (bounded) before TMEM goes
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
    constexpr int TQ2 = 2 * (PF_ROWS / G);  // new tokens per CTA (two query tiles)
    if (cudaFuncSetAttribute(kq8_prefill_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PF_SMEM) != cudaSuccess)
        return KQ8_ERR_CUDA;
    const dim3 grid((unsigned)((p.max_q_len + TQ2 - 1) / TQ2), (unsigned)nkv, (unsigned)p.B);
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

}  // extern "C"

namespace {

int prefill_impl(float* out, const float* q, int32_t total_q, const kq8_cache_t* cache,
                 const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                 const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len, int32_t B,
                 int32_t nq, float scale, void* workspace, size_t workspace_bytes,
                 kq8_stream_t stream, int32_t withhold_sub) {
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
    p.withhold_sub = withhold_sub;
    return launch_prefill(p, nq / nkv, nkv, (cudaStream_t)stream);
}

}  // namespace

extern "C" {

int kq8_prefill_attn(float* out, const float* q, int32_t total_q, const kq8_cache_t* cache,
                     const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len, int32_t B,
                     int32_t nq, float scale, void* workspace, size_t workspace_bytes,
                     kq8_stream_t stream) {
    return prefill_impl(out, q, total_q, cache, page_table, max_pages, seq_lens, q_offsets,
                        max_seq_len, max_q_len, B, nq, scale, workspace, workspace_bytes, stream,
                        -1);
}

int kq8_debug_prefill_withhold(float* out, const float* q, int32_t total_q,
                               const kq8_cache_t* cache, const int32_t* page_table,
                               int32_t max_pages, const int32_t* seq_lens,
                               const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len,
                               int32_t B, int32_t nq, float scale, void* workspace,
                               size_t workspace_bytes, int32_t withhold_sub,
                               kq8_stream_t stream) {
    if (withhold_sub < 0) return KQ8_ERR_INVALID_ARG;
    return prefill_impl(out, q, total_q, cache, page_table, max_pages, seq_lens, q_offsets,
                        max_seq_len, max_q_len, B, nq, scale, workspace, workspace_bytes, stream,
                        withhold_sub);
}

}  // extern "C"
