// kq8_misc.cu -- the write path (article 9-3 §2, kv_quantize_per_head) and the
// test-only kernels that expose the hot path's integer building blocks.
#include "kq8_common.cuh"
#include "kq8_internal.h"

namespace kq8 {

// roundf(x / d) for the elements of a row whose step is d, |x / d| < 128, with
// r = RN(1 / d).  r and the product q = RN(x * r) each round once (relative
// 2^-24), so |q - x / d| <= 128 * 2^-23 and |fl(x / d) - x / d| <= 2^-18:
// q is within 2^-15.5 of the IEEE quotient fl(x / d).  Unless q lies within
// 2^-14 of a half-integer both therefore round to the same integer, and the
// nearest integer to q (no tie possible) is roundf(fl(x / d)).  The rare
// near-half case (about 1 in 8000 elements), and a non-finite q (d subnormal
// or 0), take the IEEE quotient itself, so the result always equals the
// method's roundf(x / d) bit for bit.
// The nearest integer comes from adding 1.5 * 2^23 + off (exact for |q| < 2^22):
// the sum's low byte is then (n + off) mod 256, the code byte itself.  On the
// fast path |q| < 127.5 (and < 7.5 for q4), so no clamp is needed there.
// Returns the lane's four code bytes (element i in byte i); r = RN(1 / d) (the
// caller computes it once per row), lo / hi clamp the slow path, off is 0 (q8,
// two's complement) or 8 (q4, offset binary).
__device__ __forceinline__ uint32_t quantize4(const float4 x, float d, float r, float lo, float hi,
                                              int off) {
    const float magic = 12582912.0f + (float)off;  // 1.5 * 2^23 + off
    const float q0 = __fmul_rn(x.x, r), q1 = __fmul_rn(x.y, r);
    const float q2 = __fmul_rn(x.z, r), q3 = __fmul_rn(x.w, r);
    const float t0 = __fadd_rn(q0, magic), t1 = __fadd_rn(q1, magic);
    const float t2 = __fadd_rn(q2, magic), t3 = __fadd_rn(q3, magic);
    const float far = 0.5f - 0x1p-14f;  // NaN / inf compare false
    const bool ok = fabsf(q0 - (t0 - magic)) < far && fabsf(q1 - (t1 - magic)) < far &&
                    fabsf(q2 - (t2 - magic)) < far && fabsf(q3 - (t3 - magic)) < far;
    if (ok)
        return __byte_perm(__byte_perm(__float_as_uint(t0), __float_as_uint(t1), 0x0040),
                           __byte_perm(__float_as_uint(t2), __float_as_uint(t3), 0x0040), 0x5410);
    auto slow = [&](float v) -> uint32_t {
        const float n = fminf(fmaxf(roundf(__fdiv_rn(v, d)), lo), hi);
        return (uint32_t)((int)n + off) & 0xffu;
    };
    return slow(x.x) | (slow(x.y) << 8) | (slow(x.z) << 16) | (slow(x.w) << 24);
}

__device__ __forceinline__ float absmax4(const float4 x) {
    return fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
}

// The q8 write path: one (token, KV head) row per group of LPR lanes, 32 / LPR
// rows per warp (consecutive items: the heads of a token, whose fp32 rows are
// contiguous).  Lane j of a group holds the float4s LPR * i + j (i < 32 / LPR)
// of its row's K and V, elements 4 (LPR i + j) .. + 3, so every load
// instruction reads whole 128-byte lines and every store writes whole 32-byte
// sectors.  Bulk appends take LPR = 8 (16 elements per lane: the row's max
// reduction, reciprocal and addressing are shared by four rows per warp); a
// decode step's few new rows take LPR = 32 (a short chain per lane).  The scale
// m = max |x| (exact, order-free) is stored; codes are roundf(x / (m *
// (1/127))) clamped to [-127, 127], as the oracle computes them (IEEE quotient,
// see quantize4); an all-zero row gives zero codes.
template <int LPR>
__global__ void __launch_bounds__(256)
    kq8_append_kernel(const kq8_cache_t c, const float* __restrict__ k, const float* __restrict__ v,
                      const int32_t* __restrict__ slot, int32_t T, uint32_t* status) {
    constexpr int RPW = 32 / LPR, NI = HD / 4 / LPR;  // rows per warp, float4s per lane
    // launched programmatically: nothing is read or written before the kernel
    // before this one has completed
    griddep_wait();
    // the decode attention launched after this kernel may start its prologue
    // now; it waits for this grid's completion before reading global memory
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31, j = lane % LPR, grp = lane / LPR;
    const int64_t item0 =
        ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;
    const int nkv = c.num_kv_heads, kv_bs = c.kv_bs;
    const int64_t items = (int64_t)T * nkv;
    if (item0 >= items) return;  // warp-uniform
    const int64_t item = item0 + grp;
    int64_t t = item0 / nkv;  // one division per warp, then the group's offset
    int h = (int)(item0 - t * nkv) + grp;
    while (h >= nkv) {
        h -= nkv;
        t++;
    }
    int32_t sl = -1;
    float4 xk[NI], xv[NI];
    if (item < items) {
        sl = __ldg(slot + t);
        const float4* kr = reinterpret_cast<const float4*>(k + (size_t)item * HD) + j;
        const float4* vr = reinterpret_cast<const float4*>(v + (size_t)item * HD) + j;
#pragma unroll
        for (int i = 0; i < NI; i++) {
            xk[i] = __ldcs(kr + LPR * i);
            xv[i] = __ldcs(vr + LPR * i);
        }
    } else {
#pragma unroll
        for (int i = 0; i < NI; i++) xk[i] = xv[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    float mk = 0.0f, mv = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; i++) {
        mk = fmaxf(mk, absmax4(xk[i]));
        mv = fmaxf(mv, absmax4(xv[i]));
    }
#pragma unroll
    for (int o = 1; o < LPR; o <<= 1) {  // within the group
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        mv = fmaxf(mv, __shfl_xor_sync(0xffffffffu, mv, o));
    }
    if (sl < 0) return;  // past the end, or a skipped token (no collectives follow)
    if ((int64_t)sl >= (int64_t)c.num_pages * kv_bs) {
        if (j == 0 && status) atomicOr(status, KQ8_STATUS_BAD_SLOT);
        return;
    }
    uint32_t ck[NI], cv[NI];
#pragma unroll
    for (int i = 0; i < NI; i++) ck[i] = cv[i] = 0u;
    if (mk != 0.0f) {
        const float d = __fmul_rn(mk, inv127()), r = __frcp_rn(d);
#pragma unroll
        for (int i = 0; i < NI; i++) ck[i] = quantize4(xk[i], d, r, -127.0f, 127.0f, 0);
    }
    if (mv != 0.0f) {
        const float d = __fmul_rn(mv, inv127()), r = __frcp_rn(d);
#pragma unroll
        for (int i = 0; i < NI; i++) cv[i] = quantize4(xv[i], d, r, -127.0f, 127.0f, 0);
    }
    const int32_t page = sl / kv_bs;
    const int rr = sl - page * kv_bs;
    // K: element e of row rr at sub-tile rr/32, block e/32, position kpos(rr%32), byte e%32
    int8_t* ko = c.k + kv_sub_off(page, h, nkv, kv_bs, rr / TILE) + (size_t)kpos(rr % TILE) * 32;
    int8_t* vo = c.v + (page_head(page, h, nkv) * (size_t)kv_bs + rr) * HD;
#pragma unroll
    for (int i = 0; i < NI; i++) {
        const int e = 4 * (LPR * i + j);
        *reinterpret_cast<uint32_t*>(ko + (e >> 5) * 1024 + (e & 31)) = ck[i];
        *reinterpret_cast<uint32_t*>(vo + e) = cv[i];
    }
    if (j == 0) {
        const size_t so = page_head(page, h, nkv) * (size_t)kv_bs + rr;
        c.kscale[so] = mk;
        c.vscale[so] = mv;
    }
}

constexpr int APPEND_WARPS = 8;

// q4 write path (the q8 rule with 7 for 127): lane l holds elements 4l..4l+3
// and returns their codes as offset-binary nibbles (code + 8) in the low
// nibble of each byte.
__device__ __forceinline__ uint32_t kv_quantize_lane_q4(const float4 x, float& m_out) {
    float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    m = warp_max(m);
    m_out = m;
    if (m == 0.0f) return 0x08080808u;
    const float d = __fmul_rn(m, inv7());
    return quantize4(x, d, __frcp_rn(d), -7.0f, 7.0f, 8);
}

// One warp per (token, head) as above; lanes 2w and 2w+1 hold the 8 elements of
// packed word w (byte i = element i | element i + 4 << 4), which the even lane
// writes: K at sub-tile r/32, block w/4, position kpos(r%32), bytes 4*(w%4);
// V at row r, bytes 4w.
__global__ void __launch_bounds__(APPEND_WARPS * 32)
    kq8_append_q4_kernel(const kq8_cache_t c, const float* __restrict__ k,
                         const float* __restrict__ v, const int32_t* __restrict__ slot, int32_t T,
                         uint32_t* status) {
    griddep_wait();  // see kq8_append_kernel
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * APPEND_WARPS + (threadIdx.x >> 5);
    const int nkv = c.num_kv_heads, kv_bs = c.kv_bs;
    if (item >= (int64_t)T * nkv) return;
    const int64_t t = item / nkv;
    const int h = (int)(item % nkv);
    const int32_t sl = slot[t];
    if (sl < 0) return;
    if ((int64_t)sl >= (int64_t)c.num_pages * kv_bs) {
        if (lane == 0 && status) atomicOr(status, KQ8_STATUS_BAD_SLOT);
        return;
    }
    const int32_t page = sl / kv_bs;
    const int r = sl % kv_bs;
    const size_t row = (size_t)item * HD;
    const float4 xk = __ldcs(reinterpret_cast<const float4*>(k + row) + lane);
    const float4 xv = __ldcs(reinterpret_cast<const float4*>(v + row) + lane);
    float mk, mv;
    const uint32_t ck = kv_quantize_lane_q4(xk, mk);
    const uint32_t cv = kv_quantize_lane_q4(xv, mv);
    const uint32_t ck_hi = __shfl_down_sync(0xffffffffu, ck, 1);
    const uint32_t cv_hi = __shfl_down_sync(0xffffffffu, cv, 1);
    if ((lane & 1) == 0) {
        const int w = lane >> 1;  // packed word: elements 8w .. 8w+7
        const size_t ko = kv4_sub_off(page, h, nkv, kv_bs, r / TILE) + (size_t)(w >> 2) * 512 +
                          (size_t)kpos(r % TILE) * 16 + (size_t)(w & 3) * 4;
        *reinterpret_cast<uint32_t*>(c.k + ko) = ck | (ck_hi << 4);
        const size_t vo = page_head(page, h, nkv) * (size_t)kv_bs * (HD / 2) + (size_t)r * (HD / 2) +
                          (size_t)w * 4;
        *reinterpret_cast<uint32_t*>(c.v + vo) = cv | (cv_hi << 4);
    }
    if (lane == 0) {
        const size_t so = page_head(page, h, nkv) * (size_t)kv_bs + r;
        c.kscale[so] = mk;
        c.vscale[so] = mv;
    }
}

// The appends are programmatic launches: their CTAs may be scheduled while the
// kernel before them (typically the previous layer's attention) finishes, and
// wait for its completion before they read or write anything, so the stream
// order of the call's effects is unchanged; only the launch latency overlaps.
template <typename... KArgs, typename... Args>
static int launch_pdl(void (*kern)(KArgs...), int64_t blocks, int threads, cudaStream_t stream,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, args...) != cudaSuccess) return KQ8_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

int launch_append_q4(const kq8_cache_t& c, const float* k, const float* v, const int32_t* slot,
                     int32_t T, uint32_t* status, cudaStream_t stream) {
    const int64_t items = (int64_t)T * c.num_kv_heads;
    if (items == 0) return KQ8_OK;
    const int64_t blocks = (items + APPEND_WARPS - 1) / APPEND_WARPS;
    return launch_pdl(kq8_append_q4_kernel, blocks, APPEND_WARPS * 32, stream, c, k, v, slot, T,
                      status);
}

int launch_append(const kq8_cache_t& c, const float* k, const float* v, const int32_t* slot,
                  int32_t T, uint32_t* status, cudaStream_t stream) {
    const int64_t items = (int64_t)T * c.num_kv_heads;
    if (items == 0) return KQ8_OK;
    // bulk: four rows per warp; a small append (a decode step's new tokens):
    // one row per warp, so that each lane's chain stays short
    if (items < 8192)
        return launch_pdl(kq8_append_kernel<32>, (items + 7) / 8, 256, stream, c, k, v, slot, T,
                          status);
    return launch_pdl(kq8_append_kernel<8>, (items + 31) / 32, 256, stream, c, k, v, slot, T,
                      status);
}

// ---------------------------------------------------------------------------
// Batched prefill as per-token rows (article 10-1 §1): packed query row r of
// sequence b, the i-th of its nb new tokens, sits at position
// seq_lens[b] - nb + i and attends the prefix of length position + 1 of b's
// pages.  Writes row_seq[r] = b and row_len[r] = that length; rows outside
// every sequence get length 0, rows of an inconsistent sequence -1 (skipped
// by the attention kernels, which set KQ8_STATUS_BAD_SEQLEN).
// ---------------------------------------------------------------------------
__global__ void kq8_prefill_rows_kernel(int32_t* row_seq, int32_t* row_len, const int32_t* q_off,
                                        const int32_t* seq_lens, int32_t B, int32_t total_q,
                                        int32_t max_seq_len, int32_t max_q_len) {
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < total_q; r += gridDim.x * blockDim.x) {
        int lo = 0, hi = B + 1;  // first k in [0, B] with q_off[k] > r
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (q_off[mid] > r) hi = mid; else lo = mid + 1;
        }
        const int b = lo - 1;
        int32_t seq = 0, len = 0;
        if (b >= 0 && b < B && q_off[b] <= r && r < q_off[b + 1]) {
            const int n = seq_lens[b], nb = q_off[b + 1] - q_off[b];
            seq = b;
            const bool bad = n < 0 || n > max_seq_len || nb > n || nb > max_q_len ||
                             q_off[b] < 0 || q_off[b + 1] > total_q;
            len = bad ? -1 : n - nb + (r - q_off[b]) + 1;
        }
        row_seq[r] = seq;
        row_len[r] = len;
    }
}

int launch_prefill_rows(int32_t* row_seq, int32_t* row_len, const int32_t* q_off,
                        const int32_t* seq_lens, int32_t B, int32_t total_q, int32_t max_seq_len,
                        int32_t max_q_len, cudaStream_t s) {
    if (total_q == 0) return KQ8_OK;
    const int blocks = (int)((total_q + 255) / 256 < 1024 ? (total_q + 255) / 256 : 1024);
    kq8_prefill_rows_kernel<<<blocks, 256, 0, s>>>(row_seq, row_len, q_off, seq_lens, B, total_q,
                                                   max_seq_len, max_q_len);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Test-only: Q quantisation, one warp per row of 128.
// ---------------------------------------------------------------------------
__global__ void kq8_debug_quantize_kernel(int8_t* qi, float* qsc, const float* q, int32_t rows) {
    const int lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const float4 x = reinterpret_cast<const float4*>(q + row * HD)[lane];
    float s;
    const uint32_t codes = quantize_q_lane(x, s);
    reinterpret_cast<uint32_t*>(qi + row * HD)[lane] = codes;
    if ((lane & 7) == 0) qsc[row * NB + (lane >> 3)] = s;
}

int launch_debug_quantize(int8_t* qi, float* qsc, const float* q, int32_t rows, cudaStream_t s) {
    if (rows == 0) return KQ8_OK;
    kq8_debug_quantize_kernel<<<(rows + 3) / 4, 128, 0, s>>>(qi, qsc, q, rows);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Test-only: int32 block dots of every token with every query head, with the
// same data path as the attention kernel's score phase (K sub-tile in shared
// memory, lane = token, half-swizzled 16-byte loads, dp4a).
// grid (ceil(max_seq_len/32), nkv, B), 1 warp.
// ---------------------------------------------------------------------------
__global__ void kq8_debug_dots_kernel(int32_t* dots, const float* q, const kq8_cache_t c,
                                      const int32_t* page_table, int32_t max_pages,
                                      const int32_t* seq_lens, int32_t max_seq_len, int32_t nq) {
    __shared__ __align__(16) int8_t kt[SUB_K_BYTES];
    __shared__ __align__(16) int8_t qi[MAX_G][HD];
    const int lane = threadIdx.x;
    const int tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int nkv = c.num_kv_heads, G = nq / nkv;
    const int n = seq_lens[b];
    if (n < 0 || n > max_seq_len || tile * TILE >= n) return;
    const int32_t pg = page_table[(size_t)b * max_pages + tile / (c.kv_bs / TILE)];
    if (pg < 0 || pg >= c.num_pages) return;
    for (int g = 0; g < G; g++) {
        const float4 x = reinterpret_cast<const float4*>(q + ((size_t)b * nq + h * G + g) * HD)[lane];
        float s;
        reinterpret_cast<uint32_t*>(qi[g])[lane] = quantize_q_lane(x, s);
    }
    const int8_t* src = c.k + kv_sub_off(pg, h, nkv, c.kv_bs, tile % (c.kv_bs / TILE));
    for (int i = lane; i < SUB_K_BYTES / 16; i += 32)
        reinterpret_cast<uint4*>(kt)[i] = reinterpret_cast<const uint4*>(src)[i];
    __syncwarp();
    const int kq = lane;       // K position read by this lane
    const int t = krow(kq);    // token row it holds
    const int hs = (kq >> 2) & 1;
    for (int g = 0; g < G; g++) {
        for (int bb = 0; bb < NB; bb++) {
            const uint4 kA = *reinterpret_cast<const uint4*>(kt + bb * 1024 + kq * 32 + hs * 16);
            const uint4 kB = *reinterpret_cast<const uint4*>(kt + bb * 1024 + kq * 32 + (hs ^ 1) * 16);
            const uint4 qA = *reinterpret_cast<const uint4*>(qi[g] + bb * 32 + hs * 16);
            const uint4 qB = *reinterpret_cast<const uint4*>(qi[g] + bb * 32 + (hs ^ 1) * 16);
            int d = __dp4a((int)kA.x, (int)qA.x, 0);
            d = __dp4a((int)kA.y, (int)qA.y, d);
            d = __dp4a((int)kA.z, (int)qA.z, d);
            d = __dp4a((int)kA.w, (int)qA.w, d);
            d = __dp4a((int)kB.x, (int)qB.x, d);
            d = __dp4a((int)kB.y, (int)qB.y, d);
            d = __dp4a((int)kB.z, (int)qB.z, d);
            d = __dp4a((int)kB.w, (int)qB.w, d);
            const int tok = tile * TILE + t;
            if (tok < n)
                dots[(((size_t)b * nq + h * G + g) * max_seq_len + tok) * NB + bb] = d;
        }
    }
}

int launch_debug_dots(int32_t* dots, const float* q, const kq8_cache_t& c,
                      const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                      int32_t max_seq_len, int32_t B, int32_t nq, cudaStream_t s) {
    if (B == 0 || max_seq_len == 0) return KQ8_OK;
    dim3 grid((max_seq_len + TILE - 1) / TILE, c.num_kv_heads, B);
    kq8_debug_dots_kernel<<<grid, 32, 0, s>>>(dots, q, c, page_table, max_pages, seq_lens,
                                               max_seq_len, nq);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

}  // namespace kq8
