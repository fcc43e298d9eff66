// kq8_common.cuh -- device helpers shared by the libkq8 kernels (sm_103a).
//
// Cache layout, per (page p, KV head h), head_dim 128, kv_bs a multiple of 32:
//   K: kv_bs/32 sub-tiles of 4 KB; sub-tile = 4 blocks (32 elements each) x
//      32 row positions x 32 B -> byte (r, i) at
//      (r/32)*4096 + (i/32)*1024 + kpos(r%32)*32 + i%32, where row r of a
//      sub-tile sits at position kpos(r) = (r%4)*8 + r/4: rows 0, 4, 8, ...
//      are adjacent, so a block probe at a stride of 4 rows reads whole lines
//   V: kv_bs rows of 128 B (token-major)
//   kscale, vscale: kv_bs floats (the row's max |x|)
// One 32-token sub-tile of one head is therefore 4096 B of K + 4096 B of V +
// 128 B + 128 B of scales, each a contiguous, 16-byte aligned range: it is
// staged into shared memory by four bulk-async copies.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "kq8.h"

namespace kq8 {

constexpr int HD = 128;              // supported head dim
constexpr int NB = HD / 32;          // 32-element blocks per row
constexpr int TILE = 32;             // tokens per sub-tile
constexpr int SUB_K_BYTES = TILE * HD;
constexpr int SUB_V_BYTES = TILE * HD;
constexpr int SUB_S_BYTES = TILE * 4;
constexpr int STAGE_BYTES = SUB_K_BYTES + SUB_V_BYTES + 2 * SUB_S_BYTES;  // 8448
constexpr float M_INIT = -1e9f;      // running-max start of the online softmax
constexpr int MAX_G = 8;             // query heads per KV head handled

// The inverse of 127 as a float: the per-row step is max|x| * (1/127) and the
// readers multiply stored maxima by it (article 9-2 §2, article 9-3 §2).
__host__ __device__ constexpr float inv127() { return 1.0f / 127.0f; }
// q4 cache (the --kv-q4 switch of article 10-1 §2; no page gives the format):
// the same rule with 7 levels a side -- step max|x| * (1/7), codes in [-7, 7].
__host__ __device__ constexpr float inv7() { return 1.0f / 7.0f; }

// ---------------------------------------------------------------------------
// Cache addressing
// ---------------------------------------------------------------------------
// Position of row r (0..31) of a K sub-tile, and the row held at position q.
__host__ __device__ __forceinline__ int kpos(int r) { return (r & 3) * 8 + (r >> 2); }
__host__ __device__ __forceinline__ int krow(int q) { return (q & 7) * 4 + (q >> 3); }
__device__ __forceinline__ size_t page_head(int32_t page, int h, int nkv) {
    return (size_t)page * (size_t)nkv + (size_t)h;
}
// q4 cache layout, per (page p, KV head h): codes as 4-bit offset binary
// (nibble = code + 8); within every 4-byte word of a row, byte i holds
// element i in its low nibble and element i + 4 in its high nibble, so a
// word covers 8 consecutive elements.
//   K: kv_bs/32 sub-tiles of 2 KB = 4 blocks x 32 row positions (kpos) x 16 B
//   V: kv_bs rows of 64 B;  kscale, vscale as for q8
constexpr int SUB_K4_BYTES = TILE * HD / 2;
constexpr int SUB_V4_BYTES = TILE * HD / 2;
__device__ __forceinline__ size_t kv4_sub_off(int32_t page, int h, int nkv, int kv_bs, int sub) {
    return page_head(page, h, nkv) * (size_t)kv_bs * (HD / 2) + (size_t)sub * SUB_K4_BYTES;
}

// Byte offset of sub-tile `sub` of (page, head) in the K or V array.
__device__ __forceinline__ size_t kv_sub_off(int32_t page, int h, int nkv, int kv_bs, int sub) {
    return page_head(page, h, nkv) * (size_t)kv_bs * HD + (size_t)sub * (TILE * HD);
}
__device__ __forceinline__ size_t scale_sub_off(int32_t page, int h, int nkv, int kv_bs, int sub) {
    return page_head(page, h, nkv) * (size_t)kv_bs + (size_t)sub * TILE;
}

// ---------------------------------------------------------------------------
// PTX wrappers: mbarrier + bulk async copies (global -> shared)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
// Ends a barrier's life (no copy may be pending on it) so that it can be
// initialised again.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
        "%2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// Tensor copy of one box of a 3-D tensor map (global -> shared), completion on
// an mbarrier; coordinates innermost first.  The destination must be aligned
// to the map's swizzle span (1024 bytes for the 128-byte swizzle).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)),
        "l"(policy)
        : "memory");
}

// Four 8x8 matrices of 16-bit elements from shared memory, transposed: lanes
// 8i..8i+7 give the row addresses of matrix i; lane (g = lane/4, c = lane%4)
// receives in register i the elements (row 2c, column g) and (row 2c+1, column g).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D (16x8 fp32) += A (16x16 fp16, row-major) * B (16x8 fp16, column-major), one warp.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two floats -> fp16x2 (round to nearest): x in the low half, y in the high half.
__device__ __forceinline__ uint32_t f2_to_h2(float x, float y) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(y), "f"(x));
    return r;
}
// fp16x2 -> two floats (exact).
__device__ __forceinline__ float2 h2_to_f2(uint32_t h) {
    float x, y;
    asm("{ .reg .f16 lo, hi; mov.b32 {lo, hi}, %2; cvt.f32.f16 %0, lo; cvt.f32.f16 %1, hi; }"
        : "=f"(x), "=f"(y)
        : "r"(h));
    return make_float2(x, y);
}
// Packed fp16 subtract a - b.
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// Programmatic dependent launch: let the next kernel in the stream (launched
// with programmatic serialisation) start, and, in that kernel, wait until the
// kernel before it has completed and its writes are visible.  Both are no-ops
// for an ordinary launch.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// (a & b) | c in one three-input logic op.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
// Packed fp16 a * b + c, one rounding.
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
// 2^k as a float for k in [-126, 127].
__device__ __forceinline__ float pow2i(int k) { return __uint_as_float((uint32_t)(k + 127) << 23); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, "
        "p; }"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after 2^28 SM clocks (~0.13 s at 2 GHz) and returns
// false; the caller records KQ8_STATUS_TIMEOUT.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > (1ll << 28)) return false;
    }
    return true;
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------
// Exact int32 -> float for |x| < 2^22: place x in the mantissa of 1.5 * 2^23.
__device__ __forceinline__ float i2f_exact(int x) {
    return __int_as_float(0x4B400000 + x) - 12582912.0f;
}

// Four int8 codes in one word -> four floats, exactly: flip the sign bits to
// get offset-binary u = c + 128, drop each byte into the mantissa of 2^23
// (one byte permute each) and subtract 2^23 + 128 (two packed adds).
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float& f0, float& f1, float& f2, float& f3) {
    const uint32_t u = w ^ 0x80808080u;
    uint32_t a = __byte_perm(u, 0x4B000000u, 0x7540);
    uint32_t b = __byte_perm(u, 0x4B000000u, 0x7541);
    uint32_t c = __byte_perm(u, 0x4B000000u, 0x7542);
    uint32_t d = __byte_perm(u, 0x4B000000u, 0x7543);
    const float bias = 8388736.0f;  // 2^23 + 128
    uint64_t ab, cd;
    asm("{ .reg .b64 x, y; mov.b64 x, {%1, %2}; mov.b64 y, {%3, %3};"
        " sub.rn.f32x2 %0, x, y; }"
        : "=l"(ab)
        : "r"(a), "r"(b), "f"(bias));
    asm("{ .reg .b64 x, y; mov.b64 x, {%1, %2}; mov.b64 y, {%3, %3};"
        " sub.rn.f32x2 %0, x, y; }"
        : "=l"(cd)
        : "r"(c), "r"(d), "f"(bias));
    f0 = __uint_as_float((uint32_t)ab);
    f1 = __uint_as_float((uint32_t)(ab >> 32));
    f2 = __uint_as_float((uint32_t)cd);
    f3 = __uint_as_float((uint32_t)(cd >> 32));
}

// acc (2 floats) += x (2 floats) * p (scalar), one packed FMA.
__device__ __forceinline__ void ffma2(float2& acc, float x0, float x1, float p) {
    uint64_t a;
    asm("{ .reg .b64 x, y, z; mov.b64 x, {%1, %2}; mov.b64 y, {%3, %3}; mov.b64 z, {%4, %5};"
        " fma.rn.f32x2 %0, x, y, z; }"
        : "=l"(a)
        : "f"(x0), "f"(x1), "f"(p), "f"(acc.x), "f"(acc.y));
    acc.x = __uint_as_float((uint32_t)a);
    acc.y = __uint_as_float((uint32_t)(a >> 32));
}

__device__ __forceinline__ void fmul2(float2& acc, float c) {
    uint64_t a;
    asm("{ .reg .b64 x, y; mov.b64 x, {%1, %2}; mov.b64 y, {%3, %3}; mul.rn.f32x2 %0, x, y; }"
        : "=l"(a)
        : "f"(acc.x), "f"(acc.y), "f"(c));
    acc.x = __uint_as_float((uint32_t)a);
    acc.y = __uint_as_float((uint32_t)(a >> 32));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------------------
// Q quantisation (article 9-2 §2 segment 1), one warp per query head.
// Lane l holds elements 4l..4l+3 (block l/8).  Per 32-element block: qm =
// max |x| (qm < 1e-6 -> 1), qsc = qm * (1/127), iq = 127 / qm (IEEE divide),
// code = trunc(clamp(x * iq, -128, 127)).  Bit-identical to the oracle: every
// operation is a single IEEE-rounded fp32 op and the max is order-free.
// Writes the 4 codes of the lane as one word and returns the lane's block
// scale.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t quantize_q_lane(const float4 x, float& qsc_out) {
    float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    if (m < 1e-6f) m = 1.0f;
    qsc_out = __fmul_rn(m, inv127());
    const float iq = __fdiv_rn(127.0f, m);
    auto code = [&](float v) -> uint32_t {
        float t = __fmul_rn(v, iq);
        t = fminf(fmaxf(t, -128.0f), 127.0f);
        return (uint32_t)(__float2int_rz(t) & 0xff);
    };
    return code(x.x) | (code(x.y) << 8) | (code(x.z) << 16) | (code(x.w) << 24);
}

// Score of one token from its 4 int32 block dots (article 9-2 §2 segment 2):
// s = ((((0 + d0*c0) + d1*c1) + d2*c2) + d3*c3), s = (s * ks) * scale with
// ks = kscale * (1/127); every product and sum rounded separately, in that
// order, so the value matches the oracle bit for bit.
__device__ __forceinline__ float score_exact(const int d[NB], const float c[NB], float kstored,
                                             float scale) {
    const float ks = __fmul_rn(kstored, inv127());
    float s = 0.0f;
#pragma unroll
    for (int b = 0; b < NB; b++) s = __fadd_rn(s, __fmul_rn(i2f_exact(d[b]), c[b]));
    return __fmul_rn(__fmul_rn(s, ks), scale);
}

}  // namespace kq8
