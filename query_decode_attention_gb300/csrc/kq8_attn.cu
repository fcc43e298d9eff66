// kq8_attn.cu -- launchers of the split-KV attention kernel and the merge.
#include "kq8_attn.cuh"
#include "kq8_internal.h"

namespace kq8 {

size_t attn_smem_bytes(int G);

template <int G, bool SPARSE, bool Q4, bool WITHHOLD = false>
static int launch_attn_g(const AttnParams& p, int B, int nkv, cudaStream_t s) {
    auto kern = kq8_attn_kernel<G, SPARSE, Q4, WITHHOLD>;
    const size_t smem = attn_smem_bytes(G);
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return KQ8_ERR_CUDA;
    dim3 grid(p.num_chunks, nkv, B);
    {
        // programmatic launch: the CTAs may start, and set up their barriers,
        // while the kernel before them (the append of the new tokens, or the
        // selection) finishes; they wait for its completion before they read or
        // write global memory.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(ATTN_THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return KQ8_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return KQ8_ERR_CUDA;
    if (p.num_chunks > 1 && p.counters == nullptr) {
        kq8_merge_kernel<SPARSE><<<B * p.nq, HD, 0, s>>>(p);
        if (cudaGetLastError() != cudaSuccess) return KQ8_ERR_CUDA;
    }
    return KQ8_OK;
}

template <bool SPARSE, bool Q4>
static int launch_attn_s(const AttnParams& p, int G, int B, int nkv, cudaStream_t s) {
    switch (G) {
        case 1: return launch_attn_g<1, SPARSE, Q4>(p, B, nkv, s);
        case 2: return launch_attn_g<2, SPARSE, Q4>(p, B, nkv, s);
        case 3: return launch_attn_g<3, SPARSE, Q4>(p, B, nkv, s);
        case 4: return launch_attn_g<4, SPARSE, Q4>(p, B, nkv, s);
        case 5: return launch_attn_g<5, SPARSE, Q4>(p, B, nkv, s);
        case 6: return launch_attn_g<6, SPARSE, Q4>(p, B, nkv, s);
        case 7: return launch_attn_g<7, SPARSE, Q4>(p, B, nkv, s);
        case 8: return launch_attn_g<8, SPARSE, Q4>(p, B, nkv, s);
        default: return KQ8_ERR_UNSUPPORTED;
    }
}

int launch_attn(const AttnParams& p, int G, bool sparse, int B, int nkv, cudaStream_t s) {
    if (B == 0) return KQ8_OK;
    return sparse ? launch_attn_s<true, false>(p, G, B, nkv, s)
                  : launch_attn_s<false, false>(p, G, B, nkv, s);
}

int launch_attn_q4(const AttnParams& p, int G, int B, int nkv, cudaStream_t s) {
    if (B == 0) return KQ8_OK;
    return launch_attn_s<false, true>(p, G, B, nkv, s);
}

// The exact decode with the failure-detection hook compiled in (p.withhold).
int launch_attn_withhold(const AttnParams& p, int G, int B, int nkv, cudaStream_t s) {
    if (B == 0) return KQ8_OK;
    switch (G) {
        case 1: return launch_attn_g<1, false, false, true>(p, B, nkv, s);
        case 2: return launch_attn_g<2, false, false, true>(p, B, nkv, s);
        case 4: return launch_attn_g<4, false, false, true>(p, B, nkv, s);
        case 8: return launch_attn_g<8, false, false, true>(p, B, nkv, s);
        default: return KQ8_ERR_UNSUPPORTED;
    }
}

// Running states: reset to empty (max -1e9, sum 0, acc 0) and finalise to
// out = acc / S (0 for an empty state), one block of HD threads per row.
__global__ void __launch_bounds__(HD) kq8_state_reset_kernel(float* acc, float2* ms) {
    acc[(size_t)blockIdx.x * HD + threadIdx.x] = 0.0f;
    if (threadIdx.x == 0) ms[blockIdx.x] = make_float2(M_INIT, 0.0f);
}
__global__ void __launch_bounds__(HD) kq8_state_finalize_kernel(float* out, const float* acc,
                                                                const float2* ms) {
    const float s = ms[blockIdx.x].y;
    const size_t i = (size_t)blockIdx.x * HD + threadIdx.x;
    out[i] = (s > 0.0f) ? acc[i] / s : 0.0f;
}

// Folds `parts` partial states (each [rows][HD] + [rows] (max, sum), the
// running-state format) into the running state in order, by their
// log-sum-exp: M = max, both sides scaled by 2^(their max - M) and added.
__global__ void __launch_bounds__(HD) kq8_state_merge_kernel(float* acc, float2* ms,
                                                             const float* pacc, const float2* pms,
                                                             int parts, int rows) {
    const int row = blockIdx.x, d = threadIdx.x;
    float2 cur = ms[row];
    float a = acc[(size_t)row * HD + d];
    for (int r = 0; r < parts; r++) {
        const size_t pr = (size_t)r * rows + row;
        const float2 p = pms[pr];
        float M, S, fo, fn;
        fold_state(cur.x, cur.y, p.x, p.y, M, S, fo, fn);
        a = a * fo + pacc[pr * HD + d] * fn;
        cur = make_float2(M, S);
    }
    acc[(size_t)row * HD + d] = a;
    if (d == 0) ms[row] = cur;
}

int launch_state_merge(float* acc, float2* ms, const float* pacc, const float2* pms, int parts,
                       int rows, cudaStream_t s) {
    if (rows == 0 || parts == 0) return KQ8_OK;
    kq8_state_merge_kernel<<<rows, HD, 0, s>>>(acc, ms, pacc, pms, parts, rows);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

int launch_state_reset(float* acc, float2* ms, int rows, cudaStream_t s) {
    if (rows == 0) return KQ8_OK;
    kq8_state_reset_kernel<<<rows, HD, 0, s>>>(acc, ms);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

int launch_state_finalize(float* out, const float* acc, const float2* ms, int rows, cudaStream_t s) {
    if (rows == 0) return KQ8_OK;
    kq8_state_finalize_kernel<<<rows, HD, 0, s>>>(out, acc, ms);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

// Dynamic shared memory of the attention kernel: its AttnSmem plus 1 KB of
// slack to align the V tiles to 1024 bytes.
size_t attn_smem_bytes(int G) {
    size_t b;
    switch (G) {
        case 1: b = sizeof(AttnSmem<1>); break;
        case 2: b = sizeof(AttnSmem<2>); break;
        case 3: b = sizeof(AttnSmem<3>); break;
        case 4: b = sizeof(AttnSmem<4>); break;
        case 5: b = sizeof(AttnSmem<5>); break;
        case 6: b = sizeof(AttnSmem<6>); break;
        case 7: b = sizeof(AttnSmem<7>); break;
        default: b = sizeof(AttnSmem<8>); break;
    }
    return b + 1024;
}

}  // namespace kq8
