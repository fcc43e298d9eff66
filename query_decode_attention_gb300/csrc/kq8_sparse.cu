// kq8_sparse.cu -- launchers of the block-sparse probe and top-k kernels.
#include "kq8_internal.h"
#include "kq8_sparse.cuh"

namespace kq8 {

// The probe is a programmatic launch: its CTAs may be scheduled, and set up
// their barriers, while the kernel before it (the append of the new tokens, or
// the previous call's attention) finishes; they wait for its completion before
// they read or write global memory.
template <int G>
static int launch_probe_g(const SparseParams& p, int B, int nkv, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.max_nblk + p.probe_bpc - 1) / p.probe_bpc, nkv, B);
    cfg.blockDim = dim3(PROBE_WARPS * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.probe_tma) {
        auto kern = kq8_probe_kernel<G, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)PROBE_RING_BYTES) != cudaSuccess)
            return KQ8_ERR_CUDA;
        cfg.dynamicSmemBytes = PROBE_RING_BYTES;
        if (cudaLaunchKernelEx(&cfg, kern, p) != cudaSuccess) return KQ8_ERR_CUDA;
    } else {
        cfg.dynamicSmemBytes = 0;
        if (cudaLaunchKernelEx(&cfg, kq8_probe_kernel<G, false>, p) != cudaSuccess)
            return KQ8_ERR_CUDA;
    }
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

template <int G>
static int launch_topk_g(const SparseParams& p, int B, int nkv, cudaStream_t s) {
    dim3 grid(nkv, B);
    kq8_topk_kernel<G><<<grid, TOPK_THREADS, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

#define KQ8_SWITCH_G(F, ...)                 \
    switch (G) {                             \
        case 1: return F<1>(__VA_ARGS__);    \
        case 2: return F<2>(__VA_ARGS__);    \
        case 3: return F<3>(__VA_ARGS__);    \
        case 4: return F<4>(__VA_ARGS__);    \
        case 5: return F<5>(__VA_ARGS__);    \
        case 6: return F<6>(__VA_ARGS__);    \
        case 7: return F<7>(__VA_ARGS__);    \
        case 8: return F<8>(__VA_ARGS__);    \
        default: return KQ8_ERR_UNSUPPORTED; \
    }

// Blocks per probe CTA: as many as keep the pages they span within the CTA's
// staged page ids (a CTA's blocks span at most bpc * block / kv_bs + 1 pages).
int probe_blocks_per_cta(int block, int kv_bs) {
    const long long bpc = (long long)(PROBE_MAX_PAGES - 1) * kv_bs / block;
    return (int)(bpc < 1 ? 1 : (bpc > PROBE_MAX_BPC ? PROBE_MAX_BPC : bpc));
}

int launch_probe(const SparseParams& p, int G, int B, int nkv, cudaStream_t s) {
    if (B == 0) return KQ8_OK;
    if (p.max_nblk == 0) {
        if (!p.tickets) return KQ8_OK;
        // every sequence is empty: CTA 0 of each (sequence, KV head) still
        // writes its (empty) list and clears its selection
        SparseParams q = p;
        q.max_nblk = 1;
        KQ8_SWITCH_G(launch_probe_g, q, B, nkv, s)
    }
    if (p.probe_bpc < 1 || (long long)p.probe_bpc * p.block / p.cache.kv_bs + 1 > PROBE_MAX_PAGES)
        return KQ8_ERR_INVALID_ARG;
    KQ8_SWITCH_G(launch_probe_g, p, B, nkv, s)
}

// Only needed without tickets: otherwise the probe kernel's last CTA of each
// (sequence, KV head) has already selected.
int launch_topk(const SparseParams& p, int G, int B, int nkv, cudaStream_t s) {
    if (B == 0 || p.tickets) return KQ8_OK;
    KQ8_SWITCH_G(launch_topk_g, p, B, nkv, s)
}

}  // namespace kq8
