// kq8_api.cu -- the C ABI of libkq8 (declared in include/kq8.h): argument
// checks, workspace planning and kernel dispatch.  All compute runs in the
// CUDA kernels; this file only validates, plans and launches.
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "kq8_attn.cuh"
#include "kq8_internal.h"
#include "kq8_sparse.cuh"

namespace kq8 {

size_t attn_smem_bytes(int G);

namespace {

constexpr size_t WS_ALIGN = 256;
constexpr size_t STATUS_BYTES = 256;
// Chunk counters for the merge folded into the attention kernel: one per
// (sequence, KV head), in a fixed region right after the status word, zero
// between calls (kq8_workspace_init clears them, the merging CTA resets its
// own).  Larger batches fall back to the separate merge kernel.
constexpr size_t MAX_COUNTERS = 16384;
constexpr size_t HEADER_BYTES = STATUS_BYTES + MAX_COUNTERS * sizeof(uint32_t);

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// SMs of the current device; without one (plans asked for on a host without a
// GPU) a GB300's 152.
int device_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 152;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return 152;
    return sms;
}

#ifndef KQ8_MAX_CHUNK
#define KQ8_MAX_CHUNK 128
#endif
// Split of each (sequence, KV head) list of `tiles_max` 32-token tiles into
// chunks of `chunk_tiles` tiles (a multiple of the CTA's 4 warps), for
// `per_sm` resident attention CTAs per SM.  If every list fits one wave of CTAs
// with chunks of at most KQ8_MAX_CHUNK tiles, the chunks are sized for exactly
// one wave (no tail of a few long CTAs that cannot keep HBM busy), with at most
// 16 chunks per list.  Otherwise
// they are sized for about four waves, between 4 and KQ8_MAX_CHUNK tiles (128 to
// 4096 tokens): each CTA has a prologue and a merge tail in which it streams
// nothing, so large problems take long chunks.
void chunking(int64_t B, int64_t nkv, int64_t tiles_max, int sms, int per_sm, int& ct, int& nch) {
    static_assert(KQ8_MAX_CHUNK % ATTN_WARPS == 0 && KQ8_MAX_CHUNK <= MAX_CHUNK_TILES, "chunk");
    const int64_t pairs = B * nkv > 0 ? B * nkv : 1;
    const int64_t slots = (int64_t)sms * per_sm;
    // chunks per list that one wave holds; at most 16: past that (batch 1 or 2)
    // the merge of the chunks' partials costs more than the added streams give
    int64_t per = slots / pairs;
    if (per > 16) per = 16;
    int64_t c;
    if (per >= 1 && (tiles_max + per - 1) / per <= KQ8_MAX_CHUNK) {
        c = (tiles_max + per - 1) / per;
    } else {
        const int64_t total = pairs * tiles_max;
        const int64_t target = slots * 4;
        c = (total + target - 1) / (target > 0 ? target : 1);
    }
    c = (c + ATTN_WARPS - 1) / ATTN_WARPS * ATTN_WARPS;
    if (c < ATTN_WARPS) c = ATTN_WARPS;
    if (c > KQ8_MAX_CHUNK) c = KQ8_MAX_CHUNK;
    ct = (int)c;
    nch = (int)((tiles_max + c - 1) / c);
    if (nch < 1) nch = 1;
}

// Resident attention CTAs per SM (registers and shared memory of the kernel).
int attn_ctas_per_sm(int G) { return G <= 4 ? 3 : 2; }

// The block-sparse lists are short (at most G * k blocks): sized for a single
// wave of resident CTAs instead, as few chunks per list as fill it, so
// that no CTA is left with a prologue and a merge for a couple of tiles.
void chunking_one_wave(int64_t B, int64_t nkv, int64_t tiles_max, int sms, int per_sm, int& ct,
                       int& nch) {
    const int64_t pairs = B * nkv > 0 ? B * nkv : 1;
    int64_t per = ((int64_t)sms * per_sm) / pairs;  // chunks per list that still fit one wave
    if (per < 1) per = 1;
    int64_t c = (tiles_max + per - 1) / per;
    c = (c + ATTN_WARPS - 1) / ATTN_WARPS * ATTN_WARPS;
    if (c < ATTN_WARPS) c = ATTN_WARPS;
    if (c > KQ8_MAX_CHUNK) c = KQ8_MAX_CHUNK;
    ct = (int)c;
    nch = (int)((tiles_max + c - 1) / c);
    if (nch < 1) nch = 1;
}

struct Plan {
    int chunk_tiles = ATTN_WARPS, num_chunks = 1;
    size_t off_ms = 0, off_acc = 0;
    int max_nblk = 0, list_cap = 0;
    size_t off_scores = 0, off_masks = 0, off_list = 0, off_len = 0;
    size_t total = HEADER_BYTES;
};

Plan plan_exact(int B, int nq, int nkv, int max_seq_len) {
    Plan p;
    const int64_t tiles = ((int64_t)max_seq_len + TILE - 1) / TILE;
    chunking(B, nkv, tiles, device_sms(), attn_ctas_per_sm(nkv > 0 ? nq / nkv : 1), p.chunk_tiles,
             p.num_chunks);
    size_t o = HEADER_BYTES;
    p.off_ms = o;
    o = align_up(o + (size_t)B * nq * p.num_chunks * sizeof(float2), WS_ALIGN);
    p.off_acc = o;
    o = align_up(o + (size_t)B * nq * p.num_chunks * HD * sizeof(float), WS_ALIGN);
    p.total = o;
    return p;
}

// The exact plan's workspace layout with chunks sized for token ranges of at
// most max_range tokens (streaming updates): more, shorter chunks per range, but
// never more chunks than the full plan, so its workspace still suffices.
Plan plan_exact_range(int B, int nq, int nkv, int max_seq_len, int max_range) {
    Plan p = plan_exact(B, nq, nkv, max_seq_len);
    if (max_range <= 0 || max_range >= max_seq_len) return p;
    // a range not starting on a tile boundary touches one tile more
    const int64_t tiles = ((int64_t)max_range + TILE - 1) / TILE + 1;
    int ct, nch;
    chunking(B, nkv, tiles, device_sms(), attn_ctas_per_sm(nkv > 0 ? nq / nkv : 1), ct, nch);
    if (nch > p.num_chunks) {
        ct = (int)((tiles + p.num_chunks - 1) / p.num_chunks);
        ct = (ct + ATTN_WARPS - 1) / ATTN_WARPS * ATTN_WARPS;
        nch = (int)((tiles + ct - 1) / ct);
    }
    p.chunk_tiles = ct;
    p.num_chunks = nch;
    return p;
}

Plan plan_sparse(int B, int nq, int nkv, int max_seq_len, int block, int topk) {
    Plan p;
    const int G = nq / nkv;
    const int m = block / TILE;
    const int64_t tiles = ((int64_t)max_seq_len + TILE - 1) / TILE;
    p.max_nblk = (int)(((int64_t)max_seq_len + block - 1) / block);
    int64_t cap = (int64_t)(p.max_nblk < (int64_t)G * topk ? p.max_nblk : (int64_t)G * topk) * m;
    if (cap > tiles) cap = tiles;
    if (cap < 2 * m && cap < tiles) cap = tiles < 2 * m ? tiles : 2 * m;
    if (cap < 1) cap = 1;
    p.list_cap = (int)cap;
    chunking_one_wave(B, nkv, p.list_cap, device_sms(), attn_ctas_per_sm(G), p.chunk_tiles,
                      p.num_chunks);
    size_t o = HEADER_BYTES;
    p.off_scores = o;
    o = align_up(o + (size_t)B * nq * p.max_nblk * sizeof(float), WS_ALIGN);
    p.off_masks = o;
    o = align_up(o + (size_t)B * nkv * p.max_nblk * sizeof(uint32_t), WS_ALIGN);
    p.off_list = o;
    o = align_up(o + (size_t)B * nkv * p.list_cap * sizeof(int32_t), WS_ALIGN);
    p.off_len = o;
    o = align_up(o + (size_t)B * nkv * sizeof(int32_t), WS_ALIGN);
    p.off_ms = o;
    o = align_up(o + (size_t)B * nq * p.num_chunks * sizeof(float2), WS_ALIGN);
    p.off_acc = o;
    o = align_up(o + (size_t)B * nq * p.num_chunks * HD * sizeof(float), WS_ALIGN);
    p.total = o;
    return p;
}

int check_decode(float* out, const float* q, const kq8_cache_t* c, const int32_t* pt,
                 int32_t max_pages, const int32_t* seq_lens, int32_t max_seq_len, int32_t B,
                 int32_t nq) {
    int rc = check_cache_args(c);
    if (rc) return rc;
    if (B < 0 || nq < 1 || max_seq_len < 0 || max_pages < 0) return KQ8_ERR_INVALID_ARG;
    if (nq % c->num_kv_heads != 0) return KQ8_ERR_UNSUPPORTED;
    const int G = nq / c->num_kv_heads;
    if (G < 1 || G > MAX_G) return KQ8_ERR_UNSUPPORTED;
    if ((int64_t)max_seq_len > (int64_t)max_pages * c->kv_bs) return KQ8_ERR_INVALID_ARG;
    if (max_seq_len >= (1 << 29)) return KQ8_ERR_UNSUPPORTED;
    if (B > 65535) return KQ8_ERR_UNSUPPORTED;
    if (B > 0) {
        if (!out || !q || !seq_lens || (max_seq_len > 0 && !pt)) return KQ8_ERR_INVALID_ARG;
        if (!aligned(out, 16) || !aligned(q, 16)) return KQ8_ERR_INVALID_ARG;
    }
    return KQ8_OK;
}

int check_ws(void* ws, size_t bytes, size_t need) {
    if (!ws || !aligned(ws, WS_ALIGN)) return KQ8_ERR_WORKSPACE;
    if (bytes < need) return KQ8_ERR_WORKSPACE;
    return KQ8_OK;
}

AttnParams attn_params(float* out, const float* q, const kq8_cache_t* c, const int32_t* pt,
                       int32_t max_pages, const int32_t* seq_lens, int32_t max_seq_len, int32_t B,
                       int32_t nq, float scale, const Plan& plan, void* ws) {
    AttnParams p;
    std::memset(&p, 0, sizeof(p));
    p.out = out;
    p.q = q;
    p.cache = *c;
    p.page_table = pt;
    p.max_pages = max_pages;
    p.seq_lens = seq_lens;
    p.max_seq_len = max_seq_len;
    p.B = B;
    p.nq = nq;
    p.scale = scale;
    p.chunk_tiles = plan.chunk_tiles;
    p.num_chunks = plan.num_chunks;
    p.part_ms = reinterpret_cast<float2*>(static_cast<char*>(ws) + plan.off_ms);
    p.part_acc = reinterpret_cast<float*>(static_cast<char*>(ws) + plan.off_acc);
    p.status = static_cast<uint32_t*>(ws);
    p.counters = ((size_t)B * (size_t)c->num_kv_heads <= MAX_COUNTERS)
                     ? reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + STATUS_BYTES)
                     : nullptr;
    p.withhold = -1;
    return p;
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link to the
// driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The V array as the 3-D tensor the attention kernel copies sub-tiles of:
// {row bytes, kv_bs rows, num_pages * nkv (page, head) pairs}, boxes of 32 rows.
// q8 rows are 128 bytes (128-byte swizzle in shared memory), q4 rows 64 bytes
// (64-byte swizzle).
int set_vmap(AttnParams& p, bool q4 = false) {
    const kq8_cache_t& c = p.cache;
    const uint64_t pairs = (uint64_t)c.num_pages * (uint64_t)c.num_kv_heads;
    if (pairs > 0x7FFFFFFFull) return KQ8_ERR_UNSUPPORTED;  // the copy's coordinate is int32
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return KQ8_ERR_CUDA;
    const cuuint64_t row = q4 ? HD / 2 : HD;
    const cuuint64_t dims[3] = {row, (cuuint64_t)c.kv_bs, (cuuint64_t)pairs};
    const cuuint64_t strides[2] = {row, (cuuint64_t)c.kv_bs * row};
    const cuuint32_t box[3] = {(cuuint32_t)row, (cuuint32_t)TILE, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(&p.vmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.v, dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           q4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? KQ8_OK : KQ8_ERR_CUDA;
}

// The K array as the probe's 3-D tensor {1024 B: 32 positions x 32 B, 4 element
// blocks, num_pages * nkv * kv_bs / 32 sub-tiles}, boxes of the first 8
// positions of the 4 blocks (4 x 256 B), unswizzled.  Only for block = 4 *
// probe, where every probe row sits at positions 0..7 of its sub-tile; the
// probe keeps its register form otherwise (or when the map cannot be made).
void set_probe_kmap(SparseParams& sp) {
    sp.probe_tma = 0;
    if (sp.block != 4 * sp.probe) return;
    const kq8_cache_t& c = sp.cache;
    const uint64_t subtiles =
        (uint64_t)c.num_pages * (uint64_t)c.num_kv_heads * (uint64_t)(c.kv_bs / TILE);
    if (subtiles == 0 || subtiles > 0x7FFFFFFFull) return;  // the copy's coordinate is int32
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return;
    const cuuint64_t dims[3] = {(cuuint64_t)TILE * 32, (cuuint64_t)NB, (cuuint64_t)subtiles};
    const cuuint64_t strides[2] = {(cuuint64_t)TILE * 32, (cuuint64_t)TILE * HD};
    const cuuint32_t box[3] = {8u * 32u, (cuuint32_t)NB, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (enc(&sp.kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.k, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
        sp.probe_tma = 1;
}

// Probe, top-k and bounded attention over `rows` decode rows (article 10-1
// §1-§2); row_seq (optional) maps each row to its page-table row.
int run_sparse(float* out, const float* q, const kq8_cache_t* cache, const int32_t* page_table,
               int32_t max_pages, const int32_t* row_len, const int32_t* row_seq,
               int32_t max_seq_len, int32_t rows, int32_t nq, float scale, int32_t block,
               int32_t topk, int32_t probe, int32_t* sel_blocks, const Plan& plan,
               void* workspace, cudaStream_t s, bool shared_sel = false) {
    const int nkv = cache->num_kv_heads;
    const int G = nq / nkv;
    char* ws = static_cast<char*>(workspace);
    SparseParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.q = q;
    sp.cache = *cache;
    sp.page_table = page_table;
    sp.max_pages = max_pages;
    sp.seq_lens = row_len;
    sp.max_seq_len = max_seq_len;
    sp.B = rows;
    sp.nq = nq;
    sp.scale = scale;
    sp.block = block;
    sp.topk = topk;
    sp.probe = probe;
    sp.max_nblk = plan.max_nblk;
    sp.probe_bpc = probe_blocks_per_cta(block, cache->kv_bs);
    {
        // A probe grid that does not fill the SMs once (small batches) is latency,
        // not bytes: give each (sequence, KV head) more, shorter CTAs, in steps of
        // 32 blocks (one unit of 4 blocks for each of the 8 warps).
        const long long pairs = (long long)rows * nkv;
        const int sms = device_sms();
        const long long cpp = (plan.max_nblk + sp.probe_bpc - 1) / sp.probe_bpc;
        if (pairs > 0 && pairs * cpp < sms) {
            const long long want = sms / pairs > 1 ? sms / pairs : 1;
            long long bpc = (plan.max_nblk + want - 1) / want;
            bpc = (bpc + 31) / 32 * 32;
            if (bpc < sp.probe_bpc) sp.probe_bpc = (int)bpc;
        }
    }
    set_probe_kmap(sp);
    sp.scores = reinterpret_cast<float*>(ws + plan.off_scores);
    sp.masks = reinterpret_cast<uint32_t*>(ws + plan.off_masks);
    sp.tile_list = reinterpret_cast<int32_t*>(ws + plan.off_list);
    sp.list_len = reinterpret_cast<int32_t*>(ws + plan.off_len);
    sp.list_cap = plan.list_cap;
    sp.sel_blocks = sel_blocks;
    sp.status = reinterpret_cast<uint32_t*>(ws);
    sp.row_seq = row_seq;
    sp.shared_sel = shared_sel ? 1 : 0;
    // the selection tickets (the probe kernel's last CTA of a (sequence, KV
    // head) selects) share the header's per-(sequence, KV head) counters with
    // the attention kernel's chunk merge: both leave them at zero; without
    // them a separate top-k kernel selects
    sp.tickets = ((size_t)rows * (size_t)nkv <= MAX_COUNTERS)
                     ? reinterpret_cast<uint32_t*>(ws + STATUS_BYTES)
                     : nullptr;
    int rc = launch_probe(sp, G, rows, nkv, s);
    if (rc) return rc;
    rc = launch_topk(sp, G, rows, nkv, s);
    if (rc) return rc;
    AttnParams p = attn_params(out, q, cache, page_table, max_pages, row_len, max_seq_len, rows,
                               nq, scale, plan, workspace);
    p.tile_list = sp.tile_list;
    p.list_len = sp.list_len;
    p.list_cap = sp.list_cap;
    p.row_seq = row_seq;
    rc = set_vmap(p);
    if (rc) return rc;
    return launch_attn(p, G, true, rows, nkv, s);
}

}  // namespace

int check_cache_args(const kq8_cache_t* c) {
    if (!c) return KQ8_ERR_INVALID_ARG;
    if (c->head_dim != HD) return KQ8_ERR_UNSUPPORTED;
    if (c->kv_bs < TILE || c->kv_bs > 256 || c->kv_bs % TILE != 0) return KQ8_ERR_UNSUPPORTED;
    if (c->num_kv_heads < 1 || c->num_pages < 1) return KQ8_ERR_INVALID_ARG;
    if (!c->k || !c->v || !c->kscale || !c->vscale) return KQ8_ERR_INVALID_ARG;
    if (!aligned(c->k, 16) || !aligned(c->v, 16) || !aligned(c->kscale, 16) ||
        !aligned(c->vscale, 16))
        return KQ8_ERR_INVALID_ARG;
    return KQ8_OK;
}

}  // namespace kq8

using namespace kq8;

extern "C" {

int kq8_version(void) { return 10000; }

const char* kq8_strerror(int code) {
    switch (code) {
        case KQ8_OK: return "ok";
        case KQ8_ERR_INVALID_ARG: return "invalid argument";
        case KQ8_ERR_UNSUPPORTED: return "unsupported shape";
        case KQ8_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case KQ8_ERR_CUDA: return "CUDA error";
        default: return "unknown error";
    }
}

int kq8_append_kv(const kq8_cache_t* cache, const float* k, const float* v, const int32_t* slot,
                  int32_t T, uint32_t* status, kq8_stream_t stream) {
    int rc = check_cache_args(cache);
    if (rc) return rc;
    if (T < 0) return KQ8_ERR_INVALID_ARG;
    if (T == 0) return KQ8_OK;
    if (!k || !v || !slot || !aligned(k, 16) || !aligned(v, 16)) return KQ8_ERR_INVALID_ARG;
    if (status && !aligned(status, 4)) return KQ8_ERR_INVALID_ARG;
    return launch_append(*cache, k, v, slot, T, status, (cudaStream_t)stream);
}

int kq8_append_kv_q4(const kq8_cache_t* cache, const float* k, const float* v,
                     const int32_t* slot, int32_t T, uint32_t* status, kq8_stream_t stream) {
    int rc = check_cache_args(cache);
    if (rc) return rc;
    if (T < 0) return KQ8_ERR_INVALID_ARG;
    if (T == 0) return KQ8_OK;
    if (!k || !v || !slot || !aligned(k, 16) || !aligned(v, 16)) return KQ8_ERR_INVALID_ARG;
    if (status && !aligned(status, 4)) return KQ8_ERR_INVALID_ARG;
    return launch_append_q4(*cache, k, v, slot, T, status, (cudaStream_t)stream);
}

int kq8_decode_attn_q4(float* out, const float* q, const kq8_cache_t* cache,
                       const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                       int32_t max_seq_len, int32_t B, int32_t nq, float scale, void* workspace,
                       size_t workspace_bytes, kq8_stream_t stream) {
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    const int nkv = cache->num_kv_heads;
    const Plan plan = plan_exact(B, nq, nkv, max_seq_len);
    rc = check_ws(workspace, workspace_bytes, plan.total);
    if (rc) return rc;
    if (B == 0) return KQ8_OK;
    AttnParams p = attn_params(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq,
                               scale, plan, workspace);
    rc = set_vmap(p, true);
    if (rc) return rc;
    return launch_attn_q4(p, nq / nkv, B, nkv, (cudaStream_t)stream);
}

size_t kq8_decode_workspace_bytes(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len) {
    if (B < 0 || nq < 1 || nkv < 1 || max_seq_len < 0) return 0;
    return plan_exact(B, nq, nkv, max_seq_len).total;
}

int kq8_decode_plan(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len, int32_t* chunk_tiles,
                    int32_t* num_chunks) {
    if (B < 0 || nq < 1 || nkv < 1 || max_seq_len < 0 || !chunk_tiles || !num_chunks)
        return KQ8_ERR_INVALID_ARG;
    const Plan p = plan_exact(B, nq, nkv, max_seq_len);
    *chunk_tiles = p.chunk_tiles;
    *num_chunks = p.num_chunks;
    return KQ8_OK;
}

size_t kq8_sparse_decode_workspace_bytes(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len,
                                         int32_t block, int32_t topk) {
    if (B < 0 || nq < 1 || nkv < 1 || max_seq_len < 0 || block < TILE || block % TILE || topk < 1)
        return 0;
    return plan_sparse(B, nq, nkv, max_seq_len, block, topk).total;
}

int kq8_sparse_decode_plan(int32_t B, int32_t nq, int32_t nkv, int32_t max_seq_len, int32_t block,
                           int32_t topk, int32_t* chunk_tiles, int32_t* num_chunks) {
    if (B < 0 || nq < 1 || nkv < 1 || nq % nkv || max_seq_len < 0 || block < TILE ||
        block % TILE || topk < 1 || !chunk_tiles || !num_chunks)
        return KQ8_ERR_INVALID_ARG;
    const Plan p = plan_sparse(B, nq, nkv, max_seq_len, block, topk);
    *chunk_tiles = p.chunk_tiles;
    *num_chunks = p.num_chunks;
    return KQ8_OK;
}

int kq8_workspace_init(void* workspace, size_t workspace_bytes, kq8_stream_t stream) {
    if (check_ws(workspace, workspace_bytes, STATUS_BYTES)) return KQ8_ERR_WORKSPACE;
    const size_t n = workspace_bytes < HEADER_BYTES ? workspace_bytes : HEADER_BYTES;
    return cudaMemsetAsync(workspace, 0, n, (cudaStream_t)stream) == cudaSuccess
               ? KQ8_OK
               : KQ8_ERR_CUDA;
}

int kq8_decode_attn(float* out, const float* q, const kq8_cache_t* cache,
                    const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                    int32_t max_seq_len, int32_t B, int32_t nq, float scale, void* workspace,
                    size_t workspace_bytes, kq8_stream_t stream) {
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    const int nkv = cache->num_kv_heads;
    const Plan plan = plan_exact(B, nq, nkv, max_seq_len);
    rc = check_ws(workspace, workspace_bytes, plan.total);
    if (rc) return rc;
    if (B == 0) return KQ8_OK;
    AttnParams p = attn_params(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq,
                               scale, plan, workspace);
    rc = set_vmap(p);
    if (rc) return rc;
    return launch_attn(p, nq / nkv, false, B, nkv, (cudaStream_t)stream);
}

int kq8_sparse_decode_attn(float* out, const float* q, const kq8_cache_t* cache,
                           const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t B, int32_t nq, float scale, int32_t block,
                           int32_t topk, int32_t probe, int32_t* sel_blocks, void* workspace,
                           size_t workspace_bytes, kq8_stream_t stream) {
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    if (block < TILE || block % TILE != 0 || topk < 1 || probe < 1 || probe > block)
        return KQ8_ERR_UNSUPPORTED;
    if (sel_blocks && !aligned(sel_blocks, 4)) return KQ8_ERR_INVALID_ARG;
    const Plan plan = plan_sparse(B, nq, cache->num_kv_heads, max_seq_len, block, topk);
    rc = check_ws(workspace, workspace_bytes, plan.total);
    if (rc) return rc;
    if (B == 0) return KQ8_OK;
    return run_sparse(out, q, cache, page_table, max_pages, seq_lens, nullptr, max_seq_len, B, nq,
                      scale, block, topk, probe, sel_blocks, plan, workspace, (cudaStream_t)stream);
}

int kq8_sparse_decode_attn_shared(float* out, const float* q, const kq8_cache_t* cache,
                                  const int32_t* page_table, int32_t max_pages,
                                  const int32_t* seq_lens, int32_t max_seq_len, int32_t B,
                                  int32_t nq, float scale, int32_t block, int32_t topk,
                                  int32_t probe, int32_t* sel_blocks, void* workspace,
                                  size_t workspace_bytes, kq8_stream_t stream) {
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    if (block < TILE || block % TILE != 0 || topk < 1 || probe < 1 || probe > block)
        return KQ8_ERR_UNSUPPORTED;
    if (sel_blocks && !aligned(sel_blocks, 4)) return KQ8_ERR_INVALID_ARG;
    const Plan plan = plan_sparse(B, nq, cache->num_kv_heads, max_seq_len, block, topk);
    rc = check_ws(workspace, workspace_bytes, plan.total);
    if (rc) return rc;
    if (B == 0) return KQ8_OK;
    return run_sparse(out, q, cache, page_table, max_pages, seq_lens, nullptr, max_seq_len, B, nq,
                      scale, block, topk, probe, sel_blocks, plan, workspace, (cudaStream_t)stream,
                      true);
}

size_t kq8_sparse_prefill_workspace_bytes(int32_t total_q, int32_t nq, int32_t nkv,
                                          int32_t max_seq_len, int32_t block, int32_t topk) {
    const size_t base = kq8_sparse_decode_workspace_bytes(total_q, nq, nkv, max_seq_len, block, topk);
    if (base == 0) return 0;
    return base + align_up(2 * sizeof(int32_t) * (size_t)total_q, WS_ALIGN);
}

int kq8_sparse_prefill_attn(float* out, const float* q, int32_t total_q, const kq8_cache_t* cache,
                            const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                            const int32_t* q_offsets, int32_t max_seq_len, int32_t max_q_len,
                            int32_t B, int32_t nq, float scale, int32_t block, int32_t topk,
                            int32_t probe, int32_t* sel_blocks, void* workspace,
                            size_t workspace_bytes, kq8_stream_t stream) {
    // the rows are the packed queries: total_q plays the decode batch
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, total_q, nq);
    if (rc) return rc;
    if (B < 0 || B > 65535 || max_q_len < 0 || max_q_len > max_seq_len) return KQ8_ERR_INVALID_ARG;
    if (block < TILE || block % TILE != 0 || topk < 1 || probe < 1 || probe > block)
        return KQ8_ERR_UNSUPPORTED;
    if (sel_blocks && !aligned(sel_blocks, 4)) return KQ8_ERR_INVALID_ARG;
    const Plan plan = plan_sparse(total_q, nq, cache->num_kv_heads, max_seq_len, block, topk);
    rc = check_ws(workspace, workspace_bytes,
                  kq8_sparse_prefill_workspace_bytes(total_q, nq, cache->num_kv_heads,
                                                     max_seq_len, block, topk));
    if (rc) return rc;
    if (total_q == 0) return KQ8_OK;
    if (B > 0 && !q_offsets) return KQ8_ERR_INVALID_ARG;
    int32_t* row_seq = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + plan.total);
    int32_t* row_len = row_seq + total_q;
    cudaStream_t s = (cudaStream_t)stream;
    rc = launch_prefill_rows(row_seq, row_len, q_offsets, seq_lens, B, total_q, max_seq_len,
                             max_q_len, s);
    if (rc) return rc;
    return run_sparse(out, q, cache, page_table, max_pages, row_len, row_seq, max_seq_len, total_q,
                      nq, scale, block, topk, probe, sel_blocks, plan, workspace, s);
}

int kq8_state_reset(float* state_acc, float* state_ms, int32_t rows, kq8_stream_t stream) {
    if (rows < 0 || (rows > 0 && (!state_acc || !state_ms || !aligned(state_acc, 16) ||
                                  !aligned(state_ms, 8))))
        return KQ8_ERR_INVALID_ARG;
    return launch_state_reset(state_acc, reinterpret_cast<float2*>(state_ms), rows,
                              (cudaStream_t)stream);
}

int kq8_decode_attn_update(float* state_acc, float* state_ms, const float* q,
                           const kq8_cache_t* cache, const int32_t* page_table, int32_t max_pages,
                           const int32_t* seq_begin, const int32_t* seq_end, int32_t max_seq_len,
                           int32_t max_range_len, int32_t B, int32_t nq, float scale,
                           void* workspace, size_t workspace_bytes, kq8_stream_t stream) {
    int rc = check_decode(state_acc, q, cache, page_table, max_pages, seq_end, max_seq_len, B, nq);
    if (rc) return rc;
    if (B > 0 && (!state_ms || !aligned(state_ms, 8))) return KQ8_ERR_INVALID_ARG;
    if (max_range_len < 0) return KQ8_ERR_INVALID_ARG;
    const int nkv = cache->num_kv_heads;
    const Plan plan = plan_exact_range(B, nq, nkv, max_seq_len, max_range_len);
    rc = check_ws(workspace, workspace_bytes, plan.total);
    if (rc) return rc;
    if (B == 0) return KQ8_OK;
    AttnParams p = attn_params(nullptr, q, cache, page_table, max_pages, seq_end, max_seq_len, B,
                               nq, scale, plan, workspace);
    p.seq_begin = seq_begin;
    p.state_acc = state_acc;
    p.state_ms = reinterpret_cast<float2*>(state_ms);
    rc = set_vmap(p);
    if (rc) return rc;
    return launch_attn(p, nq / nkv, false, B, nkv, (cudaStream_t)stream);
}

int kq8_state_finalize(float* out, const float* state_acc, const float* state_ms, int32_t rows,
                       kq8_stream_t stream) {
    if (rows < 0 || (rows > 0 && (!out || !state_acc || !state_ms || !aligned(state_ms, 8))))
        return KQ8_ERR_INVALID_ARG;
    return launch_state_finalize(out, state_acc, reinterpret_cast<const float2*>(state_ms), rows,
                                 (cudaStream_t)stream);
}

int kq8_state_merge(float* state_acc, float* state_ms, const float* part_acc,
                    const float* part_ms, int32_t parts, int32_t rows, kq8_stream_t stream) {
    if (rows < 0 || parts < 0) return KQ8_ERR_INVALID_ARG;
    if (rows == 0 || parts == 0) return KQ8_OK;
    if (!state_acc || !state_ms || !part_acc || !part_ms || !aligned(state_ms, 8) ||
        !aligned(part_ms, 8))
        return KQ8_ERR_INVALID_ARG;
    return launch_state_merge(state_acc, reinterpret_cast<float2*>(state_ms), part_acc,
                              reinterpret_cast<const float2*>(part_ms), parts, rows,
                              (cudaStream_t)stream);
}

int kq8_read_status(void* status_word, uint32_t* status, kq8_stream_t stream) {
    if (!status_word || !status || !aligned(status_word, 4)) return KQ8_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KQ8_ERR_CUDA;
    if (cudaMemcpy(status, status_word, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess)
        return KQ8_ERR_CUDA;
    if (cudaMemsetAsync(status_word, 0, sizeof(uint32_t), s) != cudaSuccess) return KQ8_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? KQ8_OK : KQ8_ERR_CUDA;
}

int kq8_debug_quantize_q(int8_t* qi, float* qsc, const float* q, int32_t rows, int32_t hd,
                         kq8_stream_t stream) {
    if (hd != HD) return KQ8_ERR_UNSUPPORTED;
    if (rows < 0 || (rows > 0 && (!qi || !qsc || !q || !aligned(q, 16) || !aligned(qi, 4))))
        return KQ8_ERR_INVALID_ARG;
    return launch_debug_quantize(qi, qsc, q, rows, (cudaStream_t)stream);
}

int kq8_debug_block_dots(int32_t* dots, const float* q, const kq8_cache_t* cache,
                         const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                         int32_t max_seq_len, int32_t B, int32_t nq, kq8_stream_t stream) {
    int rc = check_decode(reinterpret_cast<float*>(dots), q, cache, page_table, max_pages, seq_lens,
                          max_seq_len, B, nq);
    if (rc) return rc;
    return launch_debug_dots(dots, q, *cache, page_table, max_pages, seq_lens, max_seq_len, B, nq,
                             (cudaStream_t)stream);
}

int kq8_debug_decode_withhold(float* out, const float* q, const kq8_cache_t* cache,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* seq_lens, int32_t max_seq_len, int32_t B, int32_t nq,
                              float scale, void* workspace, size_t workspace_bytes,
                              int32_t withhold_tile, kq8_stream_t stream) {
    if (withhold_tile < 0) return KQ8_ERR_INVALID_ARG;
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    const int nkv = cache->num_kv_heads;
    const Plan plan = plan_exact(B, nq, nkv, max_seq_len);
    rc = check_ws(workspace, workspace_bytes, plan.total);
    if (rc) return rc;
    if (B == 0) return KQ8_OK;
    AttnParams p = attn_params(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq,
                               scale, plan, workspace);
    p.withhold = withhold_tile;
    rc = set_vmap(p);
    if (rc) return rc;
    return launch_attn_withhold(p, nq / nkv, B, nkv, (cudaStream_t)stream);
}

int kq8_debug_probe_scores(float* scores, const float* q, const kq8_cache_t* cache,
                           const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                           int32_t max_seq_len, int32_t B, int32_t nq, float scale, int32_t block,
                           int32_t probe, kq8_stream_t stream) {
    int rc = check_decode(scores, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    if (block < TILE || block % TILE != 0 || probe < 1 || probe > block) return KQ8_ERR_UNSUPPORTED;
    SparseParams sp;
    std::memset(&sp, 0, sizeof(sp));
    sp.q = q;
    sp.cache = *cache;
    sp.page_table = page_table;
    sp.max_pages = max_pages;
    sp.seq_lens = seq_lens;
    sp.max_seq_len = max_seq_len;
    sp.B = B;
    sp.nq = nq;
    sp.scale = scale;
    sp.block = block;
    sp.probe = probe;
    sp.max_nblk = (int)(((int64_t)max_seq_len + block - 1) / block);
    sp.probe_bpc = probe_blocks_per_cta(block, cache->kv_bs);
    set_probe_kmap(sp);
    sp.scores = scores;
    sp.status = nullptr;  // bad page ids are skipped without a status word
    return launch_probe(sp, nq / cache->num_kv_heads, B, cache->num_kv_heads,
                        (cudaStream_t)stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free exact decode.  Some callers may not allocate device memory at
// all: plugins that run inside another runtime's allocator or launch path
// (cudaMalloc there can re-enter that runtime, and it may synchronise the
// device, stalling every other stream), and serving loops that forbid device
// allocation once they have started.  For them, kq8_decode_attn_noalloc uses a
// fixed scratch array compiled into this library instead of a caller-provided
// workspace.  The array lives in a device's global memory from the moment this
// file's module is loaded on it -- with CUDA's default lazy loading, at the
// first use of the array there, i.e. the first call's cudaGetSymbolAddress --
// until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

namespace kq8 {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)KQ8_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[NOALLOC_MAX_DEVICES] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device, with that device current, and cached.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KQ8_ERR_CUDA;
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return KQ8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KQ8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return KQ8_OK;
}

}  // namespace
}  // namespace kq8

extern "C" int kq8_decode_attn_noalloc(float* out, const float* q, const kq8_cache_t* cache,
                                       const int32_t* page_table, int32_t max_pages,
                                       const int32_t* seq_lens, int32_t max_seq_len, int32_t B,
                                       int32_t nq, float scale, kq8_stream_t stream) {
    int rc = check_decode(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq);
    if (rc) return rc;
    const int nkv = cache->num_kv_heads;
    const Plan plan = plan_exact(B, nq, nkv, max_seq_len);
    if (plan.total > NOALLOC_SCRATCH_BYTES) return KQ8_ERR_WORKSPACE;  // sizes beyond the array
    if (B == 0) return KQ8_OK;
    void* ws = nullptr;
    rc = noalloc_scratch(&ws);
    if (rc) return rc;
    // Only the chunk counters must start at zero: a __device__ array is zeroed
    // when the library loads and every call leaves its counters at zero again.
    // Partials are written before they are read, and the status word only
    // collects error bits that this entry point does not report.
    AttnParams p = attn_params(out, q, cache, page_table, max_pages, seq_lens, max_seq_len, B, nq,
                               scale, plan, ws);
    rc = set_vmap(p);
    if (rc) return rc;
    return launch_attn(p, nq / nkv, false, B, nkv, (cudaStream_t)stream);
}
