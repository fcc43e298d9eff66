// kq8_internal.h -- launchers shared between the libkq8 translation units.
#pragma once

#include <cuda_runtime.h>

#include "kq8.h"

namespace kq8 {

struct AttnParams;
struct SparseParams;
struct PrefillParams;

// Shared argument checks of a kq8_cache_t (head_dim 128, kv_bs a multiple of
// 32 up to 256, 16-byte aligned arrays); returns a KQ8_ERR_* code or KQ8_OK.
int check_cache_args(const kq8_cache_t* c);

int launch_append(const kq8_cache_t& c, const float* k, const float* v, const int32_t* slot,
                  int32_t T, uint32_t* status, cudaStream_t stream);
int launch_append_q4(const kq8_cache_t& c, const float* k, const float* v, const int32_t* slot,
                     int32_t T, uint32_t* status, cudaStream_t stream);
int launch_debug_quantize(int8_t* qi, float* qsc, const float* q, int32_t rows, cudaStream_t s);
int launch_debug_dots(int32_t* dots, const float* q, const kq8_cache_t& c,
                      const int32_t* page_table, int32_t max_pages, const int32_t* seq_lens,
                      int32_t max_seq_len, int32_t B, int32_t nq, cudaStream_t s);

// Attention over KV chunks (+ the merge when any sequence spans > 1 chunk).
int launch_attn(const AttnParams& p, int G, bool sparse, int B, int nkv, cudaStream_t s);
int launch_attn_q4(const AttnParams& p, int G, int B, int nkv, cudaStream_t s);
int launch_attn_withhold(const AttnParams& p, int G, int B, int nkv, cudaStream_t s);
int launch_probe(const SparseParams& p, int G, int B, int nkv, cudaStream_t s);
int launch_state_reset(float* acc, float2* ms, int rows, cudaStream_t s);
int launch_state_finalize(float* out, const float* acc, const float2* ms, int rows, cudaStream_t s);
int launch_state_merge(float* acc, float2* ms, const float* pacc, const float2* pms, int parts,
                       int rows, cudaStream_t s);
int probe_blocks_per_cta(int block, int kv_bs);
int launch_prefill(const PrefillParams& p, int G, int nkv, cudaStream_t s);
int launch_prefill_rows(int32_t* row_seq, int32_t* row_len, const int32_t* q_off,
                        const int32_t* seq_lens, int32_t B, int32_t total_q, int32_t max_seq_len,
                        int32_t max_q_len, cudaStream_t s);
int launch_topk(const SparseParams& p, int G, int B, int nkv, cudaStream_t s);

}  // namespace kq8
