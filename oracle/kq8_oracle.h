/*
 * kq8_oracle.h -- declarations of the plain CPU oracle (test infrastructure only;
 * see kq8_oracle.c for the definitions, their sources and the readings taken).
 */
#ifndef KQ8_ORACLE_H
#define KQ8_ORACLE_H

#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KQ8O_MAX_HD 512

void kq8o_kv_quantize_row(const float* v, int hd, int8_t* q, float* stored_max);
void kq8o_kv_quantize_rows(const float* x, int64_t T, int nkv, int hd, int8_t* codes, float* maxima);
float kq8o_dequant(int8_t q, float stored_max);
void kq8o_quantize_q(const float* q, int hd, int8_t* qi, float* qsc);
void kq8o_block_dots(const int8_t* qi, const int8_t* krow, int hd, int32_t* dots);
float kq8o_score(const int32_t* dots, const float* qsc, int nblk, float kscale_stored, float scale);

void kq8o_attn_single_q(float* out, const float* q, int8_t* const* k_blocks,
                        int8_t* const* v_blocks, const float* kscale, const float* vscale,
                        int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                        float scale, const int32_t* tokens, int n_tokens, float* m_trace,
                        int* n_visited);
void kq8o_stream_reset(float* M, float* S, float* acc, int hd);
void kq8o_attn_stream(float* M_io, float* S_io, float* acc, const float* q, int8_t* const* k_blocks,
                      int8_t* const* v_blocks, const float* kscale, const float* vscale,
                      int t_begin, int t_end, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                      float scale);
void kq8o_stream_output(float* out, float S, const float* acc, int hd);
void kq8o_attn_two_pass_f64(double* out, const float* q, int8_t* const* k_blocks,
                            int8_t* const* v_blocks, const float* kscale, const float* vscale,
                            int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                            float scale, const int32_t* tokens, int n_tokens);
void kq8o_attn_ref_f64(double* out, const float* q, const float* K, const float* V, int n, int hd,
                       double scale);
void kq8o_attn_exact_sum(double* out, const float* q, int8_t* const* k_blocks,
                         int8_t* const* v_blocks, const float* kscale, const float* vscale,
                         int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                         float scale);

void kq8o_probe_block_scores(float* block_scores, const float* q, int8_t* const* k_blocks,
                             const float* kscale, int seq_len, int kv_dim, int kv_bs, int nkv,
                             int kh_off, int hd, float scale, int block, int probe);
int kq8o_topk_blocks(int32_t* sel, const float* scores, int nblk, int k);
int kq8o_sparse_attn_head(float* out, const float* q, int8_t* const* k_blocks,
                          int8_t* const* v_blocks, const float* kscale, const float* vscale,
                          int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                          float scale, int block, int topk, int probe, int32_t* sel_out);

int kq8o_decode_batch(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                      const float* kscale, const float* vscale, const int64_t* row_offset,
                      const int32_t* seq_lens, int B, int nq, int nkv, int hd, int kv_bs,
                      float scale, int sparse, int block, int topk, int probe, int32_t* sel_out,
                      int nthreads);
int kq8o_prefill_batch(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                       const float* kscale, const float* vscale, const int64_t* row_offset,
                       const int32_t* seq_lens, const int32_t* q_off, int B, int nq, int nkv,
                       int hd, int kv_bs, float scale, int sparse, int block, int topk, int probe,
                       int32_t* sel_out, int nthreads);
void kq8o_kv_quantize_row_q4(const float* v, int hd, int8_t* q, float* stored_max);
void kq8o_kv_quantize_rows_q4(const float* x, int64_t T, int nkv, int hd, int8_t* codes,
                              float* maxima);
void kq8o_attn_single_q_q4(float* out, const float* q, int8_t* const* k_blocks,
                           int8_t* const* v_blocks, const float* kscale, const float* vscale,
                           int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                           float scale);
int kq8o_decode_batch_q4(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                         const float* kscale, const float* vscale, const int64_t* row_offset,
                         const int32_t* seq_lens, int B, int nq, int nkv, int hd, int kv_bs,
                         float scale, int nthreads);
int kq8o_sparse_attn_group(float* out, const float* q, int G, int8_t* const* k_blocks,
                           int8_t* const* v_blocks, const float* kscale, const float* vscale,
                           int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                           float scale, int block, int topk, int probe, int32_t* sel_out);
int kq8o_decode_batch_shared(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                             const float* kscale, const float* vscale, const int64_t* row_offset,
                             const int32_t* seq_lens, int B, int nq, int nkv, int hd, int kv_bs,
                             float scale, int block, int topk, int probe, int32_t* sel_out,
                             int nthreads);
int kq8o_has_openmp(void);

#endif
