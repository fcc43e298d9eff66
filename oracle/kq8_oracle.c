/*
 * kq8_oracle.c -- plain, slow CPU oracle for q8-KV single-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference leg of bench.py may build, load or call this file.
 * The product (the CUDA library under query_decode_attention_gb300/) never
 * links, imports or executes it, and shares no code, header, table or
 * constant with it.
 *
 * Sources (the three web pages this method is described on):
 *   [9-2]  "0.8MB 跑通 Qwen | 第 9-2 篇：推理引擎的 flash_attn_single_q_q8_neon
 *           ——单 q 单遍扫全 KV" (single q, one pass over all KV)
 *           §1 why decode attention can be one pass; §2 code walkthrough
 *           (signature, segment 1 = Q quantization, segment 2 = online softmax,
 *           segment 3 = final normalisation); §3 the two-pass alternative.
 *   [10-1] "长上下文为什么必须稀疏" (article 10-1, why long context must be
 *           sparse) §1 block-sparse cost model, §2 sparse knobs and gates.
 *   [9-3]  "q8 KV 精度对照实验" (article 9-3, q8 KV precision comparison)
 *           §1 experiment design, §2 the write-path quantization rule,
 *           §3 measured fp32-KV vs q8-KV output difference.
 *
 * Arithmetic is IEEE fp32 exactly as the pages write it (the pages fix fp32);
 * the file must be compiled with -ffp-contract=off so that no multiply-add is
 * fused.  The fp64 functions are brute-force references used to pin the fp32
 * ones.  Every reading of a point the pages leave open is marked READING.
 *
 * Data structure (as on [9-2] §2 signature and segment 2): a layer's K cache is
 * an array of block pointers; block j holds kv_bs tokens, each a row of
 * kv_dim = nkv*hd int8 values, token-major; head kh starts at column
 * kh_off = kh*hd.  kscale/vscale are per-(token, head) floats holding the row's
 * max |x|; token t of head kh is at kscale[t*nkv] once the caller has offset
 * the pointer by kh.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kq8_oracle.h"

/* [9-2] §2 segment 1 comment and [9-3] §2: the inverse of 127 as a float
 * constant.  READING: the garbled "KVQ_SCALE ... 的逆" on [9-3] §2 and the
 * "KVQ_INV = 1/127" of [9-2] name this same constant. */
static const float KVQ_INV = 1.0f / 127.0f;

/* q4 KV ([10-1] §2 names the --kv-q4 switch and excludes it from the sparse
 * path; no page gives its format).  READING: the q8 rule with 7 in place of
 * 127 -- stored max m, step m * (1/7), codes roundf(x / step) clamped to
 * [-7, 7], readers multiply the stored max by 1/7; Q stays int8 ([9-2] §2). */
static const float Q4_INV = 1.0f / 7.0f;

/* READING: the online-softmax running max starts at -1e9 ([9-2] §2 seg. 2). */
static const float M_INIT = -1e9f;

static float clampf(float x, float lo, float hi) {
    if (x < lo) return lo;
    if (x > hi) return hi;
    return x;
}

/* ------------------------------------------------------------------------ */
/* Write path: kv_quantize_per_head ([9-3] §2).                              */
/* For one (token, head) row of hd floats: max_abs over the row, the step is  */
/* max_abs/127, q = round(v/step) clamped to [-127, 127].  The stored scale is */
/* max_abs itself; readers multiply by KVQ_INV ([9-2] §2 segment 2, "ks =     */
/* kscale[t*nkv] * KVQ_INV").                                                 */
/* READING: storing max_abs and multiplying by KVQ_INV on both sides satisfies */
/* both "scale = max_abs/127" ([9-3] §2) and the read side of [9-2].          */
/* READING: "round" is C roundf (half away from zero).                       */
/* READING (pages silent): an all-zero row stores 0 and all-zero codes.      */
/* ------------------------------------------------------------------------ */
void kq8o_kv_quantize_row(const float* v, int hd, int8_t* q, float* stored_max) {
    float m = 0.0f;
    for (int i = 0; i < hd; i++) {
        float a = fabsf(v[i]);
        if (a > m) m = a;
    }
    *stored_max = m;
    if (m == 0.0f) {
        for (int i = 0; i < hd; i++) q[i] = 0;
        return;
    }
    float d = m * KVQ_INV;
    for (int i = 0; i < hd; i++) {
        float r = roundf(v[i] / d);
        r = clampf(r, -127.0f, 127.0f);
        q[i] = (int8_t)(int)r;
    }
}

/* q4 write path: the same steps with the q4 step and clamp (reading above). */
void kq8o_kv_quantize_row_q4(const float* v, int hd, int8_t* q, float* stored_max) {
    float m = 0.0f;
    for (int i = 0; i < hd; i++) {
        float a = fabsf(v[i]);
        if (a > m) m = a;
    }
    *stored_max = m;
    if (m == 0.0f) {
        for (int i = 0; i < hd; i++) q[i] = 0;
        return;
    }
    float d = m * Q4_INV;
    for (int i = 0; i < hd; i++) {
        float r = roundf(v[i] / d);
        r = clampf(r, -7.0f, 7.0f);
        q[i] = (int8_t)(int)r;
    }
}

/* Dequantised value of one code: q * (stored_max * KVQ_INV) ([9-3] §2,
 * "v' = q x scale"). */
float kq8o_dequant(int8_t q, float stored_max) {
    float d = stored_max * KVQ_INV;
    return (float)q * d;
}

/* ------------------------------------------------------------------------ */
/* Q quantization once per call ([9-2] §2 segment 1): per block of 32         */
/* elements, qm = max |x| folded from 0 with fmaxf; qm < 1e-6 -> 1;           */
/* qsc = qm * KVQ_INV; iq = 127 / qm; qi = (int8)clamp(x * iq, -128, 127).    */
/* READING: the printed C cast truncates toward zero; that literal reading is */
/* kept (the "same structure as Q8_0" remark does not override the code).    */
/* ------------------------------------------------------------------------ */
void kq8o_quantize_q(const float* q, int hd, int8_t* qi, float* qsc) {
    int nblk = hd / 32;
    for (int b = 0; b < nblk; b++) {
        const float* qb = q + b * 32;
        float qm = 0.0f;
        for (int i = 0; i < 32; i++) qm = fmaxf(qm, fabsf(qb[i]));
        if (qm < 1e-6f) qm = 1.0f;
        qsc[b] = qm * KVQ_INV;
        float iq = 127.0f / qm;
        for (int i = 0; i < 32; i++) {
            float x = clampf(qb[i] * iq, -128.0f, 127.0f);
            qi[b * 32 + i] = (int8_t)(int)x; /* C conversion: truncation */
        }
    }
}

/* int32 dot of each 32-element block of qi with the K row ([9-2] §2 seg. 2,
 * "each 32-block one int32 accumulation"). */
void kq8o_block_dots(const int8_t* qi, const int8_t* krow, int hd, int32_t* dots) {
    int nblk = hd / 32;
    for (int b = 0; b < nblk; b++) {
        int32_t acc = 0;
        for (int i = 0; i < 32; i++) acc += (int32_t)qi[b * 32 + i] * (int32_t)krow[b * 32 + i];
        dots[b] = acc;
    }
}

/* Score of one token ([9-2] §2 segment 2 and its point 1): s starts at 0,
 * s += dot_b * qsc[b] block by block in order, then s = s * ks * scale with
 * ks = kscale * KVQ_INV.  Evaluated left to right in fp32. */
static float score_steps(const int32_t* dots, const float* qsc, int nblk, float kscale_stored,
                         float scale, float kv_inv) {
    float ks = kscale_stored * kv_inv;
    float s = 0.0f;
    for (int b = 0; b < nblk; b++) s += (float)dots[b] * qsc[b];
    s = s * ks * scale;
    return s;
}

float kq8o_score(const int32_t* dots, const float* qsc, int nblk, float kscale_stored, float scale) {
    float ks = kscale_stored * KVQ_INV;
    float s = 0.0f;
    for (int b = 0; b < nblk; b++) s += (float)dots[b] * qsc[b];
    s = s * ks * scale;
    return s;
}

static const int8_t* row_ptr(int8_t* const* blocks, int t, int kv_bs, int kv_dim, int kh_off) {
    /* [9-2] §2 segment 2: block t / kv_bs, row t % kv_bs, column kh_off. */
    return blocks[t / kv_bs] + (size_t)(t % kv_bs) * (size_t)kv_dim + kh_off;
}

/* ------------------------------------------------------------------------ */
/* flash_attn_single_q_q8: one query head over a list of tokens of one KV    */
/* head, in one pass ([9-2] §1 and §2).  With tokens == NULL the list is      */
/* 0..seq_len-1, i.e. the exact kernel of the page.                          */
/*   per token: score (above); if s > M: S *= expf(M - s), acc *= that same   */
/*   factor, M = s, w = 1; else w = expf(s - M).  S += w;                     */
/*   acc[i] += (float)v[i] * (w * vs), vs = vscale * KVQ_INV ([9-2] seg. 2).  */
/*   end: out[i] = acc[i] / S, one divide per output ([9-2] segment 3).      */
/* READING: the elided new-max branch uses w = 1 (= expf(s - M) with M = s);  */
/* segment 3's "together with the final scale handling" applies nothing else. */
/* READING (pages silent): an empty token list gives out = 0.                */
/* m_trace (optional, [n]) receives M after each token; *n_visited (optional) */
/* the number of tokens the loop visited (the [9-2] §4 debug invariants).     */
/* ------------------------------------------------------------------------ */
static void attn_one_pass(float* out, const float* q, int8_t* const* k_blocks,
                          int8_t* const* v_blocks, const float* kscale, const float* vscale,
                          int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                          float scale, const int32_t* tokens, int n_tokens, float* m_trace,
                          int* n_visited, float kv_inv);

void kq8o_attn_single_q(float* out, const float* q,
                        int8_t* const* k_blocks, int8_t* const* v_blocks,
                        const float* kscale, const float* vscale,
                        int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                        float scale, const int32_t* tokens, int n_tokens,
                        float* m_trace, int* n_visited) {
    attn_one_pass(out, q, k_blocks, v_blocks, kscale, vscale, seq_len, kv_dim, kv_bs, nkv, kh_off,
                  hd, scale, tokens, n_tokens, m_trace, n_visited, KVQ_INV);
}

/* The same one pass over a q4 cache: codes in [-7, 7] held as int8, scales
 * read with 1/7 (reading above). */
void kq8o_attn_single_q_q4(float* out, const float* q, int8_t* const* k_blocks,
                           int8_t* const* v_blocks, const float* kscale, const float* vscale,
                           int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                           float scale) {
    attn_one_pass(out, q, k_blocks, v_blocks, kscale, vscale, seq_len, kv_dim, kv_bs, nkv, kh_off,
                  hd, scale, NULL, 0, NULL, NULL, Q4_INV);
}

static void attn_one_pass(float* out, const float* q, int8_t* const* k_blocks,
                          int8_t* const* v_blocks, const float* kscale, const float* vscale,
                          int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                          float scale, const int32_t* tokens, int n_tokens, float* m_trace,
                          int* n_visited, float kv_inv) {
    int nblk = hd / 32;
    int8_t qi[KQ8O_MAX_HD];
    float qsc[KQ8O_MAX_HD / 32];
    float acc[KQ8O_MAX_HD];
    int32_t dots[KQ8O_MAX_HD / 32];

    kq8o_quantize_q(q, hd, qi, qsc); /* once per call ([9-2] §2 seg. 1) */

    int n = tokens ? n_tokens : seq_len;
    for (int i = 0; i < hd; i++) acc[i] = 0.0f;
    float M = M_INIT, S = 0.0f;
    int visited = 0;
    for (int j = 0; j < n; j++) {
        int t = tokens ? tokens[j] : j;
        const int8_t* kt = row_ptr(k_blocks, t, kv_bs, kv_dim, kh_off);
        const int8_t* vt = row_ptr(v_blocks, t, kv_bs, kv_dim, kh_off);
        kq8o_block_dots(qi, kt, hd, dots);
        float s = score_steps(dots, qsc, nblk, kscale[(size_t)t * nkv], scale, kv_inv);
        float w;
        if (s > M) {
            float c = expf(M - s);
            S *= c;
            for (int i = 0; i < hd; i++) acc[i] *= c;
            M = s;
            w = 1.0f;
        } else {
            w = expf(s - M);
        }
        S += w;
        float vs = vscale[(size_t)t * nkv] * kv_inv;
        float pv = w * vs;
        for (int i = 0; i < hd; i++) acc[i] += (float)vt[i] * pv;
        if (m_trace) m_trace[j] = M;
        visited++;
    }
    if (n_visited) *n_visited = visited;
    for (int i = 0; i < hd; i++) out[i] = (n > 0) ? acc[i] / S : 0.0f;
}

/* ------------------------------------------------------------------------ */
/* Streaming form ([9-2] §3: the one-pass kernel "can compute while KV blocks */
/* arrive one by one", the two-pass one cannot).  The running state (M, S,    */
/* acc[hd]) of the loop above is kept by the caller between calls; one call   */
/* continues the loop over tokens [t_begin, t_end) exactly as the one-pass    */
/* kernel would, so feeding a sequence in pieces reproduces the one-call      */
/* result bit for bit.  A fresh state is M = -1e9, S = 0, acc = 0; the output */
/* is acc / S (0 for an empty state), the single divide of [9-2] segment 3.   */
/* ------------------------------------------------------------------------ */
void kq8o_stream_reset(float* M, float* S, float* acc, int hd) {
    *M = M_INIT;
    *S = 0.0f;
    for (int i = 0; i < hd; i++) acc[i] = 0.0f;
}

void kq8o_attn_stream(float* M_io, float* S_io, float* acc, const float* q,
                      int8_t* const* k_blocks, int8_t* const* v_blocks,
                      const float* kscale, const float* vscale, int t_begin, int t_end,
                      int kv_dim, int kv_bs, int nkv, int kh_off, int hd, float scale) {
    int nblk = hd / 32;
    int8_t qi[KQ8O_MAX_HD];
    float qsc[KQ8O_MAX_HD / 32];
    int32_t dots[KQ8O_MAX_HD / 32];
    kq8o_quantize_q(q, hd, qi, qsc);
    float M = *M_io, S = *S_io;
    for (int t = t_begin; t < t_end; t++) {
        const int8_t* kt = row_ptr(k_blocks, t, kv_bs, kv_dim, kh_off);
        const int8_t* vt = row_ptr(v_blocks, t, kv_bs, kv_dim, kh_off);
        kq8o_block_dots(qi, kt, hd, dots);
        float s = kq8o_score(dots, qsc, nblk, kscale[(size_t)t * nkv], scale);
        float w;
        if (s > M) {
            float c = expf(M - s);
            S *= c;
            for (int i = 0; i < hd; i++) acc[i] *= c;
            M = s;
            w = 1.0f;
        } else {
            w = expf(s - M);
        }
        S += w;
        float vs = vscale[(size_t)t * nkv] * KVQ_INV;
        float pv = w * vs;
        for (int i = 0; i < hd; i++) acc[i] += (float)vt[i] * pv;
    }
    *M_io = M;
    *S_io = S;
}

void kq8o_stream_output(float* out, float S, const float* acc, int hd) {
    for (int i = 0; i < hd; i++) out[i] = (S > 0.0f) ? acc[i] / S : 0.0f;
}

/* ------------------------------------------------------------------------ */
/* Naive two-pass attention over the same quantised data, in fp64 ([9-2] §3: */
/* store every score, take the max, exponentiate, weight V -- "functionally   */
/* equivalent" to the one-pass kernel).  Q, K and V enter through their codes */
/* and float scales exactly as the one-pass kernel sees them; everything      */
/* after that is double.  This is the brute-force truth for the one pass.     */
/* ------------------------------------------------------------------------ */
void kq8o_attn_two_pass_f64(double* out, const float* q,
                            int8_t* const* k_blocks, int8_t* const* v_blocks,
                            const float* kscale, const float* vscale,
                            int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                            float scale, const int32_t* tokens, int n_tokens) {
    int nblk = hd / 32;
    int8_t qi[KQ8O_MAX_HD];
    float qsc[KQ8O_MAX_HD / 32];
    kq8o_quantize_q(q, hd, qi, qsc);
    int n = tokens ? n_tokens : seq_len;
    for (int i = 0; i < hd; i++) out[i] = 0.0;
    if (n <= 0) return;
    double* sc = (double*)malloc(sizeof(double) * (size_t)n);
    double mx = -INFINITY;
    for (int j = 0; j < n; j++) {
        int t = tokens ? tokens[j] : j;
        const int8_t* kt = row_ptr(k_blocks, t, kv_bs, kv_dim, kh_off);
        double ks = (double)(kscale[(size_t)t * nkv] * KVQ_INV);
        double s = 0.0;
        for (int b = 0; b < nblk; b++) {
            int64_t d = 0;
            for (int i = 0; i < 32; i++) d += (int64_t)qi[b * 32 + i] * (int64_t)kt[b * 32 + i];
            s += (double)d * (double)qsc[b];
        }
        sc[j] = s * ks * (double)scale;
        if (sc[j] > mx) mx = sc[j];
    }
    double den = 0.0;
    for (int j = 0; j < n; j++) {
        sc[j] = exp(sc[j] - mx);
        den += sc[j];
    }
    for (int j = 0; j < n; j++) {
        int t = tokens ? tokens[j] : j;
        const int8_t* vt = row_ptr(v_blocks, t, kv_bs, kv_dim, kh_off);
        double vs = (double)(vscale[(size_t)t * nkv] * KVQ_INV);
        double p = sc[j] / den;
        for (int i = 0; i < hd; i++) out[i] += p * (double)vt[i] * vs;
    }
    free(sc);
}

/* ------------------------------------------------------------------------ */
/* The method's result with exact sums ([9-2] §3: the one pass and the two    */
/* passes are the same computation, so they differ only by rounding).  The    */
/* scores are the method's fp32 scores, formed exactly as segment 2 writes    */
/* them (kq8o_score), and the V steps are its fp32 vscale * KVQ_INV; the      */
/* softmax and the weighted sum of the dequantised V rows then run in fp64, in */
/* two passes.  This is the value the fp32 one-pass loop approximates: its    */
/* own rounding grows with the sequence (many small weights added to a large  */
/* running sum lose their low bits), and over ~10^5 tokens it can exceed      */
/* 1e-4 on an output.                                                          */
/* ------------------------------------------------------------------------ */
void kq8o_attn_exact_sum(double* out, const float* q, int8_t* const* k_blocks,
                         int8_t* const* v_blocks, const float* kscale, const float* vscale,
                         int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                         float scale) {
    int nblk = hd / 32;
    int8_t qi[KQ8O_MAX_HD];
    float qsc[KQ8O_MAX_HD / 32];
    int32_t dots[KQ8O_MAX_HD / 32];
    kq8o_quantize_q(q, hd, qi, qsc);
    for (int i = 0; i < hd; i++) out[i] = 0.0;
    if (seq_len <= 0) return;
    double* w = (double*)malloc(sizeof(double) * (size_t)seq_len);
    double mx = -INFINITY;
    for (int t = 0; t < seq_len; t++) {
        const int8_t* kt = row_ptr(k_blocks, t, kv_bs, kv_dim, kh_off);
        kq8o_block_dots(qi, kt, hd, dots);
        w[t] = (double)kq8o_score(dots, qsc, nblk, kscale[(size_t)t * nkv], scale);
        if (w[t] > mx) mx = w[t];
    }
    double den = 0.0;
    for (int t = 0; t < seq_len; t++) {
        w[t] = exp(w[t] - mx);
        den += w[t];
    }
    for (int t = 0; t < seq_len; t++) {
        const int8_t* vt = row_ptr(v_blocks, t, kv_bs, kv_dim, kh_off);
        const double step = (double)(vscale[(size_t)t * nkv] * KVQ_INV);
        const double p = w[t] / den;
        for (int i = 0; i < hd; i++) out[i] += p * ((double)vt[i] * step);
    }
    free(w);
}

/* ------------------------------------------------------------------------ */
/* Standard attention on float K/V, fp64 inside ([9-3] §1 baseline arm:      */
/* score = Q.K^T * scale, max-subtracted softmax, weighted V).  K and V are   */
/* dense [n][hd].  Used for both arms of the [9-3] experiment (raw fp32 K/V   */
/* and K/V quantised then dequantised).                                       */
/* ------------------------------------------------------------------------ */
void kq8o_attn_ref_f64(double* out, const float* q, const float* K, const float* V,
                       int n, int hd, double scale) {
    for (int i = 0; i < hd; i++) out[i] = 0.0;
    if (n <= 0) return;
    double* sc = (double*)malloc(sizeof(double) * (size_t)n);
    double mx = -INFINITY;
    for (int t = 0; t < n; t++) {
        double s = 0.0;
        for (int i = 0; i < hd; i++) s += (double)q[i] * (double)K[(size_t)t * hd + i];
        sc[t] = s * scale;
        if (sc[t] > mx) mx = sc[t];
    }
    double den = 0.0;
    for (int t = 0; t < n; t++) {
        sc[t] = exp(sc[t] - mx);
        den += sc[t];
    }
    for (int t = 0; t < n; t++) {
        double p = sc[t] / den;
        for (int i = 0; i < hd; i++) out[i] += p * (double)V[(size_t)t * hd + i];
    }
    free(sc);
}

/* ------------------------------------------------------------------------ */
/* Block-sparse decode ([10-1] §1 and §2).  The pages name the knobs          */
/* (block = 32 positions, k = 32 blocks kept per head, probe = 8 samples per  */
/* block, "max-dot fusion") and the gate, but the probe itself is described   */
/* on a page that is not available.  READINGS:                                */
/*  - gate: seq_len <= 2*block -> the exact kernel ([10-1] §2);               */
/*  - nblk = ceil(seq_len / block); probe p of block j sits at token          */
/*    j*block + p*(block/probe) (integer division), kept if < seq_len;        */
/*  - block score = max of the one-pass scores (above) at its probe tokens;   */
/*  - per query head, keep the k highest block scores, ties to the lower      */
/*    block index; k >= nblk keeps every block;                               */
/*  - exact one-pass attention over the kept blocks' tokens, blocks in        */
/*    ascending order, no forced first/last block.                            */
/* ------------------------------------------------------------------------ */
void kq8o_probe_block_scores(float* block_scores, const float* q,
                             int8_t* const* k_blocks, const float* kscale,
                             int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                             float scale, int block, int probe) {
    int nblk_q = hd / 32;
    int8_t qi[KQ8O_MAX_HD];
    float qsc[KQ8O_MAX_HD / 32];
    int32_t dots[KQ8O_MAX_HD / 32];
    kq8o_quantize_q(q, hd, qi, qsc);
    int nb = (seq_len + block - 1) / block;
    int stride = block / probe;
    for (int j = 0; j < nb; j++) {
        float best = -INFINITY;
        for (int p = 0; p < probe; p++) {
            int t = j * block + p * stride;
            if (t >= seq_len) continue;
            const int8_t* kt = row_ptr(k_blocks, t, kv_bs, kv_dim, kh_off);
            kq8o_block_dots(qi, kt, hd, dots);
            float s = kq8o_score(dots, qsc, nblk_q, kscale[(size_t)t * nkv], scale);
            if (s > best) best = s;
        }
        block_scores[j] = best;
    }
}

typedef struct {
    float score;
    int32_t idx;
} scored_t;

static int cmp_desc_score_then_idx(const void* a, const void* b) {
    const scored_t* x = (const scored_t*)a;
    const scored_t* y = (const scored_t*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

static int cmp_int32_asc(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x < y) ? -1 : (x > y);
}

/* Top-k by a full sort: scores descending, equal scores by ascending index;
 * the first k are returned in ascending block order.  Returns their count. */
int kq8o_topk_blocks(int32_t* sel, const float* scores, int nblk, int k) {
    if (nblk <= 0 || k <= 0) return 0;
    scored_t* v = (scored_t*)malloc(sizeof(scored_t) * (size_t)nblk);
    for (int j = 0; j < nblk; j++) {
        v[j].score = scores[j];
        v[j].idx = j;
    }
    qsort(v, (size_t)nblk, sizeof(scored_t), cmp_desc_score_then_idx);
    int m = k < nblk ? k : nblk;
    for (int i = 0; i < m; i++) sel[i] = v[i].idx;
    qsort(sel, (size_t)m, sizeof(int32_t), cmp_int32_asc);
    free(v);
    return m;
}

/* One query head of the block-sparse kernel.  Returns 1 when the sparse path
 * ran, 0 when the gate sent it to the exact kernel.  sel_out (optional, [k])
 * receives the kept blocks in ascending order, -1 padded; it is all -1 when
 * the exact kernel ran. */
int kq8o_sparse_attn_head(float* out, const float* q,
                          int8_t* const* k_blocks, int8_t* const* v_blocks,
                          const float* kscale, const float* vscale,
                          int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                          float scale, int block, int topk, int probe, int32_t* sel_out) {
    if (sel_out)
        for (int i = 0; i < topk; i++) sel_out[i] = -1;
    if (seq_len <= 2 * block) {
        kq8o_attn_single_q(out, q, k_blocks, v_blocks, kscale, vscale, seq_len, kv_dim, kv_bs,
                           nkv, kh_off, hd, scale, NULL, 0, NULL, NULL);
        return 0;
    }
    int nb = (seq_len + block - 1) / block;
    float* bs = (float*)malloc(sizeof(float) * (size_t)nb);
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)(topk < nb ? topk : nb));
    kq8o_probe_block_scores(bs, q, k_blocks, kscale, seq_len, kv_dim, kv_bs, nkv, kh_off, hd,
                            scale, block, probe);
    int m = kq8o_topk_blocks(sel, bs, nb, topk);
    int32_t* toks = (int32_t*)malloc(sizeof(int32_t) * (size_t)m * (size_t)block);
    int nt = 0;
    for (int i = 0; i < m; i++) {
        int j = sel[i];
        for (int t = j * block; t < (j + 1) * block && t < seq_len; t++) toks[nt++] = t;
        if (sel_out) sel_out[i] = j;
    }
    kq8o_attn_single_q(out, q, k_blocks, v_blocks, kscale, vscale, seq_len, kv_dim, kv_bs, nkv,
                       kh_off, hd, scale, toks, nt, NULL, NULL);
    free(toks);
    free(sel);
    free(bs);
    return 1;
}

/* ------------------------------------------------------------------------ */
/* Shared selection per KV head (not on the pages: the variant that lets the */
/* G query heads of a KV head read the same blocks once).  READING: the      */
/* group's score of block j is the max over its G query heads of their       */
/* [10-1] block scores; one top-k on that (ties to the lower block); every   */
/* head then runs the one pass over the same kept blocks in ascending order. */
/* The gate is the same.  q, out: [G][hd]; sel_out (optional): [topk].       */
/* ------------------------------------------------------------------------ */
int kq8o_sparse_attn_group(float* out, const float* q, int G, int8_t* const* k_blocks,
                           int8_t* const* v_blocks, const float* kscale, const float* vscale,
                           int seq_len, int kv_dim, int kv_bs, int nkv, int kh_off, int hd,
                           float scale, int block, int topk, int probe, int32_t* sel_out) {
    if (sel_out)
        for (int i = 0; i < topk; i++) sel_out[i] = -1;
    if (seq_len <= 2 * block) {
        for (int g = 0; g < G; g++)
            kq8o_attn_single_q(out + (size_t)g * hd, q + (size_t)g * hd, k_blocks, v_blocks,
                               kscale, vscale, seq_len, kv_dim, kv_bs, nkv, kh_off, hd, scale,
                               NULL, 0, NULL, NULL);
        return 0;
    }
    int nb = (seq_len + block - 1) / block;
    float* best = (float*)malloc(sizeof(float) * (size_t)nb);
    float* bs = (float*)malloc(sizeof(float) * (size_t)nb);
    for (int g = 0; g < G; g++) {
        kq8o_probe_block_scores(bs, q + (size_t)g * hd, k_blocks, kscale, seq_len, kv_dim, kv_bs,
                                nkv, kh_off, hd, scale, block, probe);
        for (int j = 0; j < nb; j++) best[j] = (g == 0 || bs[j] > best[j]) ? bs[j] : best[j];
    }
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)(topk < nb ? topk : nb));
    int m = kq8o_topk_blocks(sel, best, nb, topk);
    int32_t* toks = (int32_t*)malloc(sizeof(int32_t) * (size_t)m * (size_t)block);
    int nt = 0;
    for (int i = 0; i < m; i++) {
        int j = sel[i];
        for (int t = j * block; t < (j + 1) * block && t < seq_len; t++) toks[nt++] = t;
        if (sel_out) sel_out[i] = j;
    }
    for (int g = 0; g < G; g++)
        kq8o_attn_single_q(out + (size_t)g * hd, q + (size_t)g * hd, k_blocks, v_blocks, kscale,
                           vscale, seq_len, kv_dim, kv_bs, nkv, kh_off, hd, scale, toks, nt, NULL,
                           NULL);
    free(toks);
    free(sel);
    free(bs);
    free(best);
    return 1;
}

/* ------------------------------------------------------------------------ */
/* Batch drivers over the pages' layout.  All B sequences of one layer live  */
/* in one token-major array rows[total_tokens][nkv*hd] (int8) with           */
/* row_offset[b] the first row of sequence b, and scales[total_tokens][nkv]; */
/* blocks of sequence b are its consecutive kv_bs-row slices.  Query head h  */
/* reads KV head h / (nq / nkv).                                              */
/* READING (pages silent): query head h shares KV head h / G, G = nq / nkv.   */
/* ------------------------------------------------------------------------ */
static int8_t** make_block_ptrs(int8_t* rows, int64_t first_row, int seq_len, int kv_bs, int kv_dim) {
    int nb = (seq_len + kv_bs - 1) / kv_bs;
    if (nb == 0) nb = 1;
    int8_t** p = (int8_t**)malloc(sizeof(int8_t*) * (size_t)nb);
    for (int j = 0; j < nb; j++) p[j] = rows + (size_t)(first_row + (int64_t)j * kv_bs) * (size_t)kv_dim;
    return p;
}

int kq8o_decode_batch(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                      const float* kscale, const float* vscale, const int64_t* row_offset,
                      const int32_t* seq_lens, int B, int nq, int nkv, int hd, int kv_bs,
                      float scale, int sparse, int block, int topk, int probe,
                      int32_t* sel_out, int nthreads) {
    if (hd > KQ8O_MAX_HD || hd % 32 != 0 || nkv <= 0 || nq % nkv != 0) return -1;
    int G = nq / nkv;
    int kv_dim = nkv * hd;
    int64_t units = (int64_t)B * nq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; u++) {
        int b = (int)(u / nq), h = (int)(u % nq);
        int kh = h / G;
        int8_t** kb = make_block_ptrs(k_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        int8_t** vb = make_block_ptrs(v_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        const float* ks = kscale + (size_t)row_offset[b] * nkv + kh;
        const float* vs = vscale + (size_t)row_offset[b] * nkv + kh;
        float* o = out + (size_t)u * hd;
        const float* qq = q + (size_t)u * hd;
        if (sparse)
            kq8o_sparse_attn_head(o, qq, kb, vb, ks, vs, seq_lens[b], kv_dim, kv_bs, nkv,
                                  kh * hd, hd, scale, block, topk, probe,
                                  sel_out ? sel_out + (size_t)u * topk : NULL);
        else
            kq8o_attn_single_q(o, qq, kb, vb, ks, vs, seq_lens[b], kv_dim, kv_bs, nkv, kh * hd,
                               hd, scale, NULL, 0, NULL, NULL);
        free(kb);
        free(vb);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Batched prefill over the same layout ([10-1] §1: a batch of nb new tokens */
/* scores against the whole history, O(nb*n) exact or O(nb*k*block) sparse;  */
/* §2: the prefill gate picks the exact or the block-sparse batched kernel).  */
/* Queries are packed: sequence b owns query rows q_off[b] .. q_off[b+1]-1,   */
/* nb_b = q_off[b+1] - q_off[b] of them, and its cache already holds those    */
/* tokens, so seq_lens[b] >= nb_b.                                            */
/* READING (the pages give no formula for the batched kernel): query i of     */
/* sequence b is the token at position p = seq_lens[b] - nb_b + i and sees    */
/* tokens 0..p (causal), each query handled exactly as one decode query with  */
/* seq_len = p + 1 -- same Q quantisation, score, one-pass online softmax and */
/* single divide; with sparse set, the block-sparse head over that prefix,    */
/* whose own gate (n <= 2*block -> exact) applies per query.                  */
/* out: [total_q][nq][hd]; sel_out (sparse, optional): [total_q][nq][topk].   */
/* ------------------------------------------------------------------------ */
int kq8o_prefill_batch(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                       const float* kscale, const float* vscale, const int64_t* row_offset,
                       const int32_t* seq_lens, const int32_t* q_off, int B, int nq, int nkv,
                       int hd, int kv_bs, float scale, int sparse, int block, int topk, int probe,
                       int32_t* sel_out, int nthreads) {
    if (hd > KQ8O_MAX_HD || hd % 32 != 0 || nkv <= 0 || nq % nkv != 0) return -1;
    for (int b = 0; b < B; b++) {
        int nb = q_off[b + 1] - q_off[b];
        if (nb < 0 || nb > seq_lens[b]) return -1;
    }
    int G = nq / nkv;
    int kv_dim = nkv * hd;
    int64_t units = (int64_t)q_off[B] * nq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; u++) {
        int r = (int)(u / nq), h = (int)(u % nq);
        int b = 0;
        while (q_off[b + 1] <= r) b++;
        int nb = q_off[b + 1] - q_off[b];
        int n = seq_lens[b] - nb + (r - q_off[b]) + 1; /* visible prefix */
        int kh = h / G;
        int8_t** kb = make_block_ptrs(k_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        int8_t** vb = make_block_ptrs(v_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        const float* ks = kscale + (size_t)row_offset[b] * nkv + kh;
        const float* vs = vscale + (size_t)row_offset[b] * nkv + kh;
        float* o = out + (size_t)u * hd;
        const float* qq = q + (size_t)u * hd;
        if (sparse)
            kq8o_sparse_attn_head(o, qq, kb, vb, ks, vs, n, kv_dim, kv_bs, nkv, kh * hd, hd, scale,
                                  block, topk, probe, sel_out ? sel_out + (size_t)u * topk : NULL);
        else
            kq8o_attn_single_q(o, qq, kb, vb, ks, vs, n, kv_dim, kv_bs, nkv, kh * hd, hd, scale,
                               NULL, 0, NULL, NULL);
        free(kb);
        free(vb);
    }
    return 0;
}

/* Write path over a batch of rows: x[T][nkv][hd] -> codes[T][nkv][hd] and
 * stored maxima[T][nkv] ([9-3] §2, applied per (token, head)). */
void kq8o_kv_quantize_rows(const float* x, int64_t T, int nkv, int hd, int8_t* codes, float* maxima) {
    for (int64_t t = 0; t < T; t++)
        for (int h = 0; h < nkv; h++) {
            size_t r = (size_t)t * nkv + h;
            kq8o_kv_quantize_row(x + r * hd, hd, codes + r * hd, maxima + r);
        }
}

/* Block-sparse decode with one selection per KV head (kq8o_sparse_attn_group)
 * over the batch layout of kq8o_decode_batch; sel_out: [B][nq][topk], the
 * group's selection repeated for each of its query heads. */
int kq8o_decode_batch_shared(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                             const float* kscale, const float* vscale, const int64_t* row_offset,
                             const int32_t* seq_lens, int B, int nq, int nkv, int hd, int kv_bs,
                             float scale, int block, int topk, int probe, int32_t* sel_out,
                             int nthreads) {
    if (hd > KQ8O_MAX_HD || hd % 32 != 0 || nkv <= 0 || nq % nkv != 0) return -1;
    int G = nq / nkv;
    int kv_dim = nkv * hd;
    int64_t units = (int64_t)B * nkv;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; u++) {
        int b = (int)(u / nkv), kh = (int)(u % nkv);
        int8_t** kb = make_block_ptrs(k_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        int8_t** vb = make_block_ptrs(v_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        size_t row0 = (size_t)b * nq + (size_t)kh * G;
        int32_t* sel = sel_out ? sel_out + row0 * topk : NULL;
        kq8o_sparse_attn_group(out + row0 * hd, q + row0 * hd, G, kb, vb,
                               kscale + (size_t)row_offset[b] * nkv + kh,
                               vscale + (size_t)row_offset[b] * nkv + kh, seq_lens[b], kv_dim,
                               kv_bs, nkv, kh * hd, hd, scale, block, topk, probe, sel);
        if (sel)
            for (int g = 1; g < G; g++) memcpy(sel + (size_t)g * topk, sel, sizeof(int32_t) * topk);
        free(kb);
        free(vb);
    }
    return 0;
}

/* q4 write path over a batch of rows (reading above). *//* q4 write path over a batch of rows (reading above). */
void kq8o_kv_quantize_rows_q4(const float* x, int64_t T, int nkv, int hd, int8_t* codes,
                              float* maxima) {
    for (int64_t t = 0; t < T; t++)
        for (int h = 0; h < nkv; h++) {
            size_t r = (size_t)t * nkv + h;
            kq8o_kv_quantize_row_q4(x + r * hd, hd, codes + r * hd, maxima + r);
        }
}

/* Exact decode over a q4 cache (codes as int8 in [-7, 7]), the batch driver
 * of kq8o_decode_batch with the q4 one pass.  The block-sparse path is not
 * offered for q4 ([10-1] §2: sparse attention is unavailable with --kv-q4). */
int kq8o_decode_batch_q4(float* out, const float* q, int8_t* k_rows, int8_t* v_rows,
                         const float* kscale, const float* vscale, const int64_t* row_offset,
                         const int32_t* seq_lens, int B, int nq, int nkv, int hd, int kv_bs,
                         float scale, int nthreads) {
    if (hd > KQ8O_MAX_HD || hd % 32 != 0 || nkv <= 0 || nq % nkv != 0) return -1;
    int G = nq / nkv;
    int kv_dim = nkv * hd;
    int64_t units = (int64_t)B * nq;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#else
    (void)nthreads;
#endif
    for (int64_t u = 0; u < units; u++) {
        int b = (int)(u / nq), h = (int)(u % nq);
        int kh = h / G;
        int8_t** kb = make_block_ptrs(k_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        int8_t** vb = make_block_ptrs(v_rows, row_offset[b], seq_lens[b], kv_bs, kv_dim);
        kq8o_attn_single_q_q4(out + (size_t)u * hd, q + (size_t)u * hd, kb, vb,
                              kscale + (size_t)row_offset[b] * nkv + kh,
                              vscale + (size_t)row_offset[b] * nkv + kh, seq_lens[b], kv_dim,
                              kv_bs, nkv, kh * hd, hd, scale);
        free(kb);
        free(vb);
    }
    return 0;
}

int kq8o_has_openmp(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 0;
#endif
}
