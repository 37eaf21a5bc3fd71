/*
 * moe_oracle.h -- CPU fp64 oracle of the MoE FFN layer with SelectedSoftmax
 * routing.  TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU-baseline leg of
 * the benchmark).  Independent of the CUDA library: no shared code or headers.
 *
 * Storage dtypes: 0 = fp32, 1 = bf16 bit patterns (uint16), 2 = Q8_0 rows of
 * 34-byte blocks {fp16 scale, int8 q[32]} along the contiguous axis, 3 = affine
 * 4-bit rows of 36-byte blocks of 64 values {fp16 scale, fp16 bias, 32 bytes:
 * value 2j in the low nibble of byte j, 2j+1 in the high}, value = scale*q + bias,
 * 4 = Q4_K rows of 144-byte super-blocks of 256 values, 5 = Q6_K rows of 210-byte
 * super-blocks of 256 values (GGUF layouts; see moe_oracle.c), 6 = fp8 rows
 * {fp32 scale, E4M3 codes[cols]} (4 + cols bytes), value = scale * E4M3(code).
 * Activations (x, W_r) are fp32 or bf16; expert weights may also be Q8_0.
 * Layouts (row-major): x[T,d], W_r[E,d], W_g[E,F,d], W_u[E,F,d], W_d[E,d,F].
 * All functions return 0 on success, -1 on invalid arguments.
 * parity: pinned by tests/test_oracle.py (invariants, closed forms, a
 * hand-derived worked example, a dense numpy brute force).
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_Q8_0 = 2, ORACLE_Q4_A64 = 3, ORACLE_Q4_K = 4, ORACLE_Q6_K = 5,
       ORACLE_FP8 = 6 };

int oracle_default_threads(void);

/* logits[t,e] = sum_i x[t,i] W_r[e,i]; W_r has the dtype of x. */
int oracle_router_logits(const void *x, int x_dt, int T, int d, const void *w_router,
                         int E, double *logits, int nthreads);

/* SelectedSoftmax: top-k of logit+bias (ties -> lower index), weights =
 * softmax of the selected unbiased logits.  topk_idx/topk_w are [T,k], slots in
 * rank order.  margin[t] (optional) = k-th minus (k+1)-th ranking score,
 * +inf when k == E.  bias may be NULL (all zero). */
int oracle_selected_softmax(const double *logits, const float *bias, int T, int E, int k,
                            int32_t *topk_idx, double *topk_w, double *margin);

/* Scoring mode 0: SelectedSoftmax (as above).  Mode 1 / 2: p = softmax over
 * all E logits / sigmoid of each logit; top-k of p + bias (ties -> lower
 * index); weights = p of the selected experts (not renormalised); margin on
 * p + bias. */
int oracle_route_scored(const double *logits, const float *bias, int T, int E, int k, int mode,
                        int32_t *topk_idx, double *topk_w, double *margin);

/* Weights for a given selected set: softmax of logits over topk_idx[t,:]. */
int oracle_softmax_of_set(const double *logits, int T, int E, int k, const int32_t *topk_idx,
                          double *topk_w);

/* counts[E], offsets[E+1] (exclusive scan), perm_tok[T*k] (token of each
 * grouped row, tokens ascending within an expert), inv[T*k] (grouped row of
 * flat slot t*k+j). */
int oracle_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                   int32_t *offsets, int32_t *perm_tok, int32_t *inv);

/* out[t,:] = sum_j topk_w[t,j] * W_d[e] (SiLU(W_g[e] x_t) * (W_u[e] x_t)),
 * e = topk_idx[t,j]; out is fp64 [T,d]. */
int oracle_expert_combine(const void *x, int x_dt, int T, int d, const int32_t *topk_idx,
                          const double *topk_w, int k, const void *w_gate, const void *w_up,
                          const void *w_down, int w_dt, int E, int F, double *out, int nthreads);

/* Whole layer: router, SelectedSoftmax, experts, combine. */
int oracle_moe_forward(const void *x, int x_dt, int T, int d, const void *w_router,
                       const float *bias, int E, int k, const void *w_gate, const void *w_up,
                       const void *w_down, int w_dt, int F, double *out, int32_t *topk_idx,
                       double *topk_w, double *margin, int nthreads);

/* Whole layer with scoring mode `mode` (see oracle_route_scored). */
int oracle_moe_forward_scored(const void *x, int x_dt, int T, int d, const void *w_router,
                              const float *bias, int E, int k, int mode, const void *w_gate,
                              const void *w_up, const void *w_down, int w_dt, int F, double *out,
                              int32_t *topk_idx, double *topk_w, double *margin, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
