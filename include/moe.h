/*
 * moe.h -- C ABI of the GB300 (sm_103a) mixture-of-experts FFN layer with
 * SelectedSoftmax routing.
 *
 * The layer, per token t with input row x_t[d]:
 *   1. router projection  l[t,e] = sum_i x[t,i] * W_r[e,i]
 *   2. SelectedSoftmax    rank experts by l[t,e] + b[e], keep the top k
 *      (equal scores: lower expert index first), weight each kept expert by
 *      the softmax of the kept *unbiased* logits
 *      ("New Community Model: ZONOS3-Mini (Zyphra) - #1271", §Framework change)
 *   3. token grouping     per-expert counts, exclusive scan, stable permutation
 *      (grouped expert compute as in ggml's mul_mat_id,
 *       "zonos2.cpp internals", §Performance)
 *   4. SwiGLU experts     h = SiLU(W_g[e] x) * (W_u[e] x),  y = W_d[e] h
 *      ("zonos2.cpp internals", §Recommended: expert stacks ffn_{gate,up,down}_exps;
 *       "... - #1271", §Summary: SwiGLU FFN)
 *   5. combine            out[t] = sum_j w[t,j] * y_j, fp32 (residual streams
 *      are F32, "zonos2.cpp internals", §Notes)
 *
 * Conventions for every entry point:
 *  - All tensor arguments are DEVICE pointers owned by the caller, row-major,
 *    16-byte aligned.  The library never allocates, frees or synchronises on
 *    these paths; work is enqueued on `stream` (a cudaStream_t; NULL = the
 *    legacy default stream) and the call returns once it is enqueued.
 *  - Argument errors are reported synchronously, before anything is
 *    enqueued.  A kernel launch failure returns MOE_ERR_CUDA.  Nothing aborts.
 *  - Shapes: T tokens (T >= 0; T == 0 is a no-op), d model width, E experts
 *    (1..256), k experts per token (1..min(E, 8)), F expert ffn width.
 *  - Activation storage (x, W_r): MOE_F32 or MOE_BF16; logits, routing
 *    weights and the output are fp32.  Expert weights: MOE_F32 (with F32
 *    activations), MOE_BF16, MOE_Q8_0, MOE_Q4_A64, MOE_Q4_K, MOE_Q6_K or MOE_FP8
 *    (with BF16 activations).
 *  - Calls on distinct workspaces and outputs are independent; there is no
 *    global mutable state.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

/* A cudaStream_t, passed as an opaque pointer. */
typedef void *moe_stream;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, k > E ... */
    MOE_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype combination, E > 256 ...) */
    MOE_ERR_WORKSPACE = 3,     /* workspace smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (see moe_check) */
    MOE_ERR_DEVICE_CHECK = 6   /* a device-side consistency check failed (see moe_check) */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_Q8_0 = 2, MOE_Q4_A64 = 3, MOE_Q4_K = 4, MOE_Q6_K = 5,
               MOE_FP8 = 6 } moe_dtype;

/* Which expert-compute kernels moe_forward uses.  AUTO picks by shape.
 * DECODE: few rows per expert -- tcgen05 weight-streaming kernels for bf16,
 *   4-bit (affine, Q4_K) and 8-bit-plane (Q8_0, Q6_K, fp8) weights (converted to
 *   fp16 on chip) with d % 128 == 0, F % 128 == 0 and T*k <= 8192, otherwise
 *   the CUDA-core kernels.  PREFILL: tcgen05 grouped GEMMs.  DECODE_SIMT:
 *   always the CUDA-core decode kernels (the decode path for fp32). */
typedef enum {
    MOE_PATH_AUTO = 0,
    MOE_PATH_DECODE = 1,
    MOE_PATH_PREFILL = 2,
    MOE_PATH_DECODE_SIMT = 3
} moe_path;

/* Static description of a status code (never NULL). */
MOE_API const char *moe_status_str(int status);

/* ABI version of this library (major * 100 + minor). */
MOE_API int moe_version(void);

/*
 * moe_route -- steps 1-2 (router projection + SelectedSoftmax).
 *   x[T,d], w_router[E,d]: storage act_dt (F32 or BF16), fp32 accumulation.
 *   sel_bias[E] fp32, or NULL for no bias; it changes which experts are kept,
 *   never their weights.
 *   topk_idx[T,k] int32 out: kept experts in ranking order (score descending,
 *   then index ascending).
 *   topk_w[T,k] fp32 out: softmax over the kept experts' unbiased logits;
 *   with k == 1 every weight is exactly 1.0f.
 *   Kernel: the router moe_forward runs for the same x -- the clustered
 *   tensor-core router for bf16 batches of T <= 128 (moe_forward's bf16
 *   decode path), the tensor-core router for bf16 batches of T >= 512, the
 *   CUDA-core router otherwise.
 */
MOE_API moe_status moe_route(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                     const float *sel_bias, int E, int k, int32_t *topk_idx, float *topk_w,
                     moe_stream stream);

/*
 * Scoring modes of the router ("New Community Model: ZONOS3-Mini (Zyphra) -
 * #1271", §Framework change: SelectedSoftmax is added beside the older modes,
 * which apply a softmax or a sigmoid before ranking and so weigh experts
 * differently; the pages give no formulas, the reading taken here is):
 *   MOE_SCORE_SELECTED_SOFTMAX  rank by logit + bias, weights = softmax of the
 *                               kept experts' logits (moe_route, moe_forward);
 *   MOE_SCORE_SOFTMAX           p = softmax of the logits over all E experts,
 *                               rank by p + bias, weights = p of the kept
 *                               experts (not renormalised);
 *   MOE_SCORE_SIGMOID           p = sigmoid(logit), rank by p + bias,
 *                               weights = p of the kept experts.
 * Ties in the ranking score go to the lower expert index in every mode.
 */
typedef enum {
    MOE_SCORE_SELECTED_SOFTMAX = 0,
    MOE_SCORE_SOFTMAX = 1,
    MOE_SCORE_SIGMOID = 2
} moe_scoring;

/*
 * moe_route_scored -- moe_route with scoring mode `scoring` (a moe_scoring
 *   value; anything else is MOE_ERR_INVALID_ARG).
 */
MOE_API moe_status moe_route_scored(const void *x, moe_dtype act_dt, int T, int d,
                                    const void *w_router, const float *sel_bias, int E, int k,
                                    int scoring, int32_t *topk_idx, float *topk_w,
                                    moe_stream stream);

/*
 * moe_permute -- step 3 (token grouping), integer-exact and atomic-free.
 *   topk_idx[T,k] int32 in, each value in [0, E).
 *   counts[E]      out: number of (t, j) slots routed to expert e.
 *   offsets[E+1]   out: exclusive prefix sum of counts (offsets[E] == T*k).
 *   perm_tok[T*k]  out: token of grouped row r; rows of expert e are
 *                  [offsets[e], offsets[e+1]) in increasing flat slot order
 *                  t*k + j (i.e. increasing t).
 *   inv[T*k]       out: grouped row of flat slot t*k + j.
 *   All five buffers are device memory, 4-byte aligned, owned by the caller.
 *   An expert id outside [0, E) is left out of counts and of the permutation
 *   (its inv entry is not written, no other memory is touched); moe_forward's
 *   own indices always come from its router.
 */
MOE_API moe_status moe_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                       int32_t *offsets, int32_t *perm_tok, int32_t *inv, moe_stream stream);

/*
 * Q8_0 expert weights.  Input format: rows of `cols` values along the
 * contiguous (reduction) axis, stored as cols/32 blocks of 34 bytes
 * {fp16 scale (little endian), int8 q[32]}; value = scale * q.
 * moe_forward consumes them repacked into two planes in one buffer:
 *   bytes [0, rows*cols)                     int8 q plane [rows, cols]
 *   bytes [align256(rows*cols), ... + rows*cols/16)  fp16 scale plane [cols/32, rows]
 *   (the scale of block b of row r is at index b*rows + r)
 * moe_q8_0_packed_size returns the buffer size (0 if cols % 32 != 0 or
 * rows < 0).  moe_pack_q8_0 repacks `blocks` (device, any alignment) into
 * `packed` (device, 256-byte aligned) on `stream`; pack W_g and W_u as
 * rows = E*F, cols = d and W_d as rows = E*d, cols = F.
 * Range: the Q8_0 grouped GEMMs (MOE_PATH_PREFILL) multiply fp16 operands.
 * Each token row enters them scaled by an exact power of two so that its
 * largest magnitude is at most 1, and h is held scaled by the square of that
 * factor; both are undone exactly in the epilogues, so any finite bf16
 * activations are taken.  An h that still leaves fp16's range (|h| > 65504
 * after the scaling: expert weights with dot products above ~256 against a
 * unit row) makes moe_check report MOE_ERR_DEVICE_CHECK.  The tensor-core
 * decode kernels (MOE_PATH_DECODE, d and F multiples of 128) take Q8_0 the
 * same way; the CUDA-core Q8_0 decode kernels compute in fp32.
 */
MOE_API size_t moe_q8_0_packed_size(long long rows, int cols);
MOE_API moe_status moe_pack_q8_0(const void *blocks, long long rows, int cols, void *packed,
                         moe_stream stream);

/*
 * Affine 4-bit expert weights, groups of 64 (MOE_Q4_A64; the expert format of
 * the MLX build, "Zyphra-ZONOS2-4bit", §How this was quantized: experts at
 * 4 bits, group size 64, affine mode; the page gives no byte layout, this is
 * the library's).
 * Input format: rows of `cols` values along the contiguous axis, stored as
 * cols/64 blocks of 36 bytes {fp16 scale, fp16 bias (little endian), 32 bytes
 * of codes: value 2j in the low nibble of byte j, 2j+1 in the high nibble};
 * value = scale * q + bias.  Used with BF16 activations on the tensor-core
 * decode kernels (d and F multiples of 128), the grouped GEMMs of
 * MOE_PATH_PREFILL (d % 256 == 0, F % 128 == 0) or the CUDA-core decode
 * kernels.  The tensor-core kernels multiply fp16 operands: each weight is scale * q + bias rounded once to
 * fp16, each token row is x times a power of two (exact), and h is held in
 * fp16 scaled by the square of that power, as on the Q8_0 path; an h beyond
 * fp16's range there is reported as MOE_ERR_DEVICE_CHECK.  moe_forward
 * consumes them repacked into tiles of 128 rows x 64 columns (one group),
 * 4608 bytes each, so that one k-block of one row tile is one contiguous copy:
 *   tile (rt, g), rt = row / 128, g = col / 64, at byte ((rt * cols/64) + g) * 4608
 *   bytes [0, 4096)       the tile's 128 rows of 32 code bytes, in row order; each
 *                         little-endian 32-bit word holds 8 consecutive values,
 *                         value 2i in bits 4i..4i+3 and value 2i+1 in bits
 *                         16+4i..19+4i (i = 0..3)
 *   bytes [4096, 4352)    their 128 fp16 scales
 *   bytes [4352, 4608)    their 128 fp16 biases
 * Rows past `rows` in the last row tile are zero.  moe_q4_a64_packed_size
 * returns ceil(rows / 128) * (cols / 64) * 4608 (0 if cols % 64 != 0 or
 * rows < 0); moe_pack_q4_a64 repacks `blocks` (device, any alignment) into
 * `packed` (device, 256-byte aligned) on `stream`, with the same rows/cols as
 * moe_pack_q8_0.
 */
MOE_API size_t moe_q4_a64_packed_size(long long rows, int cols);
MOE_API moe_status moe_pack_q4_a64(const void *blocks, long long rows, int cols, void *packed,
                                   moe_stream stream);

/*
 * Q4_K expert weights (MOE_Q4_K): the K-quant the pages recommend for the
 * expert stacks ("zonos2.cpp internals", §Recommended: F16 spine + K-quant
 * experts: Q4_K at 4.50 bits per weight is the usable floor; the pages give
 * no byte layout, this is the GGUF one).  Input format: rows of `cols`
 * values (cols % 256 == 0), stored as cols/256 super-blocks of 144 bytes
 * {fp16 d, fp16 dmin (little endian), 12 bytes of six-bit sub-block scales
 * sc[8] and mins m[8], 128 bytes of 4-bit codes}; sub-block j holds values
 * 32j .. 32j+31 and decodes as d * sc[j] * q - dmin * m[j].  Six-bit fields:
 * for j < 4, sc[j] and m[j] are the low 6 bits of bytes j and j+4; for
 * j >= 4, sc[j] = (low nibble of byte j+4) + 16 * (top 2 bits of byte j-4)
 * and m[j] = (high nibble of byte j+4) + 16 * (top 2 bits of byte j).
 * Codes: the 32-byte run c (c = 0..3) holds sub-block 2c in its low nibbles
 * and 2c+1 in its high nibbles, value i of each in byte i of the run.
 * Used like MOE_Q4_A64 (BF16 activations; tensor-core decode kernels, grouped
 * GEMMs, CUDA-core decode kernels) with d and F multiples of 256.
 * moe_forward consumes them repacked by moe_pack_q4_k into the tiles of
 * MOE_Q4_A64 (128 rows x 64 columns, same code words) with two affine groups
 * per tile row: bytes [0, 4096) codes, [4096, 4608) fp16 scales [2][128]
 * (group 0: values 0-31 of the tile row, group 1: values 32-63), [4608, 5120)
 * fp16 biases [2][128]; a value decodes as scale * (q - 8) + bias with
 * scale = fp16(d * sc[j]) and bias = fp16(8 d sc[j] - dmin m[j]), the value at
 * code 8 (the middle of the group's range, so that the two fp16 roundings
 * stay small; the tensor-core kernels then round each weight once more, to
 * fp16).
 * moe_q4_k_packed_size returns ceil(rows / 128) * (cols / 64) * 5120 (0 if
 * cols % 256 != 0 or rows < 0); moe_pack_q4_k repacks `blocks` (device, any
 * alignment) into `packed` (device, 256-byte aligned) on `stream`.
 */
MOE_API size_t moe_q4_k_packed_size(long long rows, int cols);
MOE_API moe_status moe_pack_q4_k(const void *blocks, long long rows, int cols, void *packed,
                                 moe_stream stream);

/*
 * Q6_K expert weights (MOE_Q6_K): the K-quant the pages call the sweet spot of
 * the expert ladder ("zonos2.cpp internals", §Recommended: F16 spine + K-quant
 * experts: Q6_K at 6.56 bits per weight; the pages give no byte layout, this
 * is the GGUF one).  Input format: rows of `cols` values (cols % 256 == 0),
 * stored as cols/256 super-blocks of 210 bytes {ql[128]: low 4 bits of the
 * 6-bit codes, qh[64]: their top 2 bits, int8 scales[16], fp16 d (little
 * endian)}.  Value v = 128h + 32g + l of a block (h < 2, g < 4, l < 32): low
 * bits in the low (g < 2) or high (g >= 2) nibble of ql[64h + l + 32 (g % 2)],
 * top bits in bits 2g and 2g+1 of qh[32h + l]; it decodes as
 * d * scales[v / 16] * (q - 32).
 * moe_forward consumes them repacked like Q8_0 into two planes in one buffer,
 * with one scale per 16 values:
 *   bytes [0, rows*cols)                              int8 plane [rows, cols], q - 32
 *   bytes [align256(rows*cols), ... + rows*cols/8)    fp16 scale plane [cols/16, rows]
 *   (the scale of group j of row r, fp16(d * scales[j]), at index j*rows + r)
 * and takes them where Q8_0 goes: the grouped GEMMs and the tensor-core
 * decode kernels (fp16 operands, the same range rules) and the CUDA-core
 * decode kernels (fp32), with d and F multiples of 256.  moe_q6_k_packed_size returns the buffer size (0 if
 * cols % 256 != 0 or rows < 0); moe_pack_q6_k repacks `blocks` (device, any
 * alignment) into `packed` (device, 256-byte aligned) on `stream`.
 */
MOE_API size_t moe_q6_k_packed_size(long long rows, int cols);
MOE_API moe_status moe_pack_q6_k(const void *blocks, long long rows, int cols, void *packed,
                                 moe_stream stream);

/*
 * fp8 expert weights (MOE_FP8): the serving configurations run "fp8" ("zonos2"
 * sglang-omni cookbook, §Benchmark Results); the pages fix neither the 8-bit
 * variant nor the scaling, and this library reads it as OCP E4M3 codes (sign,
 * 4 exponent bits with bias 7, 3 mantissa bits, no infinities, NaN codes 0x7F
 * and 0xFF, largest finite 448) with one fp32 scale per row (output channel;
 * a per-tensor scale is the case of equal rows).  Input format: per row
 * {fp32 scale (little endian), cols E4M3 codes}, 4 + cols bytes; value =
 * scale * E4M3(code).
 * moe_forward consumes them repacked into one buffer:
 *   bytes [0, rows*cols)                            E4M3 plane [rows, cols]
 *   bytes [align256(rows*cols), ... + 4*rows)       fp32 scale per row
 * The tensor-core kernels (grouped GEMMs, decode) widen the codes to fp16
 * exactly, multiply by fp16 token rows with fp32 accumulation (the same range
 * rules as Q8_0) and apply each row's scale to its fp32 sums; the CUDA-core
 * decode kernels compute scale * code in fp32.  NaN codes (0x7F, 0xFF) are not
 * validated: they propagate into the outputs as NaN (some paths' range check on h
 * may also report MOE_ERR_DEVICE_CHECK).  d and F multiples of 8 (the
 * tensor-core kernels: as for bf16).  moe_fp8_packed_size returns the buffer
 * size (0 if rows < 0 or cols <= 0); moe_pack_fp8 repacks `rows_in` (device,
 * any alignment) into `packed` (device, 256-byte aligned) on `stream`.
 */
MOE_API size_t moe_fp8_packed_size(long long rows, int cols);
MOE_API moe_status moe_pack_fp8(const void *rows_in, long long rows, int cols, void *packed,
                                moe_stream stream);

/*
 * Bytes of device workspace moe_forward needs for these sizes (any path).
 * 0 on invalid sizes.  The workspace is scratch owned by the caller; its
 * first 256 bytes hold the device status word read by moe_check.
 */
MOE_API size_t moe_workspace_size(int T, int d, int E, int k, int F, moe_dtype act_dt,
                          moe_dtype w_dt);

/*
 * moe_workspace_views -- where a layer call leaves its routing and token
 * grouping (steps 2-3) inside its workspace, so that a caller can read back
 * exactly what the layer's own kernels computed (for checking, or to reuse
 * the grouping).  For a moe_forward / moe_forward_profiled /
 * moe_forward_scored / moe_ffn_dense call with these sizes (moe_ffn_dense:
 * E = 1, k = 1), `views[i]` receives the byte offset from the workspace
 * pointer of:
 *   views[0] topk_idx  int32 [T, k]   kept experts, ranking order
 *   views[1] topk_w    fp32  [T, k]   their routing weights
 *   views[2] counts    int32 [E]      rows per expert
 *   views[3] offsets   int32 [E + 1]  exclusive prefix sum of counts
 *   views[4] perm_tok  int32 [T*k]    token of grouped row r
 *   views[5] inv       int32 [T*k]    grouped row of slot t*k + j
 *   views[6] perm_w    fp32  [T*k]    routing weight of grouped row r
 * (the same conventions as moe_route and moe_permute).  The arrays hold the
 * call's values once its work on its stream has completed, until the next
 * call on the same workspace.  Returns MOE_ERR_INVALID_ARG for sizes that
 * moe_workspace_size rejects or a NULL `views`.
 */
MOE_API moe_status moe_workspace_views(int T, int d, int E, int k, int F, moe_dtype act_dt,
                                       moe_dtype w_dt, size_t *views);

/*
 * moe_forward -- the whole layer, steps 1-5.
 *   x[T,d] (act_dt), w_router[E,d] (act_dt), sel_bias[E] fp32 or NULL,
 *   w_gate[E,F,d], w_up[E,F,d], w_down[E,d,F] in w_dt (Q8_0 / Q4_A64 / Q4_K / Q6_K /
 *   fp8: the buffers written by moe_pack_q8_0 / moe_pack_q4_a64 / moe_pack_q4_k /
 *   moe_pack_q6_k / moe_pack_fp8, 256-byte aligned),
 *   out[T,d] fp32 (overwritten).
 *   workspace: device scratch of at least moe_workspace_size() bytes,
 *   256-byte aligned; it must not be shared by calls that can overlap.
 *   path: a moe_path value.  MOE_PATH_PREFILL needs bf16 activations,
 *   bf16 or Q8_0 weights, d % 256 == 0 and F % 128 == 0, and returns
 *   MOE_ERR_UNSUPPORTED otherwise.
 *   Reproducibility: every path gives bitwise identical results from run to
 *   run, for every k, and permuting the tokens permutes the output rows bit
 *   for bit: sums of split-K partials are added in split order, k = 2 outputs
 *   are two additions onto zero (whose result does not depend on their
 *   order), and with k > 2 each token's k expert outputs are added in slot
 *   order by a combine kernel.
 */
MOE_API moe_status moe_forward(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                       const float *sel_bias, int E, int k, const void *w_gate,
                       const void *w_up, const void *w_down, moe_dtype w_dt, int F,
                       float *out, void *workspace, size_t ws_bytes, int path,
                       moe_stream stream);

/*
 * moe_forward_profiled -- moe_forward that also records caller-created CUDA
 * events (cudaEvent_t, timing enabled) on `stream` at its stage boundaries,
 * so a caller can time each kernel on the stream it runs on:
 *   events[0] before routing          events[3] after the row gather
 *   events[1] after routing           events[4] after gate/up + SwiGLU
 *   events[2] after token grouping    events[5] after down + combine
 * (where no separate gather kernel runs, events[3] follows events[2]
 * immediately).  events may be NULL, which makes this moe_forward.
 */
MOE_API moe_status moe_forward_profiled(const void *x, moe_dtype act_dt, int T, int d,
                                        const void *w_router, const float *sel_bias, int E,
                                        int k, const void *w_gate, const void *w_up,
                                        const void *w_down, moe_dtype w_dt, int F, float *out,
                                        void *workspace, size_t ws_bytes, int path,
                                        void *const *events, moe_stream stream);

/*
 * moe_forward_scored -- moe_forward_profiled with scoring mode `scoring` (a
 *   moe_scoring value; anything else is MOE_ERR_INVALID_ARG).  events may be
 *   NULL.
 */
MOE_API moe_status moe_forward_scored(const void *x, moe_dtype act_dt, int T, int d,
                                      const void *w_router, const float *sel_bias, int E, int k,
                                      const void *w_gate, const void *w_up, const void *w_down,
                                      moe_dtype w_dt, int F, float *out, void *workspace,
                                      size_t ws_bytes, int path, int scoring,
                                      void *const *events, moe_stream stream);

/*
 * moe_ffn_dense -- a dense SwiGLU FFN layer: out = W_d (SiLU(W_g x) * (W_u x))
 *   per token, the E = 1, k = 1 case of the layer ("zonos2.cpp internals",
 *   §Model architecture: dense FFN layers beside the MoE ones; "New Community
 *   Model: ZONOS3-Mini (Zyphra) - #1271", §Summary: layer 0 has a dense SwiGLU
 *   FFN).  No router: every token goes to the one expert with weight 1.
 *   w_gate[F,d], w_up[F,d], w_down[d,F] in w_dt (Q8_0 / Q4_A64 / Q4_K / Q6_K / fp8: packed
 *   by the matching moe_pack_* with rows = F or d); other arguments as
 *   moe_forward, with a workspace of moe_workspace_size(T, d, 1, 1, F, act_dt,
 *   w_dt) bytes.
 */
MOE_API moe_status moe_ffn_dense(const void *x, moe_dtype act_dt, int T, int d,
                                 const void *w_gate, const void *w_up, const void *w_down,
                                 moe_dtype w_dt, int F, float *out, void *workspace,
                                 size_t ws_bytes, int path, moe_stream stream);

/*
 * moe_forward_noalloc -- moe_forward for callers that cannot allocate device
 * memory.  (No counterpart on the source pages: an addition of this library.)
 * Some hosts give the layer only its inputs and outputs -- serving runtimes
 * and plugin hosts that own all device memory through their own pool and
 * forbid cudaMalloc while serving, because it synchronises the device and can
 * fail under a fixed memory budget.  This entry point takes the same arguments
 * as moe_forward minus the workspace, runs the same kernels, and uses as
 * scratch one static 8 MiB device array inside the library instead; it calls
 * no allocator of any kind.
 *  - Errors: moe_forward's argument checks come first, with its return
 *    codes; then layers whose moe_workspace_size() exceeds 8 MiB (8388608
 *    bytes) are rejected with MOE_ERR_WORKSPACE.  Nothing is enqueued on an
 *    error.
 *  - Set-up: the first call on each device (with that device current) looks
 *    up the array's device address (again after the device's context is
 *    re-created, e.g. by cudaDeviceReset); make that first call before any
 *    stream capture.
 *  - Sharing: every call, on any stream, uses the same array, which keeps the
 *    previous call's contents (each call rewrites every scratch byte it reads,
 *    and its first kernel clears the status word).  Calls that can overlap on
 *    the GPU race on it: serialise them (one stream, or events).
 *  - Memory: every GPU that loads the library holds the 8 MiB until exit.
 *  - Device-side errors (a bounded wait that gave up, a failed consistency
 *    check) are read with moe_check_noalloc.
 */
MOE_API moe_status moe_forward_noalloc(const void *x, moe_dtype act_dt, int T, int d,
                                       const void *w_router, const float *sel_bias, int E, int k,
                                       const void *w_gate, const void *w_up, const void *w_down,
                                       moe_dtype w_dt, int F, float *out, int path,
                                       moe_stream stream);

/*
 * Test hook of the failure handling.  Every wait of the library's
 * tensor-core kernels is bounded (2 s); a wait that gives up records
 * MOE_ERR_TIMEOUT in the status word, the kernel's other roles stop, its
 * copies and MMAs in flight land, its TMEM is freed and it returns, and the
 * call's later kernels return without work.  moe_forward_expire_wait runs
 * moe_forward with one wait of one kernel family -- at its start, on a
 * barrier that nothing ever arrives on and that no copy or MMA targets --
 * limited to `wait_ns` (1 ns .. 100 ms) in every CTA of that kernel, so that
 * this path runs without any fault: moe_check then reports MOE_ERR_TIMEOUT
 * and the outputs of the call are invalid.  It returns MOE_ERR_UNSUPPORTED
 * (nothing enqueued) when the named family does not run for these arguments:
 *   MOE_KERNEL_ROUTER_CLUSTER  the clustered router (bf16 decode, T <= 128),
 *                              the MMA thread's operand wait
 *   MOE_KERNEL_ROUTER_TC       the tensor-core router (bf16, T >= 512)
 *   MOE_KERNEL_DECODE_SPLIT    the split-K tensor-core decode kernels (gate/up)
 *   MOE_KERNEL_DECODE_FUSED    the one-launch tensor-core decode kernel
 *   MOE_KERNEL_GEMM            the grouped GEMMs (gate/up; CTA pairs for Q8_0)
 * (the producer's first wait unless stated).  Not for production use.
 */
typedef enum {
    MOE_KERNEL_ROUTER_CLUSTER = 1,
    MOE_KERNEL_ROUTER_TC = 2,
    MOE_KERNEL_DECODE_SPLIT = 3,
    MOE_KERNEL_DECODE_FUSED = 4,
    MOE_KERNEL_GEMM = 5
} moe_kernel_family;
MOE_API moe_status moe_forward_expire_wait(const void *x, moe_dtype act_dt, int T, int d,
                                           const void *w_router, const float *sel_bias, int E,
                                           int k, const void *w_gate, const void *w_up,
                                           const void *w_down, moe_dtype w_dt, int F, float *out,
                                           void *workspace, size_t ws_bytes, int path,
                                           int kernel_family, uint32_t wait_ns, moe_stream stream);

/*
 * moe_check_noalloc -- moe_check for moe_forward_noalloc: wait for `stream`,
 * then read the status word the most recent moe_forward_noalloc on the
 * current device left in the library's static scratch (MOE_OK,
 * MOE_ERR_TIMEOUT or MOE_ERR_DEVICE_CHECK; `*device_word` optional).  It
 * synchronises, so it cannot be captured into a CUDA graph.
 */
MOE_API moe_status moe_check_noalloc(uint32_t *device_word, moe_stream stream);

/*
 * moe_check -- wait for `stream`, then read the device status word that the
 * most recent moe_forward on `workspace` left: MOE_OK, MOE_ERR_TIMEOUT (a
 * bounded device wait gave up; outputs of that call are invalid) or
 * MOE_ERR_DEVICE_CHECK.  `*device_word` (optional) receives the raw word.
 */
MOE_API moe_status moe_check(const void *workspace, uint32_t *device_word, moe_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
