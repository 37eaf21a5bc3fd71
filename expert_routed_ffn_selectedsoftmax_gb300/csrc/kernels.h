// kernels.h -- internal launchers of the library's kernels (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// api.cu -- moe_forward's argument checks that do not involve the workspace
// (in moe_forward's order); MOE_OK when they pass.  `dense`: moe_ffn_dense
// (no router; w_router and sel_bias are ignored).
moe_status forward_args_check(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                              const float *sel_bias, int E, int k, const void *w_gate,
                              const void *w_up, const void *w_down, moe_dtype w_dt, int F,
                              const float *out, int path, int scoring, bool dense);

// route.cu
size_t route_smem_bytes(int tpb, int d, int E);
// out_zero: rows [T, d] to zero (or NULL); zero_words[n_zero]: scratch words
// later kernels need zeroed (or NULL); rank/tile_cnt: grouping inputs for the
// scatter over tiles of route_tokens_per_block() tokens (or NULL); status:
// device status word to clear.
int route_tokens_per_block(int T, int d, int E);
cudaError_t launch_route(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                         const float *bias, int E, int k, int32_t *topk_idx, float *topk_w,
                         float *out_zero, uint32_t *zero_words, int n_zero, int32_t *rank,
                         int32_t *tile_cnt, uint32_t *status, int mode, cudaStream_t stream);
// the tensor-core router pays off from this many tokens (one 128-row tile per CTA)
constexpr int kRouteTcMinTokens = 512;

// route_tc.cu -- tensor-core router + SelectedSoftmax, then the grouping scatter
struct RouteTcArgs {
    const void *x;              // [T, d] bf16
    const void *w_router;       // [E, d] bf16
    const float *bias;          // [E] or NULL
    int T, d, E, k;
    int mode;                   // scoring: 0 SelectedSoftmax, 1 softmax / 2 sigmoid before rank
    int32_t *topk_idx;          // [T*k]
    float *topk_w;              // [T*k]
    int32_t *rank;              // [T*k] scratch, or NULL (routing only)
    int32_t *tile_cnt;          // [route_tc_tiles(T) * E] scratch, or NULL
    // grouping outputs (counts == NULL: routing only, no scatter launch)
    int32_t *counts, *offsets, *perm_tok, *inv;
    float *perm_w;
    void *xp;                   // optional [T*k, d] grouped copy of x
    int xp_fp16;                // write xp as fp16 (else bf16), row r scaled by 2^-xexp[r]
    int32_t *xexp;              // [T*k] (xp_fp16): exponent of each grouped row's scale
    float *out_zero;            // optional rows to zero
    uint32_t *zero_words;       // optional scratch words to zero
    int n_zero;
    uint32_t *status;
    cudaEvent_t ev_routed;      // optional: recorded between routing and scatter
    uint32_t expire_ns;         // > 0: one bounded wait gives up after this long (test hook)
};
bool route_tc_capable(int act_dt, int d, int E);
int route_tc_tiles(int T);
cudaError_t launch_route_tc(const RouteTcArgs &a, cudaStream_t stream);
// grouping scatter over token tiles of `tile_tokens` (counts/ranks from either router)
cudaError_t launch_scatter(const RouteTcArgs &a, int ntiles, int tile_tokens, cudaStream_t stream);

constexpr int kRouteSmallRowsMaxT = 16;   // batches the clustered router also writes fp16 rows for
// route_small.cu -- routing and grouping in one clustered kernel for T <= 128
// (bf16 activations): writes topk_idx/topk_w and counts, offsets, perm_tok,
// inv, perm_w (counts == NULL: routing only), and zeroes out_zero and
// zero_words when given; ignores rank, tile_cnt and xp.
bool route_small_capable(int act_dt, int T, int d, int E, int k);
cudaError_t launch_route_small(const RouteTcArgs &a, cudaStream_t stream);

// permute.cu
cudaError_t launch_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                           int32_t *offsets, int32_t *perm_tok, int32_t *inv,
                           const float *topk_w, float *perm_w, uint32_t *status,
                           cudaStream_t stream);
// to_fp16: rows scaled by 2^-xexp[r] (fp16_row_exponent), xexp written
cudaError_t launch_gather_rows(const void *x, int d, const int32_t *perm_tok, int rows,
                               void *xp, int to_fp16, int32_t *xexp, int T, uint32_t *status,
                               int num_sms, cudaStream_t stream);
// dense layer (E = 1, k = 1): expert 0, weight 1, identity grouping; clears
// status and zero_words[n_zero]
cudaError_t launch_identity_grouping(int T, int32_t *topk_idx, float *topk_w, int32_t *counts,
                                     int32_t *offsets, int32_t *perm_tok, int32_t *inv,
                                     float *perm_w, uint32_t *status, uint32_t *zero_words,
                                     int n_zero, int num_sms, cudaStream_t stream);

// decode.cu -- expert FFN for few rows per expert (CUDA-core, weight streaming)
struct DecodeArgs {
    const void *x;              // [T, d] act storage
    moe_dtype act_dt;
    int T, d, E, k, F;
    const void *w_gate, *w_up, *w_down;   // F32 / BF16 arrays, or Q8_0 packed buffers
    moe_dtype w_dt;
    const int32_t *offsets;     // [E+1]
    const int32_t *perm_tok;    // [T*k]
    const float *perm_w;        // [T*k]
    float *h;                   // [T*k, F] fp32 scratch
    float *out;                 // [T, d] fp32 (zeroed beforehand when k == 2)
    float *y;                   // k > 2: [T*k, d] weighted expert outputs (then combined)
    const int32_t *inv;         // [T*k] grouped row of each slot (k > 2)
    uint32_t *status;
    int num_sms;
    cudaEvent_t ev_gateup;      // optional: recorded between the two kernels
};
cudaError_t launch_decode_experts(const DecodeArgs &a, cudaStream_t stream);
// out[t] = sum_j y[inv[t*k+j]] in slot order (k > 2 combine, no atomics)
cudaError_t launch_combine_rows(const float *y, int d, const int32_t *inv, int T, int k, float *out,
                                const uint32_t *status, int num_sms, cudaStream_t stream);

// decode_tc.cu -- expert FFN for few rows per expert on tcgen05 (bf16 only)
struct DecodeTcArgs {
    moe_dtype w_dt;             // MOE_BF16 or MOE_Q4_A64 (packed planes, 4-bit converter warps)
    const void *x;              // [T, d] bf16
    const void *xp;             // [T*k, d] grouped rows of x (unused when gathering): bf16, or
                                //   for 4-bit weights fp16 rows scaled by 2^-xexp[r]
    const int32_t *xexp;        // [T*k] 4-bit weights: exponent of each grouped row's scale
    const void *x_gather;       // non-null: gather token rows from this [T, d] via perm_tok
    const int32_t *perm_tok;    // [T*k] grouped row -> token
    int T, d, E, k, F;
    const void *w_gate, *w_up, *w_down;   // bf16
    const int32_t *offsets;     // [E+1]
    const int32_t *inv;         // [T*k]
    const float *topk_w;        // [T*k]
    const float *perm_w;        // [T*k] routing weight of each grouped row
    float *pgu;                 // gate/up partials [ks_gu][2][T*k][F]
    uint16_t *h;                // h [T*k, F] scratch: bf16, or fp16 h * 2^-2 xexp[r] (4-bit)
    float *pd;                  // down partials [ks_d][T*k][d]
    float *out;                 // [T, d] fp32 (zeroed beforehand when the down kernel adds into it)
    uint32_t *status;
    int num_sms;
    cudaEvent_t ev_gateup;
    uint32_t expire_ns;         // > 0: one bounded wait gives up after this long (test hook)
};
constexpr int kDecodeTcMaxRows = 8192;   // T*k above this uses the CUDA-core kernels
bool decode_tc_capable(int act_dt, int w_dt, int d, int F, int E);
void decode_tc_splits(int T, int d, int E, int k, int F, int w_dt, int *ks_gu, int *ks_d);
// whole-K schedules: gate/up writes h itself; down adds into out (zeroed
// beforehand when k > 1) -- no reduction or combine kernels
bool decode_tc_gateup_fused(int T, int d, int E, int k, int F, int num_sms);
bool decode_tc_down_direct(int T, int d, int E, int k, int F);
// cluster mode (small bf16 batches): CTAs per cluster of the gate/up / down
// kernels, 0 when not used; K splits reduced on chip, h and out written
// directly
int decode_tc_gateup_cluster(int T, int d, int E, int k, int F, int w_dt, int num_sms);
int decode_tc_down_cluster(int T, int d, int E, int k, int F, int w_dt, int num_sms);
// the down kernel adds into out (zeroed beforehand when k > 1)
bool decode_tc_down_into_out(int T, int d, int E, int k, int F, int w_dt, int num_sms);
cudaError_t launch_decode_tc(const DecodeTcArgs &a, cudaStream_t stream);

// decode_fused.cu -- the decode expert FFN in one persistent launch (bf16,
// k <= 2, whole-K items): gate/up, SwiGLU, down and combine
struct DecodeFusedArgs {
    const void *x;              // [T, d] bf16 (token rows gathered through perm_tok)
    const int32_t *perm_tok;    // [T*k] grouped row -> token
    int T, d, E, k, F;
    const void *w_gate, *w_up, *w_down;   // bf16
    const int32_t *offsets;     // [E+1]
    const float *perm_w;        // [T*k] routing weight of each grouped row
    uint16_t *h;                // bf16 h [T*k, F] scratch
    uint32_t *flags;            // decode_fused_flag_words() words, zero at launch
    float *out;                 // [T, d] fp32 (zeroed beforehand when k == 2)
    uint32_t *status;
    int num_sms;
    cudaEvent_t ev_done;        // optional: recorded after the launch
    uint32_t expire_ns;         // > 0: one bounded wait gives up after this long (test hook)
};
// the shapes the fused kernel takes (beside decode_tc_capable's dtype rules)
bool decode_fused_fits(int T, int d, int E, int k, int F, int num_sms);
// scratch words it needs zeroed before it starts (h-ready flags, ticket counter)
int decode_fused_flag_words(int T, int E, int k, int F);
cudaError_t launch_decode_fused(const DecodeFusedArgs &a, cudaStream_t stream);

// q8.cu
cudaError_t launch_pack_q8_0(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream);
// q8.cu -- affine 4-bit group-64 weights repacked into tiles (codes, fp16 scales, biases)
size_t q4_a64_packed_bytes(long long rows, int cols);   // tiles of 128 rows x 64 columns
size_t q4_k_packed_bytes(long long rows, int cols);     // the same tiles, two groups per row
cudaError_t launch_pack_q4_k(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream);
cudaError_t launch_pack_q4_a64(const void *blocks, long long rows, int cols, void *packed,
                               cudaStream_t stream);
// q8.cu -- Q6_K super-blocks repacked into the 8-bit planes, one scale per 16 values
cudaError_t launch_pack_q6_k(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream);
// q8.cu -- fp8 rows {fp32 scale, E4M3 codes} into the E4M3 plane and fp32 row scales
cudaError_t launch_pack_fp8(const void *rows_in, long long rows, int cols, void *packed,
                            cudaStream_t stream);

}  // namespace moe
