// kernels.h -- internal launchers of the library's kernels (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// route.cu
size_t route_smem_bytes(int tpb, int d, int E);
cudaError_t launch_route(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                         const float *bias, int E, int k, int32_t *topk_idx, float *topk_w,
                         float *out_zero, uint32_t *status, cudaStream_t stream);

// permute.cu
cudaError_t launch_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                           int32_t *offsets, int32_t *perm_tok, int32_t *inv,
                           const float *topk_w, float *perm_w, uint32_t *status,
                           cudaStream_t stream);
cudaError_t launch_gather_rows(const void *x, int d, const int32_t *perm_tok, int rows,
                               void *xp, int to_fp16, int num_sms, cudaStream_t stream);

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
    float *out;                 // [T, d] fp32 (zeroed beforehand when k > 1)
    int num_sms;
    cudaEvent_t ev_gateup;      // optional: recorded between the two kernels
};
cudaError_t launch_decode_experts(const DecodeArgs &a, cudaStream_t stream);

// q8.cu
cudaError_t launch_pack_q8_0(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream);

}  // namespace moe
