// tc_gemm.h -- internal interface of the tcgen05 grouped-GEMM expert path.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

struct TcArgs {
    const void *x;              // [T, d] bf16
    int T, d, E, k, F;
    const void *w_gate, *w_up, *w_down;   // BF16 arrays, or Q8_0 packed buffers
    moe_dtype w_dt;
    const int32_t *offsets;     // [E+1]
    const int32_t *perm_tok;    // [T*k]
    const float *perm_w;        // [T*k]
    void *xp;                   // [T*k, d] 16-bit scratch (grouped rows)
    int32_t *xexp;              // [T*k] Q8_0: fp16 row r of xp is x * 2^-xexp[r]
    int xp_ready;               // xp already holds the grouped rows
    void *h;                    // [T*k, F] 16-bit scratch
    float *out;                 // [T, d] fp32
    float *y;                   // k > 2: [T*k, d] weighted outputs per grouped row (then combined)
    const int32_t *inv;         // [T*k] grouped row of each slot (k > 2)
    int zero_out;               // zero `out` in the gate/up kernel (the down kernel adds into it)
    uint32_t *status;           // device status word
    int num_sms;
    cudaEvent_t ev_gathered;    // optional: recorded after the row gather
    cudaEvent_t ev_gateup;      // optional: recorded after the gate/up GEMM
    uint32_t expire_ns;         // > 0: one bounded wait gives up after this long (test hook)
};

namespace tc {
// 2-D row-major [rows, cols] 16-bit tensor map, box {64 cols, box_rows},
// 128-byte swizzle (the K-major operand tiles of the tcgen05 kernels).
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              CUtensorMapDataType dt);
// 2-D row-major [rows, cols] int8 tensor map, box {64 cols, box_rows}, no
// swizzle or (swizzle64) the 64-byte swizzle: 16-byte chunk c of row r at
// c ^ ((r >> 1) & 3).
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 bool swizzle64 = false);
// The fp16 scale plane [cols/group, rows] of an 8-bit packed buffer (Q8_0:
// group 32, Q6_K: 16), box {box_rows rows, 64/group blocks}.
bool make_scale_map(CUtensorMap *m, const void *packed, uint64_t rows, uint64_t cols, int group,
                    uint32_t box_rows);
}  // namespace tc

// True when the tensor-core expert kernels are compiled into this library.
bool tc_gemm_available();
// True when the tensor-core expert kernels handle this weight storage type.
bool tc_gemm_supports(moe_dtype w_dt);
// Shape heuristic: prefer the grouped GEMMs over the decode kernels.
bool tc_gemm_prefer(int T, int d, int E, int k, int F);
// True when the grouped GEMMs for weights of type w_dt run as CTA pairs.
bool tc_gemm_pairs(moe_dtype w_dt);
cudaError_t launch_tc_experts(const TcArgs &a, cudaStream_t stream);

}  // namespace moe
