// decode.cu -- expert FFN for decode-sized batches (few rows per expert).
//
// With few rows per expert the layer is bound by reading the active experts'
// weights from HBM (at batch 1 a top-1 layer reads ~1/16 of the experts;
// larger batches touch more distinct experts: "Zyphra-ZONOS2-4bit",
// §Performance notes).  So these kernels stream each active expert's weight
// rows exactly once with 128-bit loads that bypass L1, on CUDA cores in fp32,
// and re-use every loaded weight chunk for up to 8 token rows held in
// registers.
//
// Kernel 1 (gate/up + SwiGLU): work item = (active expert e, tile of 8 ffn
//   rows); warp w owns ffn row f and computes g = W_g[e,f,:] . x_t and
//   u = W_u[e,f,:] . x_t for the expert's rows, then h[r, f] = SiLU(g) * u.
// Kernel 2 (down + routing weight + combine): work item = (active expert e,
//   tile of 8 output columns); warp w owns column o, computes
//   y = W_d[e,o,:] . h[r,:] and adds w_r * y into out[t_r, o] (plain store when
//   k == 1; fp32 atomic add otherwise -- with k == 2 the two addends land on a
//   zeroed word, so the sum is order-independent).
//
// Work items are walked by a grid-stride loop over a list of the experts that
// received rows, built per CTA from the device offsets, so the grid never
// depends on the routing.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kRowBlock = 8;

// List of experts with at least one row, in expert order.  blockDim >= E.
__device__ __forceinline__ int build_active_list(const int32_t *__restrict__ offsets, int E,
                                                 int *act, int *wtot)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = threadIdx.x;
    const bool a = e < E && offsets[e + 1] > offsets[e];
    const unsigned b = __ballot_sync(0xffffffffu, a);
    if (lane == 0) wtot[warp] = __popc(b);
    __syncthreads();
    int before = 0, total = 0;
    for (int w = 0; w < kDecWarps; ++w) {
        if (w < warp) before += wtot[w];
        total += wtot[w];
    }
    if (a) act[before + __popc(b & ((1u << lane) - 1u))] = e;
    __syncthreads();
    return total;
}

__device__ __forceinline__ float dot8(const Chunk8 &a, const Chunk8 &b, float acc)
{
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(a.v[i], b.v[i], acc);
    return acc;
}

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

template <typename AT, typename WT, int NCH>
__global__ void __launch_bounds__(kDecThreads)
decode_gateup_kernel(const AT *__restrict__ x, int d, WView<WT> wg, WView<WT> wu, int F,
                     const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm_tok,
                     int E, float *__restrict__ h)
{
    pdl_enter();
    __shared__ int act[kMaxExperts];
    __shared__ int wtot[kDecWarps];
    const int n_act = build_active_list(offsets, E, act, wtot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ftiles = (F + kDecWarps - 1) / kDecWarps;
    const int items = n_act * ftiles;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int ai = item / ftiles, ft = item - ai * ftiles;
        const int e = act[ai];
        const int row0 = offsets[e], M = offsets[e + 1] - row0;
        const int f = ft * kDecWarps + warp;
        if (f >= F) continue;   // warp-uniform
        const size_t wrow = (size_t)e * F + f;
        for (int rb = 0; rb < M; rb += kRowBlock) {
            float ag[kRowBlock], au[kRowBlock];
            int tok[kRowBlock];
#pragma unroll
            for (int r = 0; r < kRowBlock; ++r) {
                ag[r] = 0.f; au[r] = 0.f;
                tok[r] = rb + r < M ? perm_tok[row0 + rb + r] : -1;
            }
            for (int c0 = lane * 8; c0 < d; c0 += 32 * 8 * NCH) {
                RawW<WT> rg[NCH], ru[NCH];
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
                    if (c < d) { wg.load(wrow, c, rg[j]); wu.load(wrow, c, ru[j]); }
                }
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
                    if (c < d) {
                        Chunk8 g8, u8;
                        WView<WT>::cvt(rg[j], g8);
                        WView<WT>::cvt(ru[j], u8);
#pragma unroll
                        for (int r = 0; r < kRowBlock; ++r) {
                            if (tok[r] >= 0) {
                                Chunk8 xv;
                                load8(x + (size_t)tok[r] * d + c, xv);
                                ag[r] = dot8(g8, xv, ag[r]);
                                au[r] = dot8(u8, xv, au[r]);
                            }
                        }
                    }
                }
            }
            const float gs = warp_transpose_sum8(ag, lane);
            const float us = warp_transpose_sum8(au, lane);
            const int r = transpose8_row(lane);
            if ((lane & 3) == 0 && rb + r < M)
                h[(size_t)(row0 + rb + r) * F + f] = silu(gs) * us;
        }
    }
}

template <typename WT, int NCH>
__global__ void __launch_bounds__(kDecThreads)
decode_down_kernel(const float *__restrict__ h, int F, WView<WT> wd, int d,
                   const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm_tok,
                   const float *__restrict__ perm_w, int E, int k, float *__restrict__ out)
{
    pdl_enter();
    __shared__ int act[kMaxExperts];
    __shared__ int wtot[kDecWarps];
    const int n_act = build_active_list(offsets, E, act, wtot);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int dtiles = (d + kDecWarps - 1) / kDecWarps;
    const int items = n_act * dtiles;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int ai = item / dtiles, dt = item - ai * dtiles;
        const int e = act[ai];
        const int row0 = offsets[e], M = offsets[e + 1] - row0;
        const int o = dt * kDecWarps + warp;
        if (o >= d) continue;
        const size_t wrow = (size_t)e * d + o;
        for (int rb = 0; rb < M; rb += kRowBlock) {
            float acc[kRowBlock];
#pragma unroll
            for (int r = 0; r < kRowBlock; ++r) acc[r] = 0.f;
            const int nr = min(kRowBlock, M - rb);
            for (int c0 = lane * 8; c0 < F; c0 += 32 * 8 * NCH) {
                RawW<WT> rw[NCH];
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
                    if (c < F) wd.load(wrow, c, rw[j]);
                }
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
                    if (c < F) {
                        Chunk8 w8;
                        WView<WT>::cvt(rw[j], w8);
#pragma unroll
                        for (int r = 0; r < kRowBlock; ++r) {
                            if (r < nr) {
                                Chunk8 hv;
                                load8(h + (size_t)(row0 + rb + r) * F + c, hv);
                                acc[r] = dot8(w8, hv, acc[r]);
                            }
                        }
                    }
                }
            }
            const float s = warp_transpose_sum8(acc, lane);
            const int r = transpose8_row(lane);
            if ((lane & 3) == 0 && r < nr) {
                const int row = row0 + rb + r;
                const int t = perm_tok[row];
                const float v = perm_w[row] * s;
                float *dst = out + (size_t)t * d + o;
                if (k == 1) *dst = v;
                else atomicAdd(dst, v);
            }
        }
    }
}

template <typename K>
static int blocks_per_sm(K kern)
{
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kDecThreads, 0) != cudaSuccess
        || n < 1)
        n = 1;
    return n;
}

template <typename AT, typename WT>
static cudaError_t launch_t(const DecodeArgs &a, WView<WT> wg, WView<WT> wu, WView<WT> wd,
                            cudaStream_t stream)
{
    constexpr int NCH_GU = 4, NCH_D = 8;
    auto k1 = decode_gateup_kernel<AT, WT, NCH_GU>;
    auto k2 = decode_down_kernel<WT, NCH_D>;
    static std::atomic<int> occ1{0}, occ2{0};
    if (occ1.load() == 0) occ1.store(blocks_per_sm(k1));
    if (occ2.load() == 0) occ2.store(blocks_per_sm(k2));

    const int n_exp = a.E < a.T * a.k ? a.E : a.T * a.k;   // experts that can be active
    long long items1 = (long long)n_exp * ((a.F + kDecWarps - 1) / kDecWarps);
    long long items2 = (long long)n_exp * ((a.d + kDecWarps - 1) / kDecWarps);
    int g1 = (int)(items1 < (long long)a.num_sms * occ1 ? items1 : (long long)a.num_sms * occ1);
    int g2 = (int)(items2 < (long long)a.num_sms * occ2 ? items2 : (long long)a.num_sms * occ2);
    if (g1 < 1) g1 = 1;
    if (g2 < 1) g2 = 1;
    launch_pdl(k1, dim3(g1), dim3(kDecThreads), 0, stream, static_cast<const AT *>(a.x), a.d, wg, wu, a.F, a.offsets,
                                        a.perm_tok, a.E, a.h);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    if (a.ev_gateup && (err = cudaEventRecord(a.ev_gateup, stream)) != cudaSuccess) return err;
    launch_pdl(k2, dim3(g2), dim3(kDecThreads), 0, stream, a.h, a.F, wd, a.d, a.offsets, a.perm_tok, a.perm_w, a.E,
                                        a.k, a.out);
    return cudaGetLastError();
}

cudaError_t launch_decode_experts(const DecodeArgs &a, cudaStream_t stream)
{
    if (a.w_dt == MOE_F32) {
        WView<float> wg{static_cast<const float *>(a.w_gate), (size_t)a.d};
        WView<float> wu{static_cast<const float *>(a.w_up), (size_t)a.d};
        WView<float> wd{static_cast<const float *>(a.w_down), (size_t)a.F};
        return launch_t<float, float>(a, wg, wu, wd, stream);
    }
    if (a.w_dt == MOE_BF16) {
        WView<__nv_bfloat16> wg{static_cast<const __nv_bfloat16 *>(a.w_gate), (size_t)a.d};
        WView<__nv_bfloat16> wu{static_cast<const __nv_bfloat16 *>(a.w_up), (size_t)a.d};
        WView<__nv_bfloat16> wd{static_cast<const __nv_bfloat16 *>(a.w_down), (size_t)a.F};
        return launch_t<__nv_bfloat16, __nv_bfloat16>(a, wg, wu, wd, stream);
    }
    if (a.w_dt == MOE_Q4_A64) {
        // affine 4-bit packed planes: codes, fp16 scales, fp16 biases
        auto view4 = [](const void *p, long long rows, int cols) {
            WView<Q4Tag> v;
            const char *b = static_cast<const char *>(p);
            v.q = reinterpret_cast<const uint8_t *>(b);
            v.scales = reinterpret_cast<const __half *>(b + q4_a64_scale_offset(rows, cols));
            v.biases = reinterpret_cast<const __half *>(b + q4_a64_bias_offset(rows, cols));
            v.cols = (size_t)cols;
            v.rows = (size_t)rows;
            return v;
        };
        return launch_t<__nv_bfloat16, Q4Tag>(a, view4(a.w_gate, (long long)a.E * a.F, a.d),
                                              view4(a.w_up, (long long)a.E * a.F, a.d),
                                              view4(a.w_down, (long long)a.E * a.d, a.F), stream);
    }
    // Q8_0 packed planes: q plane, then the fp16 scales at align256(rows*cols)
    auto view = [](const void *p, long long rows, int cols) {
        WView<Q8Tag> v;
        v.q = static_cast<const int8_t *>(p);
        v.scales = reinterpret_cast<const __half *>(static_cast<const char *>(p) +
                                                    align_up((size_t)rows * cols, 256));
        v.cols = (size_t)cols;
        v.rows = (size_t)rows;
        return v;
    };
    return launch_t<__nv_bfloat16, Q8Tag>(a, view(a.w_gate, (long long)a.E * a.F, a.d),
                                          view(a.w_up, (long long)a.E * a.F, a.d),
                                          view(a.w_down, (long long)a.E * a.d, a.F), stream);
}

}  // namespace moe
