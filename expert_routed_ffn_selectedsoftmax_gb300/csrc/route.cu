// route.cu -- router projection + SelectedSoftmax (steps 1-2 of the layer).
//
// Scoring modes (same section): mode 0 is SelectedSoftmax; modes 1 and 2
// apply a softmax over all experts / a sigmoid to the logits first, rank by
// that probability plus the bias and weigh by the probability (no
// renormalisation).
//
// SelectedSoftmax ("New Community Model: ZONOS3-Mini (Zyphra) - #1271",
// §Framework change): experts are ranked by raw router logit plus a
// per-expert selection bias; the top k are kept; the kept experts are weighted
// by the softmax of their logits without the bias.  Ties in the ranking score
// go to the lower expert index.
//
// One CTA handles `tpb` tokens.  Their x rows are widened to fp32 in shared
// memory; each warp owns experts e = warp, warp + 8, ... and computes the
// tpb dot products of W_r[e] with the staged rows (fp32 accumulation), so each
// router row is read once per CTA with 128-bit loads.  Top-k then runs one
// warp per token: each lane holds up to 8 experts' scores and k rounds of a
// warp arg-max pick the winners.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteMaxTpb = 8;

template <typename AT>
__device__ __forceinline__ void load_act8(const AT *p, float *dst);
template <>
__device__ __forceinline__ void load_act8<float>(const float *p, float *dst)
{
    float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    dst[0] = a.x; dst[1] = a.y; dst[2] = a.z; dst[3] = a.w;
    dst[4] = b.x; dst[5] = b.y; dst[6] = b.z; dst[7] = b.w;
}
template <>
__device__ __forceinline__ void load_act8<__nv_bfloat16>(const __nv_bfloat16 *p, float *dst)
{
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    dst[0] = bf16lo(u.x); dst[1] = bf16hi(u.x); dst[2] = bf16lo(u.y); dst[3] = bf16hi(u.y);
    dst[4] = bf16lo(u.z); dst[5] = bf16hi(u.z); dst[6] = bf16lo(u.w); dst[7] = bf16hi(u.w);
}

// 8 consecutive activations as raw storage (bf16: one 16-byte load; fp32: two)
template <typename AT> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
    uint4 a;
    __device__ __forceinline__ void load(const __nv_bfloat16 *p) { a = __ldg(reinterpret_cast<const uint4 *>(p)); }
    __device__ __forceinline__ void cvt(float *f) const
    {
        f[0] = bf16lo(a.x); f[1] = bf16hi(a.x); f[2] = bf16lo(a.y); f[3] = bf16hi(a.y);
        f[4] = bf16lo(a.z); f[5] = bf16hi(a.z); f[6] = bf16lo(a.w); f[7] = bf16hi(a.w);
    }
};
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void load(const float *p)
    {
        a = __ldg(reinterpret_cast<const float4 *>(p));
        b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void cvt(float *f) const
    {
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    }
};

template <typename AT, int TPB>
__global__ void __launch_bounds__(kRouteThreads)
route_kernel(const AT *__restrict__ x, int T, int d, const AT *__restrict__ w_router,
             const float *__restrict__ bias, int E, int k, int32_t *__restrict__ topk_idx,
             float *__restrict__ topk_w, float *__restrict__ out_zero,
             uint32_t *__restrict__ zero_words, int n_zero, int32_t *__restrict__ rank,
             int32_t *__restrict__ tile_cnt, uint32_t *__restrict__ status, int mode)
{
    pdl_enter();
    extern __shared__ float4 smem_f4[];
    float *xs = reinterpret_cast<float *>(smem_f4);            // [TPB][d]
    float *logit = xs + (size_t)TPB * d;                        // [TPB][E]
    __shared__ int sel_s[TPB][kMaxTopK];                        // this CTA's selections

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * TPB;
    const int ntok = min(TPB, T - t0);

    if (status && blockIdx.x == 0 && threadIdx.x == 0) *status = kDevOk;
    // scratch words later kernels count on being zero (split-K semaphores)
    for (int i = blockIdx.x * kRouteThreads + threadIdx.x; i < n_zero; i += gridDim.x * kRouteThreads)
        zero_words[i] = 0u;

    // stage the x rows, widened to fp32
    for (int c = threadIdx.x * 8; c < ntok * d; c += kRouteThreads * 8) {
        int t = c / d, i = c - t * d;
        load_act8<AT>(x + (size_t)(t0 + t) * d + i, xs + (size_t)t * d + i);
    }
    // zero the output rows that the combine step accumulates into
    if (out_zero) {
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = threadIdx.x * 4; c < ntok * d; c += kRouteThreads * 4)
            *reinterpret_cast<float4 *>(out_zero + (size_t)t0 * d + c) = z;
    }
    __syncthreads();

    // router projection: warp w owns experts in groups of EG; each group's
    // router chunks (CG per lane) are loaded together before any use, so a
    // warp waits for one round trip per group rather than one per expert
    constexpr int EG = 4;
    constexpr int CG = sizeof(AT) == 4 ? 2 : 4;
    for (int e0 = warp * EG; e0 < E; e0 += kRouteWarps * EG) {
        float acc[EG][TPB];
#pragma unroll
        for (int g = 0; g < EG; ++g)
#pragma unroll
            for (int t = 0; t < TPB; ++t) acc[g][t] = 0.f;
        for (int c0 = lane * 8; c0 < d; c0 += 256 * CG) {
            Raw8<AT> raw[EG][CG];
#pragma unroll
            for (int g = 0; g < EG; ++g)
#pragma unroll
                for (int q = 0; q < CG; ++q) {
                    const int i = c0 + q * 256;
                    if (e0 + g < E && i < d) raw[g][q].load(w_router + (size_t)(e0 + g) * d + i);
                }
#pragma unroll
            for (int g = 0; g < EG; ++g) {
#pragma unroll
                for (int q = 0; q < CG; ++q) {
                    const int i = c0 + q * 256;
                    if (e0 + g < E && i < d) {
                        float wv[8];
                        raw[g][q].cvt(wv);
#pragma unroll
                        for (int t = 0; t < TPB; ++t) {
                            if (t < ntok) {
                                const float4 *xp = reinterpret_cast<const float4 *>(xs + (size_t)t * d + i);
                                const float4 a = xp[0], b = xp[1];
                                float s = acc[g][t];
                                s = fmaf(wv[0], a.x, s); s = fmaf(wv[1], a.y, s);
                                s = fmaf(wv[2], a.z, s); s = fmaf(wv[3], a.w, s);
                                s = fmaf(wv[4], b.x, s); s = fmaf(wv[5], b.y, s);
                                s = fmaf(wv[6], b.z, s); s = fmaf(wv[7], b.w, s);
                                acc[g][t] = s;
                            }
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int g = 0; g < EG; ++g)
#pragma unroll
            for (int t = 0; t < TPB; ++t) {
                const float s = warp_sum(acc[g][t]);
                if (lane == 0 && t < ntok && e0 + g < E) logit[t * E + e0 + g] = s;
            }
    }
    __syncthreads();

    // ranking and weights: one warp per token.  lg holds what the weights are
    // made of: the logit (mode 0, softmax over the selected later) or the
    // probability (modes 1, 2)
    for (int t = warp; t < ntok; t += kRouteWarps) {
        float sc[8], lg[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            int e = lane + 32 * s;
            lg[s] = e < E ? logit[t * E + e] : 0.f;
        }
        if (mode == 1) {   // softmax over all E: lane partials, xor-shuffle trees
            float m = -INFINITY;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (lane + 32 * s < E) m = fmaxf(m, lg[s]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            float den = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s)
                if (lane + 32 * s < E) den += expf(lg[s] - m);
            den = warp_sum(den);
#pragma unroll
            for (int s = 0; s < 8; ++s) lg[s] = expf(lg[s] - m) / den;
        } else if (mode == 2) {
#pragma unroll
            for (int s = 0; s < 8; ++s) lg[s] = 1.0f / (1.0f + expf(-lg[s]));
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            int e = lane + 32 * s;
            if (e < E) {
                sc[s] = lg[s] + (bias ? bias[e] : 0.f);
                if (isnan(sc[s])) sc[s] = -INFINITY;   // keep the ranking a total order
            } else {
                sc[s] = -INFINITY;
            }
        }
        unsigned taken = 0;   // bit s: slot s of this lane already selected
        int sel_e[kMaxTopK];
        float sel_l[kMaxTopK];
        for (int j = 0; j < k; ++j) {
            // this lane's best remaining: highest score, then lowest index
            float bs = -INFINITY;
            int be = 0x7fffffff;
            float bl = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                int e = lane + 32 * s;
                bool ok = e < E && !((taken >> s) & 1u);
                if (ok && (sc[s] > bs || (sc[s] == bs && e < be))) {
                    bs = sc[s]; be = e; bl = lg[s];
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                float os = __shfl_xor_sync(0xffffffffu, bs, o);
                int oe = __shfl_xor_sync(0xffffffffu, be, o);
                float ol = __shfl_xor_sync(0xffffffffu, bl, o);
                if (os > bs || (os == bs && oe < be)) { bs = os; be = oe; bl = ol; }
            }
            if ((be & 31) == lane) taken |= 1u << (be >> 5);
            sel_e[j] = be;
            sel_l[j] = bl;
        }
        if (lane == 0) {
            float p[kMaxTopK], den = 1.f;
            if (mode == 0) {   // softmax over the selected logits
                float m = sel_l[0];
                for (int j = 1; j < k; ++j) m = fmaxf(m, sel_l[j]);
                den = 0.f;
                for (int j = 0; j < k; ++j) { p[j] = expf(sel_l[j] - m); den += p[j]; }
            } else {
                for (int j = 0; j < k; ++j) p[j] = sel_l[j];
            }
            const size_t base = (size_t)(t0 + t) * k;
            for (int j = 0; j < k; ++j) {
                topk_idx[base + j] = sel_e[j];
                topk_w[base + j] = mode == 0 ? p[j] / den : p[j];
                sel_s[t][j] = sel_e[j];
            }
        }
    }
    if (!rank) return;
    // grouping inputs: per-expert count of this CTA's tokens, and each slot's
    // stable rank among them (tokens of a CTA are consecutive)
    __syncthreads();
    for (int i = threadIdx.x; i < ntok * k; i += kRouteThreads) {
        const int t = i / k, e = sel_s[t][i - t * k];
        int rk = 0;
        for (int u = 0; u < t; ++u)
            for (int j = 0; j < k; ++j) rk += sel_s[u][j] == e;
        rank[(size_t)t0 * k + i] = rk;
    }
    for (int e = threadIdx.x; e < E; e += kRouteThreads) {
        int cnt = 0;
        for (int u = 0; u < ntok; ++u)
            for (int j = 0; j < k; ++j) cnt += sel_s[u][j] == e;
        tile_cnt[(size_t)blockIdx.x * E + e] = cnt;
    }
}

size_t route_smem_bytes(int tpb, int d, int E)
{
    return sizeof(float) * ((size_t)tpb * d + (size_t)tpb * E);
}

int route_tokens_per_block(int T, int d, int E)
{
    // keep the staged rows within ~96 KB; small T favours many CTAs
    int tpb = kRouteMaxTpb;
    while (tpb > 1 && route_smem_bytes(tpb, d, E) > 96 * 1024) tpb >>= 1;
    const int sms = device_sm_count();
    while (tpb > 1 && (T + tpb - 1) / tpb < 2 * sms) tpb >>= 1;
    return tpb;
}

template <typename AT, int TPB>
static cudaError_t launch_route_t(const void *x, int T, int d, const void *w_router,
                                  const float *bias, int E, int k, int32_t *topk_idx,
                                  float *topk_w, float *out_zero, uint32_t *zero_words,
                                  int n_zero, int32_t *rank, int32_t *tile_cnt, uint32_t *status,
                                  int mode, cudaStream_t stream)
{
    size_t smem = route_smem_bytes(TPB, d, E);
    auto kern = route_kernel<AT, TPB>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((T + TPB - 1) / TPB);
    launch_pdl(kern, dim3(grid), dim3(kRouteThreads), smem, stream, static_cast<const AT *>(x), T, d,
                                                 static_cast<const AT *>(w_router), bias, E, k,
                                                 topk_idx, topk_w, out_zero, zero_words, n_zero,
                                                 rank, tile_cnt, status, mode);
    return cudaGetLastError();
}

cudaError_t launch_route(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                         const float *bias, int E, int k, int32_t *topk_idx, float *topk_w,
                         float *out_zero, uint32_t *zero_words, int n_zero, int32_t *rank,
                         int32_t *tile_cnt, uint32_t *status, int mode, cudaStream_t stream)
{
    int tpb = route_tokens_per_block(T, d, E);
    if (act_dt == MOE_F32) {
        switch (tpb) {
        case 8: return launch_route_t<float, 8>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
        case 4: return launch_route_t<float, 4>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
        case 2: return launch_route_t<float, 2>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
        default: return launch_route_t<float, 1>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
        }
    }
    switch (tpb) {
    case 8: return launch_route_t<__nv_bfloat16, 8>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
    case 4: return launch_route_t<__nv_bfloat16, 4>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
    case 2: return launch_route_t<__nv_bfloat16, 2>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
    default: return launch_route_t<__nv_bfloat16, 1>(x, T, d, w_router, bias, E, k, topk_idx, topk_w, out_zero, zero_words, n_zero, rank, tile_cnt, status, mode, stream);
    }
}

}  // namespace moe
