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
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDecThreads = 256;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kRowBlock = 8;

// List of experts with at least one row, in expert order.  blockDim >= E.
// (Debug builds: none when the offsets are inconsistent, see debug_offsets_ok.)
__device__ __forceinline__ int build_active_list(const int32_t *__restrict__ offsets, int E,
                                                 int *act, int *wtot, int rows, uint32_t *status)
{
    if (!debug_offsets_ok(offsets, E, rows, status)) return 0;
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

// RPW: weight rows per warp.  Each token chunk loaded into registers is used
// for all RPW rows, and a lane has RPW x NCH weight chunks in flight: for
// narrow weight encodings (4-bit codes, 4 bytes per 8 values) one row per warp
// leaves the loads dominated by re-reads of the token rows.
template <typename AT, typename WT, int NCH, int RPW>
__global__ void __launch_bounds__(kDecThreads)
decode_gateup_kernel(const AT *__restrict__ x, int d, WView<WT> wg, WView<WT> wu, int F,
                     const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm_tok,
                     int E, float *__restrict__ h, int rows, int T, uint32_t *status)
{
    pdl_enter();
    __shared__ int act[kMaxExperts];
    __shared__ int wtot[kDecWarps];
    const int n_act = build_active_list(offsets, E, act, wtot, rows, status);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int ROWS = kDecWarps * RPW;     // ffn rows per work item
    const int ftiles = (F + ROWS - 1) / ROWS;
    const int items = n_act * ftiles;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int ai = item / ftiles, ft = item - ai * ftiles;
        const int e = act[ai];
        const int row0 = offsets[e], M = offsets[e + 1] - row0;
        const int f0 = ft * ROWS + warp * RPW;  // this warp's rows f0 .. f0 + RPW - 1
        if (f0 >= F) continue;   // warp-uniform
        const size_t wrow = (size_t)e * F + f0;
        for (int rb = 0; rb < M; rb += kRowBlock) {
            float ag[RPW][kRowBlock], au[RPW][kRowBlock];
            int tok[kRowBlock];
#pragma unroll
            for (int r = 0; r < kRowBlock; ++r) {
#pragma unroll
                for (int i = 0; i < RPW; ++i) { ag[i][r] = 0.f; au[i][r] = 0.f; }
                int t = -1;
                if (rb + r < M) {
                    t = perm_tok[row0 + rb + r];
                    if (!debug_index_ok(t, T, status)) t = -1;   // (debug builds)
                }
                tok[r] = t;
            }
            for (int c0 = lane * 8; c0 < d; c0 += 32 * 8 * NCH) {
                RawW<WT> rg[RPW][NCH], ru[RPW][NCH];
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
#pragma unroll
                    for (int i = 0; i < RPW; ++i)
                        if (c < d && f0 + i < F) { wg.load(wrow + i, c, rg[i][j]); wu.load(wrow + i, c, ru[i][j]); }
                }
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
                    if (c < d) {
                        Chunk8 g8[RPW], u8[RPW];
#pragma unroll
                        for (int i = 0; i < RPW; ++i) {
                            WView<WT>::cvt(rg[i][j], g8[i]);
                            WView<WT>::cvt(ru[i][j], u8[i]);
                        }
#pragma unroll
                        for (int r = 0; r < kRowBlock; ++r) {
                            if (tok[r] >= 0) {
                                Chunk8 xv;
                                load8(x + (size_t)tok[r] * d + c, xv);
#pragma unroll
                                for (int i = 0; i < RPW; ++i) {
                                    ag[i][r] = dot8(g8[i], xv, ag[i][r]);
                                    au[i][r] = dot8(u8[i], xv, au[i][r]);
                                }
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float gs = warp_transpose_sum8(ag[i], lane);
                const float us = warp_transpose_sum8(au[i], lane);
                const int r = transpose8_row(lane);
                if ((lane & 3) == 0 && rb + r < M && f0 + i < F)
                    h[(size_t)(row0 + rb + r) * F + f0 + i] = silu(gs) * us;
            }
        }
    }
}

template <typename WT, int NCH, int RPW>
__global__ void __launch_bounds__(kDecThreads)
decode_down_kernel(const float *__restrict__ h, int F, WView<WT> wd, int d,
                   const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm_tok,
                   const float *__restrict__ perm_w, int E, int k, float *__restrict__ out,
                   float *__restrict__ y, int rows, int T, uint32_t *status)
{
    pdl_enter();
    __shared__ int act[kMaxExperts];
    __shared__ int wtot[kDecWarps];
    const int n_act = build_active_list(offsets, E, act, wtot, rows, status);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int COLS = kDecWarps * RPW;     // output columns per work item
    const int dtiles = (d + COLS - 1) / COLS;
    const int items = n_act * dtiles;

    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const int ai = item / dtiles, dt = item - ai * dtiles;
        const int e = act[ai];
        const int row0 = offsets[e], M = offsets[e + 1] - row0;
        const int o0 = dt * COLS + warp * RPW;  // this warp's columns o0 .. o0 + RPW - 1
        if (o0 >= d) continue;
        const size_t wrow = (size_t)e * d + o0;
        for (int rb = 0; rb < M; rb += kRowBlock) {
            float acc[RPW][kRowBlock];
#pragma unroll
            for (int i = 0; i < RPW; ++i)
#pragma unroll
                for (int r = 0; r < kRowBlock; ++r) acc[i][r] = 0.f;
            const int nr = min(kRowBlock, M - rb);
            for (int c0 = lane * 8; c0 < F; c0 += 32 * 8 * NCH) {
                RawW<WT> rw[RPW][NCH];
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
#pragma unroll
                    for (int i = 0; i < RPW; ++i)
                        if (c < F && o0 + i < d) wd.load(wrow + i, c, rw[i][j]);
                }
#pragma unroll
                for (int j = 0; j < NCH; ++j) {
                    const int c = c0 + j * 256;
                    if (c < F) {
                        Chunk8 w8[RPW];
#pragma unroll
                        for (int i = 0; i < RPW; ++i) WView<WT>::cvt(rw[i][j], w8[i]);
#pragma unroll
                        for (int r = 0; r < kRowBlock; ++r) {
                            if (r < nr) {
                                Chunk8 hv;
                                load8(h + (size_t)(row0 + rb + r) * F + c, hv);
#pragma unroll
                                for (int i = 0; i < RPW; ++i) acc[i][r] = dot8(w8[i], hv, acc[i][r]);
                            }
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float s = warp_transpose_sum8(acc[i], lane);
                const int r = transpose8_row(lane);
                if ((lane & 3) == 0 && r < nr && o0 + i < d) {
                    const int row = row0 + rb + r;
                    const float v = perm_w[row] * s;
                    if (k > 2) {
                        // the grouped row's weighted output; combine_rows_kernel adds
                        // each token's k rows in slot order
                        y[(size_t)row * d + o0 + i] = v;
                    } else {
                        // k = 1: the only contribution; k = 2: two additions onto
                        // zero, whose result does not depend on their order
                        const int t = perm_tok[row];
                        if (debug_index_ok(t, T, status)) {   // (debug builds)
                            float *dst = out + (size_t)t * d + o0 + i;
                            if (k == 1) *dst = v;
                            else atomicAdd(dst, v);
                        }
                    }
                }
            }
        }
    }
}

// out[t, :] = sum_j y[inv[t, j], :] over the k slots of token t in slot order
// (y holds each grouped row's routing-weighted expert output): the combine of
// k > 2 experts without atomics, so results do not depend on timing.
__global__ void __launch_bounds__(256)
combine_rows_kernel(const float *__restrict__ y, int d, const int32_t *__restrict__ inv, int T,
                    int k, float *__restrict__ out, const uint32_t *status)
{
    pdl_enter();
    if (upstream_failed(status)) return;
    const int vec = d / 4;
    const long long total = (long long)T * vec;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / vec), o = (int)(i - (long long)t * vec) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(y + (size_t)inv[t * k + j] * d + o));
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        *reinterpret_cast<float4 *>(out + (size_t)t * d + o) = acc;
    }
}

cudaError_t launch_combine_rows(const float *y, int d, const int32_t *inv, int T, int k, float *out,
                                const uint32_t *status, int num_sms, cudaStream_t stream)
{
    long long blocks = ((long long)T * (d / 4) + 255) / 256;
    const long long cap = (long long)num_sms * 8;
    if (blocks > cap) blocks = cap;
    launch_pdl(combine_rows_kernel, dim3((unsigned)(blocks < 1 ? 1 : blocks)), dim3(256), 0, stream, y,
               d, inv, T, k, out, status);
    return cudaGetLastError();
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

template <typename AT, typename WT, int NCH, int RPW>
static cudaError_t launch_gateup(const DecodeArgs &a, WView<WT> wg, WView<WT> wu, cudaStream_t stream)
{
    auto k1 = decode_gateup_kernel<AT, WT, NCH, RPW>;
    static PerDeviceInt occ_cache;
    const int dev = current_device();
    int occ = occ_cache.get(dev);
    if (occ <= 0) { occ = blocks_per_sm(k1); occ_cache.put(dev, occ); }
    const int n_exp = a.E < a.T * a.k ? a.E : a.T * a.k;   // experts that can be active
    const long long items = (long long)n_exp * ((a.F + kDecWarps * RPW - 1) / (kDecWarps * RPW));
    int g = (int)(items < (long long)a.num_sms * occ ? items : (long long)a.num_sms * occ);
    if (g < 1) g = 1;
    launch_pdl(k1, dim3(g), dim3(kDecThreads), 0, stream, static_cast<const AT *>(a.x), a.d, wg, wu,
               a.F, a.offsets, a.perm_tok, a.E, a.h, a.T * a.k, a.T, a.status);
    return cudaGetLastError();
}

template <typename WT, int NCH, int RPW>
static cudaError_t launch_down(const DecodeArgs &a, WView<WT> wd, cudaStream_t stream)
{
    auto k2 = decode_down_kernel<WT, NCH, RPW>;
    static PerDeviceInt occ_cache;
    const int dev = current_device();
    int occ = occ_cache.get(dev);
    if (occ <= 0) { occ = blocks_per_sm(k2); occ_cache.put(dev, occ); }
    const int n_exp = a.E < a.T * a.k ? a.E : a.T * a.k;
    const long long items = (long long)n_exp * ((a.d + kDecWarps * RPW - 1) / (kDecWarps * RPW));
    int g = (int)(items < (long long)a.num_sms * occ ? items : (long long)a.num_sms * occ);
    if (g < 1) g = 1;
    launch_pdl(k2, dim3(g), dim3(kDecThreads), 0, stream, a.h, a.F, wd, a.d, a.offsets, a.perm_tok,
               a.perm_w, a.E, a.k, a.out, a.y, a.T * a.k, a.T, a.status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess || a.k <= 2) return err;
    return launch_combine_rows(a.y, a.d, a.inv, a.T, a.k, a.out, a.status, a.num_sms, stream);
}

template <typename AT, typename WT>
static cudaError_t launch_t(const DecodeArgs &a, WView<WT> wg, WView<WT> wu, WView<WT> wd,
                            cudaStream_t stream)
{
    cudaError_t err;
    // 4-bit codes: several rows per warp (see decode_gateup_kernel) when the
    // wider items still give every SM two of them; wider types: one row
    const int n_exp = a.E < a.T * a.k ? a.E : a.T * a.k;
    const long long two_per_sm = 2LL * a.num_sms;
    if constexpr (std::is_same<WT, Q4Tag>::value) {
        err = (long long)n_exp * ((a.F + 2 * kDecWarps - 1) / (2 * kDecWarps)) >= two_per_sm
                  ? launch_gateup<AT, WT, 2, 2>(a, wg, wu, stream)
                  : launch_gateup<AT, WT, 4, 1>(a, wg, wu, stream);
    } else {
        err = launch_gateup<AT, WT, 4, 1>(a, wg, wu, stream);
    }
    if (err != cudaSuccess) return err;
    if (a.ev_gateup && (err = cudaEventRecord(a.ev_gateup, stream)) != cudaSuccess) return err;
    if constexpr (std::is_same<WT, Q4Tag>::value) {
        return (long long)n_exp * ((a.d + 4 * kDecWarps - 1) / (4 * kDecWarps)) >= two_per_sm
                   ? launch_down<WT, 4, 4>(a, wd, stream)
                   : launch_down<WT, 8, 1>(a, wd, stream);
    }
    return launch_down<WT, 8, 1>(a, wd, stream);
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
    if (is_q4(a.w_dt)) {
        // 4-bit packed tiles of 128 rows x 64 columns (affine 4-bit, Q4_K)
        const int gpr = q4_gpr(a.w_dt);
        auto view4 = [gpr](const void *p, long long rows, int cols) {
            (void)rows;
            WView<Q4Tag> v;
            v.q = static_cast<const uint8_t *>(p);
            v.groups = cols / 64;
            v.gpr = gpr;
            return v;
        };
        return launch_t<__nv_bfloat16, Q4Tag>(a, view4(a.w_gate, (long long)a.E * a.F, a.d),
                                              view4(a.w_up, (long long)a.E * a.F, a.d),
                                              view4(a.w_down, (long long)a.E * a.d, a.F), stream);
    }
    if (is_fp8(a.w_dt)) {
        // fp8 planes: E4M3 plane, then the fp32 row scales at align256(rows*cols)
        auto view8 = [](const void *p, long long rows, int cols) {
            WView<F8Tag> v;
            v.q = static_cast<const uint8_t *>(p);
            v.scales = reinterpret_cast<const float *>(static_cast<const char *>(p) +
                                                       align_up((size_t)rows * cols, 256));
            v.cols = (size_t)cols;
            return v;
        };
        return launch_t<__nv_bfloat16, F8Tag>(a, view8(a.w_gate, (long long)a.E * a.F, a.d),
                                              view8(a.w_up, (long long)a.E * a.F, a.d),
                                              view8(a.w_down, (long long)a.E * a.d, a.F), stream);
    }
    // Q8_0 / Q6_K packed planes: q plane, then the fp16 scales at align256(rows*cols)
    const int group = q8_group(a.w_dt);
    auto view = [group](const void *p, long long rows, int cols) {
        WView<Q8Tag> v;
        v.group = group;
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
