// permute.cu -- token grouping (step 3): per-expert histogram, exclusive scan
// and a stable permutation of the T*k routed slots, integer-exact and free of
// atomics; plus the row gather that lays x out in grouped order for the
// grouped GEMMs.
//
// Grouped expert compute is what ggml's mul_mat_id provides for the ZONOS2
// port ("zonos2.cpp internals", §Performance); the grouping here is its
// explicit form.
//
// One CTA of 8-32 warps (more for more slots).  Warp w owns the contiguous flat-slot range
// [w*chunk, (w+1)*chunk).  Pass 1: each warp counts its range per expert
// (__match_any_sync finds the lanes sharing an expert; the lowest of them adds
// the group size to the warp's private counter).  Scan: counts, exclusive
// offsets, and per-(warp, expert) bases in warp order.  Pass 2: each lane's
// destination = base + (lanes below it with the same expert); the group
// leader then advances the base.  Slots therefore land in increasing flat order
// within each expert (a stable sort by expert id).
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kPermMaxWarps = 32;

__global__ void __launch_bounds__(kPermMaxWarps * 32)
permute_kernel(const int32_t *__restrict__ topk_idx, int n, int k, int E,
               int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
               int32_t *__restrict__ perm_tok, int32_t *__restrict__ inv,
               const float *__restrict__ topk_w, float *__restrict__ perm_w,
               uint32_t *__restrict__ status)
{
    pdl_enter();
    __shared__ int32_t wcnt[kPermMaxWarps][kMaxExperts];
    __shared__ int32_t cnt_s[kMaxExperts];
    __shared__ int32_t off_s[kMaxExperts + 1];

    if (upstream_failed(status)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;          // >= 8, so blockDim >= E
    const unsigned lt_mask = (1u << lane) - 1u;
    const int chunk = (n + nwarps - 1) / nwarps;
    const int begin = min(n, warp * chunk), end = min(n, begin + chunk);

    for (int i = threadIdx.x; i < nwarps * kMaxExperts; i += blockDim.x)
        (&wcnt[0][0])[i] = 0;
    __syncthreads();

    bool bad = false;
    // pass 1: warp-private histograms
    for (int base = begin; base < end; base += 32) {
        int i = base + lane;
        int e = i < end ? topk_idx[i] : -1;
        if (i < end && (e < 0 || e >= E)) { bad = true; e = -1; }
        unsigned peers = __match_any_sync(0xffffffffu, e);
        int leader = __ffs(peers) - 1;
        if (e >= 0 && lane == leader) wcnt[warp][e] += __popc(peers);
    }
    __syncthreads();

    // scan: per-expert totals, exclusive offsets, per-warp bases
    if (threadIdx.x < E) {
        int e = threadIdx.x, s = 0;
        for (int w = 0; w < nwarps; ++w) s += wcnt[w][e];
        cnt_s[e] = s;
    }
    __syncthreads();
    if (warp == 0) {
        // lane l scans bins [l*per, (l+1)*per)
        const int per = (E + 31) / 32;
        int local = 0;
        for (int j = 0; j < per; ++j) {
            int e = lane * per + j;
            if (e < E) local += cnt_s[e];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int j = 0; j < per; ++j) {
            int e = lane * per + j;
            if (e < E) { off_s[e] = run; run += cnt_s[e]; }
        }
        if (lane == 31) off_s[E] = incl;
    }
    __syncthreads();
    if (threadIdx.x < E) {
        int e = threadIdx.x, run = off_s[e];
        counts[e] = cnt_s[e];
        offsets[e] = off_s[e];
        for (int w = 0; w < nwarps; ++w) {
            int c = wcnt[w][e];
            wcnt[w][e] = run;
            run += c;
        }
    }
    if (threadIdx.x == 0) offsets[E] = off_s[E];
    __syncthreads();

    // pass 2: stable scatter
    for (int base = begin; base < end; base += 32) {
        int i = base + lane;
        int e = i < end ? topk_idx[i] : -1;
        if (e < 0 || e >= E) e = -1;
        unsigned peers = __match_any_sync(0xffffffffu, e);
        int leader = __ffs(peers) - 1;
        int pos = 0;
        if (e >= 0) pos = wcnt[warp][e] + __popc(peers & lt_mask);
        __syncwarp();
        if (e >= 0) {
            if (lane == leader) wcnt[warp][e] += __popc(peers);
            perm_tok[pos] = i / k;
            inv[i] = pos;
            if (perm_w) perm_w[pos] = topk_w[i];
        }
        __syncwarp();
    }
    if (bad) flag_status(status, kDevCheckFailed);
}

cudaError_t launch_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                           int32_t *offsets, int32_t *perm_tok, int32_t *inv,
                           const float *topk_w, float *perm_w, uint32_t *status,
                           cudaStream_t stream)
{
    // about 64 slots per warp, between 8 and 32 warps
    const int n = T * k;
    int warps = (n + 63) / 64;
    warps = warps < 8 ? 8 : (warps > kPermMaxWarps ? kPermMaxWarps : warps);
    launch_pdl(permute_kernel, dim3(1), dim3(warps * 32), 0, stream, topk_idx, T * k, k, E, counts, offsets,
                                                   perm_tok, inv, topk_w, perm_w, status);
    return cudaGetLastError();
}

// xp[r, :] = x[perm_tok[r], :] (bf16 rows); with to_fp16 the rows are
// re-encoded as fp16 for the fp16 tensor-core path of Q8_0 experts, each
// scaled by 2^-xexp[r] (fp16_row_exponent), one warp per row.
__global__ void gather_rows_kernel(const uint16_t *__restrict__ x, int d,
                                   const int32_t *__restrict__ perm_tok, int rows,
                                   uint16_t *__restrict__ xp, int to_fp16, int32_t *__restrict__ xexp,
                                   int T, uint32_t *__restrict__ status)
{
    pdl_enter();
    const int vec_per_row = d / 8;
    if (to_fp16) {
        const int lane = threadIdx.x & 31;
        const int wpb = blockDim.x / 32;
        for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < rows; r += gridDim.x * wpb) {
            int t = perm_tok[r];
            if (!debug_index_ok(t, T, status)) t = 0;   // (debug builds)
            const uint16_t *src = x + (size_t)t * d;
            const int e = fp16_row_exponent(src, d, lane);
            if (lane == 0) xexp[r] = e;
            for (int c = lane; c < vec_per_row; c += 32)
                reinterpret_cast<uint4 *>(xp + (size_t)r * d)[c] =
                    bf16x8_to_fp16_scaled(__ldg(reinterpret_cast<const uint4 *>(src) + c), e);
        }
        return;
    }
    const long long total = (long long)rows * vec_per_row;
    for (long long v = blockIdx.x * (long long)blockDim.x + threadIdx.x; v < total;
         v += (long long)gridDim.x * blockDim.x) {
        int r = (int)(v / vec_per_row), c = (int)(v - (long long)r * vec_per_row);
        int t = perm_tok[r];
        if (!debug_index_ok(t, T, status)) t = 0;   // (debug builds)
        uint4 u = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)t * d) + c);
        reinterpret_cast<uint4 *>(xp + (size_t)r * d)[c] = u;
    }
}

// Routing and grouping of a dense layer (one expert, k = 1): every token to
// expert 0 with weight 1 -- the softmax of a single logit -- and grouped row
// r = token r.  Written directly instead of running a router whose answer is
// fixed.
__global__ void identity_grouping_kernel(int T, int32_t *__restrict__ topk_idx,
                                         float *__restrict__ topk_w, int32_t *__restrict__ counts,
                                         int32_t *__restrict__ offsets, int32_t *__restrict__ perm_tok,
                                         int32_t *__restrict__ inv, float *__restrict__ perm_w,
                                         uint32_t *__restrict__ status, uint32_t *__restrict__ zero_words,
                                         int n_zero)
{
    pdl_enter();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_zero; i += gridDim.x * blockDim.x)
        zero_words[i] = 0u;
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (status) *status = kDevOk;
        counts[0] = T;
        offsets[0] = 0;
        offsets[1] = T;
    }
    for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < T; r += gridDim.x * blockDim.x) {
        topk_idx[r] = 0;
        topk_w[r] = 1.0f;
        perm_tok[r] = r;
        inv[r] = r;
        perm_w[r] = 1.0f;
    }
}

cudaError_t launch_identity_grouping(int T, int32_t *topk_idx, float *topk_w, int32_t *counts,
                                     int32_t *offsets, int32_t *perm_tok, int32_t *inv,
                                     float *perm_w, uint32_t *status, uint32_t *zero_words,
                                     int n_zero, int num_sms, cudaStream_t stream)
{
    long long want = ((long long)T + 255) / 256, cap = (long long)num_sms * 4;
    int blocks = (int)(want < cap ? want : cap);
    if (blocks < 1) blocks = 1;
    launch_pdl(identity_grouping_kernel, dim3(blocks), dim3(256), 0, stream, T, topk_idx, topk_w,
               counts, offsets, perm_tok, inv, perm_w, status, zero_words, n_zero);
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void *x, int d, const int32_t *perm_tok, int rows,
                               void *xp, int to_fp16, int32_t *xexp, int T, uint32_t *status,
                               int num_sms, cudaStream_t stream)
{
    long long total = (long long)rows * (d / 8);
    long long want = (total + 255) / 256, cap = (long long)num_sms * 8;
    int blocks = (int)(want < cap ? want : cap);
    if (blocks < 1) blocks = 1;
    launch_pdl(gather_rows_kernel, dim3(blocks), dim3(256), 0, stream, static_cast<const uint16_t *>(x), d, perm_tok,
                                                   rows, static_cast<uint16_t *>(xp), to_fp16, xexp, T, status);
    return cudaGetLastError();
}

}  // namespace moe
