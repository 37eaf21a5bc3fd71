// api.cu -- the C ABI declared in include/moe.h: argument checks, workspace
// layout and kernel dispatch.  Every check happens on the host before any
// launch; nothing here allocates, frees or synchronises (except moe_check,
// which documents that it waits).
#include <stdint.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_gemm.h"
#if MOE_DEBUG
#include <atomic>

#include "moe_debug.h"

namespace {
std::atomic<bool> g_corrupt_offsets{false};   // moe_debug_corrupt_next_offsets
__global__ void corrupt_offsets_kernel(int32_t *offsets, int E) { offsets[E] += 1; }
}  // namespace

moe_status moe_debug_corrupt_next_offsets(void)
{
    g_corrupt_offsets.store(true);
    return MOE_OK;
}
#endif

using namespace moe;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool act_ok(int dt) { return dt == MOE_F32 || dt == MOE_BF16; }

bool scoring_ok(int scoring)
{
    return scoring == MOE_SCORE_SELECTED_SOFTMAX || scoring == MOE_SCORE_SOFTMAX ||
           scoring == MOE_SCORE_SIGMOID;
}

bool weights_ok(int act_dt, int w_dt)
{
    if (act_dt == MOE_F32) return w_dt == MOE_F32;
    return w_dt == MOE_BF16 || is_conv(w_dt);
}

// Largest d the router kernel can stage (one token of fp32 in <= 200 KB).
bool route_fits(int d, int E) { return route_smem_bytes(1, d, E) <= 200 * 1024; }

moe_status check_route_args(const void *x, int act_dt, int T, int d, const void *w_router,
                            const float *bias, int E, int k)
{
    if (T < 0 || d <= 0 || E <= 0 || k < 1 || k > E) return MOE_ERR_INVALID_ARG;
    if (!act_ok(act_dt)) return MOE_ERR_INVALID_ARG;
    if (d % 8) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if (!route_fits(d, E)) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && (!x || !w_router)) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!aligned16(x) || !aligned16(w_router))) return MOE_ERR_INVALID_ARG;
    if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

struct WsLayout {
    size_t status, topk_idx, topk_w, counts, offsets, perm_tok, inv, perm_w, h, xp, pgu, pd,
        flags, y, xexp, rank, tile_cnt, total;
    bool dtc;   // tensor-core decode scratch present
    int n_flags;
};

bool prefill_capable(int act_dt, int w_dt, int d, int F)
{
    return act_dt == MOE_BF16 && (w_dt == MOE_BF16 || is_conv(w_dt)) &&
           d % 256 == 0 && F % 128 == 0;
}

WsLayout ws_layout(int T, int d, int E, int k, int F, int act_dt, int w_dt)
{
    WsLayout L{};
    const size_t n = (size_t)T * k;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 256); return at; };
    L.status = take(4);
    L.topk_idx = take(4 * n);
    L.topk_w = take(4 * n);
    L.counts = take(4 * (size_t)E);
    L.offsets = take(4 * ((size_t)E + 1));
    L.perm_tok = take(4 * n);
    L.inv = take(4 * n);
    L.perm_w = take(4 * n);
    L.rank = take(4 * n);
    L.tile_cnt = take(4 * (size_t)(T > 0 ? T : 1) * (size_t)E);   // <= one tile per token
    L.h = take(4 * n * (size_t)F);            // fp32 (decode); prefill uses 2 bytes/element
    // the decode_tc_capable() shape/dtype conditions, without the driver query
    L.dtc = act_dt == MOE_BF16 && (w_dt == MOE_BF16 || is_conv(w_dt)) && d % 128 == 0 &&
            F % 128 == 0 && n <= (size_t)kDecodeTcMaxRows;
    L.xp = (prefill_capable(act_dt, w_dt, d, F) || L.dtc) ? take(2 * n * (size_t)d) : off;
    L.pgu = L.pd = L.flags = off;
    // k > 2: weighted expert outputs per grouped row, combined in slot order
    // (the CUDA-core decode kernels and the grouped GEMMs)
    L.y = k > 2 ? take(4 * n * (size_t)d) : off;
    // Q8_0 / 4-bit grouped GEMMs and 4-bit tensor-core decode: exponent of
    // each fp16 grouped row's scale
    L.xexp = ((prefill_capable(act_dt, w_dt, d, F) && w_dt != MOE_BF16) || (L.dtc && w_dt != MOE_BF16))
                 ? take(4 * n) : off;
    L.n_flags = 0;
    if (L.dtc) {
        int ks_gu = 1, ks_d = 1;
        decode_tc_splits(T, d, E, k, F, w_dt, &ks_gu, &ks_d);
        L.pgu = take(4 * (size_t)ks_gu * 2 * n * (size_t)F);
        L.pd = take(4 * (size_t)ks_d * n * (size_t)d);
        // the fused decode kernel's flags (whichever decode kernels run)
        L.n_flags = decode_fused_flag_words(T, E, k, F);
        L.flags = take(4 * (size_t)L.n_flags);
    }
    L.total = off;
    return L;
}

}  // namespace

namespace moe {

moe_status forward_args_check(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                              const float *sel_bias, int E, int k, const void *w_gate,
                              const void *w_up, const void *w_down, moe_dtype w_dt, int F,
                              const float *out, int path, int scoring, bool dense)
{
    if (!scoring_ok(scoring)) return MOE_ERR_INVALID_ARG;
    // (dense: no router; the router checks then cover x alone)
    moe_status st = check_route_args(x, act_dt, T, d, dense ? x : w_router, dense ? nullptr : sel_bias,
                                     E, k);
    if (st != MOE_OK) return st;
    if (F <= 0 || F % 8) return MOE_ERR_INVALID_ARG;
    if (!weights_ok(act_dt, w_dt)) {
        return (w_dt == MOE_F32 || w_dt == MOE_BF16 || is_conv(w_dt))
                   ? MOE_ERR_UNSUPPORTED
                   : MOE_ERR_INVALID_ARG;
    }
    if (w_dt == MOE_Q8_0 && (d % 32 || F % 32)) return MOE_ERR_INVALID_ARG;
    if (w_dt == MOE_Q4_A64 && (d % 64 || F % 64)) return MOE_ERR_INVALID_ARG;
    if ((w_dt == MOE_Q4_K || w_dt == MOE_Q6_K) && (d % 256 || F % 256))
        return MOE_ERR_INVALID_ARG;   // whole super-blocks
    if (path != MOE_PATH_AUTO && path != MOE_PATH_DECODE && path != MOE_PATH_PREFILL &&
        path != MOE_PATH_DECODE_SIMT)
        return MOE_ERR_INVALID_ARG;
    const bool can_prefill = prefill_capable(act_dt, w_dt, d, F) && tc_gemm_supports(w_dt) &&
                             tc_gemm_available();
    if (path == MOE_PATH_PREFILL && !can_prefill) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!w_gate || !w_up || !w_down || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) || !aligned16(out))
        return MOE_ERR_INVALID_ARG;
    if (is_conv(w_dt)) {
        const uintptr_t m = 255u;
        if ((reinterpret_cast<uintptr_t>(w_gate) & m) || (reinterpret_cast<uintptr_t>(w_up) & m) ||
            (reinterpret_cast<uintptr_t>(w_down) & m))
            return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

}  // namespace moe

namespace {

// the layer (defined below; `dense`: see there)
moe_status forward_impl(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                        const float *sel_bias, int E, int k, const void *w_gate, const void *w_up,
                        const void *w_down, moe_dtype w_dt, int F, float *out, void *workspace,
                        size_t ws_bytes, int path, int scoring, bool dense, void *const *events,
                        moe_stream stream, int expire_family = 0, uint32_t expire_ns = 0);

}  // namespace

extern "C" {

const char *moe_status_str(int status)
{
    switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype combination";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime or launch error";
    case MOE_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case MOE_ERR_DEVICE_CHECK: return "a device-side consistency check failed";
    default: return "unknown status";
    }
}

int moe_version(void) { return 101; }

moe_status moe_route(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                     const float *sel_bias, int E, int k, int32_t *topk_idx, float *topk_w,
                     moe_stream stream)
{
    return moe_route_scored(x, act_dt, T, d, w_router, sel_bias, E, k, MOE_SCORE_SELECTED_SOFTMAX,
                            topk_idx, topk_w, stream);
}

moe_status moe_route_scored(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                            const float *sel_bias, int E, int k, int scoring, int32_t *topk_idx,
                            float *topk_w, moe_stream stream)
{
    if (!scoring_ok(scoring)) return MOE_ERR_INVALID_ARG;
    moe_status st = check_route_args(x, act_dt, T, d, w_router, sel_bias, E, k);
    if (st != MOE_OK) return st;
    if (T == 0) return MOE_OK;
    if (!topk_idx || !topk_w) return MOE_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(topk_idx) & 3u) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
        return MOE_ERR_INVALID_ARG;
    cudaError_t e;
    if (route_small_capable(act_dt, T, d, E, k)) {
        // the clustered router moe_forward runs on bf16 decode batches (routing only)
        RouteTcArgs a{};
        a.x = x; a.w_router = w_router; a.bias = sel_bias; a.T = T; a.d = d; a.E = E; a.k = k;
        a.mode = scoring;
        a.topk_idx = topk_idx; a.topk_w = topk_w;
        e = launch_route_small(a, static_cast<cudaStream_t>(stream));
    } else if (route_tc_capable(act_dt, d, E) && T >= kRouteTcMinTokens) {
        RouteTcArgs a{};
        a.x = x; a.w_router = w_router; a.bias = sel_bias; a.T = T; a.d = d; a.E = E; a.k = k;
        a.mode = scoring;
        a.topk_idx = topk_idx; a.topk_w = topk_w;
        e = launch_route_tc(a, static_cast<cudaStream_t>(stream));
    } else {
        e = launch_route(x, act_dt, T, d, w_router, sel_bias, E, k, topk_idx, topk_w, nullptr,
                         nullptr, 0, nullptr, nullptr, nullptr, scoring,
                         static_cast<cudaStream_t>(stream));
    }
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_permute(const int32_t *topk_idx, int T, int k, int E, int32_t *counts,
                       int32_t *offsets, int32_t *perm_tok, int32_t *inv, moe_stream stream)
{
    if (T < 0 || k < 1 || E <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > kMaxExperts || k > kMaxTopK) return MOE_ERR_UNSUPPORTED;
    if ((long long)T * k > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !perm_tok || !inv)) return MOE_ERR_INVALID_ARG;
    for (const void *p : {(const void *)topk_idx, (const void *)counts, (const void *)offsets,
                          (const void *)perm_tok, (const void *)inv})
        if (reinterpret_cast<uintptr_t>(p) & 3u) return MOE_ERR_INVALID_ARG;
    // T == 0 still writes zero counts and offsets
    cudaError_t e = launch_permute(topk_idx, T, k, E, counts, offsets, perm_tok, inv, nullptr,
                                   nullptr, nullptr, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_q8_0_packed_size(long long rows, int cols)
{
    if (rows < 0 || cols <= 0 || cols % 32) return 0;
    return align_up((size_t)rows * cols, 256) + (size_t)rows * (cols / 32) * 2;
}

moe_status moe_pack_q8_0(const void *blocks, long long rows, int cols, void *packed,
                         moe_stream stream)
{
    if (rows < 0 || cols <= 0 || cols % 32) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !packed || (reinterpret_cast<uintptr_t>(packed) & 255u))
        return MOE_ERR_INVALID_ARG;
    cudaError_t e = launch_pack_q8_0(blocks, rows, cols, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_q6_k_packed_size(long long rows, int cols)
{
    if (rows < 0 || cols <= 0 || cols % 256) return 0;
    return align_up((size_t)rows * cols, 256) + (size_t)rows * (cols / 16) * 2;
}

moe_status moe_pack_q6_k(const void *blocks, long long rows, int cols, void *packed, moe_stream stream)
{
    if (rows < 0 || cols <= 0 || cols % 256) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !packed || (reinterpret_cast<uintptr_t>(packed) & 255u))
        return MOE_ERR_INVALID_ARG;
    cudaError_t e = launch_pack_q6_k(blocks, rows, cols, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_fp8_packed_size(long long rows, int cols)
{
    if (rows < 0 || cols <= 0) return 0;
    return align_up((size_t)rows * cols, 256) + (size_t)rows * 4;
}

moe_status moe_pack_fp8(const void *rows_in, long long rows, int cols, void *packed, moe_stream stream)
{
    if (rows < 0 || cols <= 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!rows_in || !packed || (reinterpret_cast<uintptr_t>(packed) & 255u))
        return MOE_ERR_INVALID_ARG;
    cudaError_t e = launch_pack_fp8(rows_in, rows, cols, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_q4_a64_packed_size(long long rows, int cols)
{
    if (rows < 0 || cols <= 0 || cols % 64) return 0;
    return q4_a64_packed_bytes(rows, cols);
}

moe_status moe_pack_q4_a64(const void *blocks, long long rows, int cols, void *packed,
                           moe_stream stream)
{
    if (rows < 0 || cols <= 0 || cols % 64) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !packed || (reinterpret_cast<uintptr_t>(packed) & 255u))
        return MOE_ERR_INVALID_ARG;
    cudaError_t e = launch_pack_q4_a64(blocks, rows, cols, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_q4_k_packed_size(long long rows, int cols)
{
    if (rows < 0 || cols <= 0 || cols % 256) return 0;
    return q4_k_packed_bytes(rows, cols);
}

moe_status moe_pack_q4_k(const void *blocks, long long rows, int cols, void *packed, moe_stream stream)
{
    if (rows < 0 || cols <= 0 || cols % 256) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!blocks || !packed || (reinterpret_cast<uintptr_t>(packed) & 255u))
        return MOE_ERR_INVALID_ARG;
    cudaError_t e = launch_pack_q4_k(blocks, rows, cols, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

size_t moe_workspace_size(int T, int d, int E, int k, int F, moe_dtype act_dt, moe_dtype w_dt)
{
    if (T < 0 || d <= 0 || E <= 0 || k < 1 || k > E || F <= 0) return 0;
    if (!act_ok(act_dt) || !weights_ok(act_dt, w_dt)) return 0;
    return ws_layout(T, d, E, k, F, act_dt, w_dt).total;
}

moe_status moe_workspace_views(int T, int d, int E, int k, int F, moe_dtype act_dt,
                               moe_dtype w_dt, size_t *views)
{
    if (!views || moe_workspace_size(T, d, E, k, F, act_dt, w_dt) == 0) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(T, d, E, k, F, act_dt, w_dt);
    views[0] = L.topk_idx; views[1] = L.topk_w; views[2] = L.counts; views[3] = L.offsets;
    views[4] = L.perm_tok; views[5] = L.inv; views[6] = L.perm_w;
    return MOE_OK;
}

moe_status moe_forward(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                       const float *sel_bias, int E, int k, const void *w_gate,
                       const void *w_up, const void *w_down, moe_dtype w_dt, int F,
                       float *out, void *workspace, size_t ws_bytes, int path,
                       moe_stream stream)
{
    return moe_forward_profiled(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down,
                                w_dt, F, out, workspace, ws_bytes, path, nullptr, stream);
}

moe_status moe_forward_profiled(const void *x, moe_dtype act_dt, int T, int d,
                                const void *w_router, const float *sel_bias, int E, int k,
                                const void *w_gate, const void *w_up, const void *w_down,
                                moe_dtype w_dt, int F, float *out, void *workspace,
                                size_t ws_bytes, int path, void *const *events,
                                moe_stream stream)
{
    return moe_forward_scored(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down,
                              w_dt, F, out, workspace, ws_bytes, path, MOE_SCORE_SELECTED_SOFTMAX,
                              events, stream);
}

moe_status moe_forward_scored(const void *x, moe_dtype act_dt, int T, int d,
                              const void *w_router, const float *sel_bias, int E, int k,
                              const void *w_gate, const void *w_up, const void *w_down,
                              moe_dtype w_dt, int F, float *out, void *workspace,
                              size_t ws_bytes, int path, int scoring, void *const *events,
                              moe_stream stream)
{
    return forward_impl(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down, w_dt, F,
                        out, workspace, ws_bytes, path, scoring, false, events, stream);
}

moe_status moe_ffn_dense(const void *x, moe_dtype act_dt, int T, int d, const void *w_gate,
                         const void *w_up, const void *w_down, moe_dtype w_dt, int F, float *out,
                         void *workspace, size_t ws_bytes, int path, moe_stream stream)
{
    return forward_impl(x, act_dt, T, d, nullptr, nullptr, 1, 1, w_gate, w_up, w_down, w_dt, F,
                        out, workspace, ws_bytes, path, MOE_SCORE_SELECTED_SOFTMAX, true, nullptr,
                        stream);
}

moe_status moe_forward_expire_wait(const void *x, moe_dtype act_dt, int T, int d,
                                   const void *w_router, const float *sel_bias, int E, int k,
                                   const void *w_gate, const void *w_up, const void *w_down,
                                   moe_dtype w_dt, int F, float *out, void *workspace,
                                   size_t ws_bytes, int path, int kernel_family, uint32_t wait_ns,
                                   moe_stream stream)
{
    if (kernel_family < MOE_KERNEL_ROUTER_CLUSTER || kernel_family > MOE_KERNEL_GEMM ||
        wait_ns == 0 || wait_ns > 100000000u)
        return MOE_ERR_INVALID_ARG;
    return forward_impl(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up, w_down, w_dt, F,
                        out, workspace, ws_bytes, path, MOE_SCORE_SELECTED_SOFTMAX, false, nullptr,
                        stream, kernel_family, wait_ns);
}

}  // extern "C"

namespace {

// The layer; `dense`: one expert and k = 1 with no router (every token to
// expert 0 with weight 1), the rows read in place where the expert kernels
// take the activation dtype as it is.
moe_status forward_impl(const void *x, moe_dtype act_dt, int T, int d, const void *w_router,
                        const float *sel_bias, int E, int k, const void *w_gate, const void *w_up,
                        const void *w_down, moe_dtype w_dt, int F, float *out, void *workspace,
                        size_t ws_bytes, int path, int scoring, bool dense, void *const *events,
                        moe_stream stream, int expire_family, uint32_t expire_ns)
{
    moe_status st = forward_args_check(x, act_dt, T, d, w_router, sel_bias, E, k, w_gate, w_up,
                                       w_down, w_dt, F, out, path, scoring, dense);
    if (st != MOE_OK || T == 0) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return MOE_ERR_INVALID_ARG;
    const bool can_prefill = prefill_capable(act_dt, w_dt, d, F) && tc_gemm_supports(w_dt) &&
                             tc_gemm_available();
    const WsLayout L = ws_layout(T, d, E, k, F, act_dt, w_dt);
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;

    char *ws = static_cast<char *>(workspace);
    uint32_t *status = reinterpret_cast<uint32_t *>(ws + L.status);
    int32_t *topk_idx = reinterpret_cast<int32_t *>(ws + L.topk_idx);
    float *topk_w = reinterpret_cast<float *>(ws + L.topk_w);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *perm_tok = reinterpret_cast<int32_t *>(ws + L.perm_tok);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
    float *perm_w = reinterpret_cast<float *>(ws + L.perm_w);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    bool use_prefill = false;
    if (path == MOE_PATH_PREFILL) use_prefill = true;
    else if (path == MOE_PATH_AUTO) use_prefill = can_prefill && tc_gemm_prefer(T, d, E, k, F);

    cudaEvent_t ev[6] = {};
    if (events)
        for (int i = 0; i < 6; ++i) ev[i] = static_cast<cudaEvent_t>(events[i]);
    auto mark = [&](int i) { return ev[i] ? cudaEventRecord(ev[i], s) : cudaSuccess; };

    if (mark(0) != cudaSuccess) return MOE_ERR_CUDA;
    const bool use_dtc = !use_prefill && path != MOE_PATH_DECODE_SIMT && L.dtc &&
                         decode_tc_capable(act_dt, w_dt, d, F, E);
    const int num_sms = device_sm_count();
    // bf16 decode batches with enough (expert, tile) units: gate/up, down and
    // combine in one persistent kernel
    const bool use_fused = use_dtc && w_dt == MOE_BF16 && decode_fused_fits(T, d, E, k, F, num_sms);
    // the expert kernels that accumulate into `out` need it zeroed first (the
    // fused kernel adds into it for k = 2 and stores for k = 1; the other
    // tensor-core decode kernels add into it only when their down kernel does)
    const bool zero_out = use_fused ? k == 2
                          : use_dtc ? k > 1 && decode_tc_down_into_out(T, d, E, k, F, w_dt, num_sms)
                                    : k == 2;   // k > 2: combined from per-row outputs
    // routing, then the grouping scatter (which also writes the grouped x rows
    // that the tensor-core expert kernels read)
    RouteTcArgs ra{};
    ra.x = x; ra.w_router = w_router; ra.bias = sel_bias; ra.T = T; ra.d = d; ra.E = E; ra.k = k;
    ra.mode = scoring;
    ra.topk_idx = topk_idx; ra.topk_w = topk_w;
    ra.rank = reinterpret_cast<int32_t *>(ws + L.rank);
    ra.tile_cnt = reinterpret_cast<int32_t *>(ws + L.tile_cnt);
    ra.counts = counts; ra.offsets = offsets; ra.perm_tok = perm_tok; ra.inv = inv; ra.perm_w = perm_w;
    const bool act16 = act_dt == MOE_BF16;
    // decode batches of up to 128 tokens: one clustered kernel routes and
    // groups (no scatter); the tensor-core decode kernel gathers x rows itself
    const bool fused_small = !dense && use_dtc && route_small_capable(act_dt, T, d, E, k);
    // the clustered router writes grouped rows only as fp16, for the 4-bit
    // tensor-core decode kernels, and only for up to 16 tokens: beyond that a
    // separate gather kernel writes them sooner than the router's owners do
    const bool router_rows = is_conv(w_dt) && T <= kRouteSmallRowsMaxT;
    ra.xp = ((use_prefill || (use_dtc && !use_fused)) && act16 && (!fused_small || router_rows)) ? ws + L.xp
                                                                                                : nullptr;
    // the Q8_0 grouped GEMMs and the 4-bit tensor-core decode kernels take fp16
    // rows (scaled)
    ra.xp_fp16 = is_conv(w_dt);
    ra.xexp = reinterpret_cast<int32_t *>(ws + L.xexp);
    ra.out_zero = (zero_out && !use_prefill) ? out : nullptr;   // the GEMM path zeroes its own
    // the fused decode kernel's flags and ticket start at zero
    ra.zero_words = use_fused ? reinterpret_cast<uint32_t *>(ws + L.flags) : nullptr;
    ra.n_zero = use_fused ? L.n_flags : 0;
    // the wait-expiry test hook: the kernel family named must run on this call
    const bool route_tc_path = !dense && !fused_small && route_tc_capable(act_dt, d, E) &&
                               T >= kRouteTcMinTokens;
    uint32_t x_route = 0, x_dtc = 0, x_fused = 0, x_gemm = 0;
    if (expire_family) {
        bool runs = false;
        switch (expire_family) {
        case MOE_KERNEL_ROUTER_CLUSTER: runs = fused_small; x_route = expire_ns; break;
        case MOE_KERNEL_ROUTER_TC: runs = route_tc_path; x_route = expire_ns; break;
        case MOE_KERNEL_DECODE_SPLIT: runs = use_dtc && !use_fused; x_dtc = expire_ns; break;
        case MOE_KERNEL_DECODE_FUSED: runs = use_fused; x_fused = expire_ns; break;
        case MOE_KERNEL_GEMM: runs = use_prefill; x_gemm = expire_ns; break;
        default: break;
        }
        if (!runs) return MOE_ERR_UNSUPPORTED;
    }
    ra.expire_ns = x_route;
    ra.status = status;
    ra.ev_routed = ev[1];
    bool xp_ready = ra.xp != nullptr;
    // grouped 16-bit rows for the tensor-core kernels: a dense layer's are x
    // itself unless the Q8_0 GEMMs or the 4-bit decode kernels need fp16 rows
    void *xp_rows = ws + L.xp;
    cudaError_t e;
    if (dense) {
        e = launch_identity_grouping(T, topk_idx, topk_w, counts, offsets, perm_tok, inv, perm_w,
                                     status, ra.zero_words, ra.n_zero, device_sm_count(), s);
        if (e != cudaSuccess || mark(1) != cudaSuccess || mark(2) != cudaSuccess) return MOE_ERR_CUDA;
        const bool in_place = act16 && w_dt == MOE_BF16;   // Q8_0 / 4-bit: fp16 rows
        if (in_place) xp_rows = const_cast<void *>(x);
        xp_ready = in_place;
    } else if (fused_small) {
        e = launch_route_small(ra, s);
        if (e != cudaSuccess || mark(2) != cudaSuccess) return MOE_ERR_CUDA;
    } else if (route_tc_path) {
        e = launch_route_tc(ra, s);
        if (e != cudaSuccess || mark(2) != cudaSuccess) return MOE_ERR_CUDA;
    } else {
        e = launch_route(x, act_dt, T, d, w_router, sel_bias, E, k, topk_idx, topk_w, ra.out_zero,
                         ra.zero_words, ra.n_zero, ra.rank, ra.tile_cnt, status, scoring, s);
        if (e != cudaSuccess || mark(1) != cudaSuccess) return MOE_ERR_CUDA;
        const int tpb = route_tokens_per_block(T, d, E);
        e = launch_scatter(ra, (T + tpb - 1) / tpb, tpb, s);
        if (e != cudaSuccess || mark(2) != cudaSuccess) return MOE_ERR_CUDA;
    }
#if MOE_DEBUG
    if (g_corrupt_offsets.exchange(false)) {   // test hook (moe_debug.h)
        corrupt_offsets_kernel<<<1, 1, 0, s>>>(offsets, E);
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
#endif

    if (use_prefill) {
        TcArgs a{};
        a.x = x; a.T = T; a.d = d; a.E = E; a.k = k; a.F = F;
        a.w_gate = w_gate; a.w_up = w_up; a.w_down = w_down; a.w_dt = w_dt;
        a.offsets = offsets; a.perm_tok = perm_tok; a.perm_w = perm_w;
        a.xp = xp_rows; a.xp_ready = xp_ready;
        a.h = ws + L.h; a.out = out; a.zero_out = zero_out; a.status = status; a.num_sms = num_sms;
        a.y = reinterpret_cast<float *>(ws + L.y); a.inv = inv;
        a.xexp = reinterpret_cast<int32_t *>(ws + L.xexp);
        a.expire_ns = x_gemm;
        a.ev_gathered = ev[3]; a.ev_gateup = ev[4];
        e = launch_tc_experts(a, s);
    } else if (use_fused) {
        DecodeFusedArgs a{};
        a.x = x; a.T = T; a.d = d; a.E = E; a.k = k; a.F = F;
        a.w_gate = w_gate; a.w_up = w_up; a.w_down = w_down;
        a.offsets = offsets; a.perm_tok = perm_tok; a.perm_w = perm_w;
        a.h = reinterpret_cast<uint16_t *>(ws + L.h);
        a.flags = reinterpret_cast<uint32_t *>(ws + L.flags);
        a.out = out; a.status = status; a.num_sms = num_sms; a.ev_done = ev[4];
        a.expire_ns = x_fused;
        if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
        e = launch_decode_fused(a, s);
    } else if (use_dtc) {
        DecodeTcArgs a{};
        a.w_dt = w_dt;
        a.x = x; a.T = T; a.d = d; a.E = E; a.k = k; a.F = F;
        a.w_gate = w_gate; a.w_up = w_up; a.w_down = w_down;
        a.offsets = offsets; a.inv = inv; a.topk_w = topk_w; a.xp = xp_rows;
        a.pgu = reinterpret_cast<float *>(ws + L.pgu); a.pd = reinterpret_cast<float *>(ws + L.pd);
        a.h = reinterpret_cast<uint16_t *>(ws + L.h);
        a.out = out; a.status = status; a.num_sms = num_sms; a.ev_gateup = ev[4];
        a.expire_ns = x_dtc;
        a.perm_tok = perm_tok;
        a.perm_w = perm_w;
        int32_t *xexp = reinterpret_cast<int32_t *>(ws + L.xexp);
        a.xexp = xexp;
        const int conv = is_conv(w_dt);   // converted weights: fp16 token rows
        if (fused_small && !conv) {
            a.x_gather = x;   // (the converted-weight kernels take fp16 token rows by TMA from xp)
        } else if (!xp_ready &&
                   launch_gather_rows(x, d, perm_tok, T * k, xp_rows, conv, xexp, T, status, num_sms, s) != cudaSuccess) {
            return MOE_ERR_CUDA;
        }
        if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
        e = launch_decode_tc(a, s);
    } else {
        DecodeArgs a{};
        a.x = x; a.act_dt = act_dt; a.T = T; a.d = d; a.E = E; a.k = k; a.F = F;
        a.w_gate = w_gate; a.w_up = w_up; a.w_down = w_down; a.w_dt = w_dt;
        a.offsets = offsets; a.perm_tok = perm_tok; a.perm_w = perm_w;
        a.h = reinterpret_cast<float *>(ws + L.h); a.out = out; a.num_sms = num_sms;
        a.y = reinterpret_cast<float *>(ws + L.y); a.inv = inv; a.status = status;
        a.ev_gateup = ev[4];
        if (mark(3) != cudaSuccess) return MOE_ERR_CUDA;
        e = launch_decode_experts(a, s);
    }
    if (e != cudaSuccess || mark(5) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_check(const void *workspace, uint32_t *device_word, moe_stream stream)
{
    if (!workspace) return MOE_ERR_INVALID_ARG;
    uint32_t w = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&w, workspace, sizeof w, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (device_word) *device_word = w;
    if (w & kDevTimeout) return MOE_ERR_TIMEOUT;
    if (w & kDevCheckFailed) return MOE_ERR_DEVICE_CHECK;
    return MOE_OK;
}

}  // extern "C"
