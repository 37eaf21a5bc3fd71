// route_small.cu -- router projection + SelectedSoftmax + token grouping in
// one kernel, for decode batches of at most 128 tokens (bf16 activations).
//
// SelectedSoftmax ("New Community Model: ZONOS3-Mini (Zyphra) - #1271",
// §Framework change): rank experts by router logit plus selection bias, keep
// the top k, weight them by the softmax of their unbiased logits; ties in the
// ranking score go to the lower expert index.  Scoring modes 1 and 2 (same
// section): rank by softmax-over-all-experts / sigmoid probability plus the
// bias and weigh by that probability (no renormalisation).  Grouping: the slots of each
// expert in increasing token order (stable), rows offset by the exclusive
// scan of the per-expert counts.
//
// At decode sizes the layer's first step is pure latency.  One thread issues
// a tcgen05.mma about every 120 ns whatever its N, so a single CTA walking all
// d/16 MMAs of the logits (64 for d = 1024) spends most of the step issuing;
// a separate grouping kernel adds a launch and a round trip.  Here a cluster
// of R = min(8, d/64) CTAs splits the reduction over d:
//   - CTA r loads its k-blocks of x (all T <= 128 token rows, one TMA box per
//     k-block) and of W_r (E rows padded to 16) at once, and one thread
//     issues M=128 x N=E_pad MMAs over them: partial logits in TMEM.
//   - CTA q owns tokens [q*tpc, q*tpc + tpc).  Each CTA stages its partial
//     logits in shared memory and sends the rows of each owner with one bulk
//     copy into slot r of the owner's receive buffer, completing on the
//     owner's mbarrier (no per-element remote traffic, no cluster barrier).
//     The owner sums the R slots in rank order (a fixed order: results do
//     not depend on timing), 8 threads per token each over every 8th expert;
//     the partial top-k lists merge with shuffles; one thread per token
//     writes indices, weights and a bit in this CTA's per-expert token mask.
//   - Every CTA sends its masks to every CTA the same way; with all masks in
//     hand, the counts, the exclusive scan over experts (offsets) and the
//     prefix over lower CTAs (which own lower tokens) give each slot its
//     grouped row = offset[e] + (e's tokens in lower CTAs) + (e's tokens
//     before it here).
//   - Optionally (the fp16 operands of the 4-bit tensor-core decode kernels)
//     each CTA also writes the grouped rows of its own tokens as fp16, scaled
//     by 2^-xexp (fp16_row_exponent): the exponents are taken from x while
//     the operands load, the rows once the grouped positions are known.
//   Cluster barriers: one after the mbarriers are initialised (before any
//   peer may signal them; it overlaps the wait for the preceding kernel) and
//   one before exit (no CTA leaves while a peer may still copy into it).
// Every mbarrier wait is bounded (see sm100.cuh); a CTA whose wait gives up
// records the timeout and still reaches every cluster barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tc_gemm.h"

namespace moe {
namespace rsm {

using namespace sm100;

constexpr int MAXR = 8;                       // CTAs per cluster (split of d)
constexpr int TPC = 16;                       // tokens a CTA ranks (T <= 128)
constexpr int BK = 64;
constexpr int A_TILE = 128 * BK * 2;          // 16 KB: the M=128 operand of one k-block
constexpr int MAXKB = 8;                      // k-blocks per CTA
constexpr int THREADS = 192;
constexpr int SUBS = 8;                       // threads per token in the ranking

__host__ __device__ constexpr int b_tile_bytes(int EP) { return (EP * BK * 2 + 1023) / 1024 * 1024; }

struct Params {
    int T, d, E, EP, k, R, kblocks, box_rows, tpc;
    int mode;                            // scoring: 0 SelectedSoftmax, 1 softmax / 2 sigmoid before rank
    const float *bias;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *counts, *offsets, *perm_tok, *inv;
    float *perm_w;
    uint32_t *status;
    float *out_zero;                     // optional [T, d] output to zero (the down kernel adds into it)
    uint32_t *zero_words;                // optional scratch words later kernels count on being zero
    int n_zero;
    uint32_t expire_ns;                  // > 0: the MMA thread's operand wait gives up after this long (test hook)
    const uint16_t *x;                   // [T, d] bf16 (the rows below)
    uint16_t *xp;                        // optional [T*k, d] fp16 grouped rows, row r = x * 2^-xexp[r]
    int32_t *xexp;                       //   and their exponents
};

struct Ctl {
    uint64_t full, tfull, rx, mx;        // operands, MMAs, partials received, masks received
    uint64_t never;                      // nothing arrives here (test hook)
    uint32_t tmem_base;
    int abort_flag;
    float bias[kMaxExperts];
    alignas(16) uint32_t mask[kMaxExperts];            // bit j: owned token j chose expert e
    alignas(16) uint32_t all_mask[MAXR][kMaxExperts];  // every CTA's masks (sent by their owners)
    int tot[kMaxExperts], pre[kMaxExperts], off[kMaxExperts + 1];
    int sel_e[TPC][kMaxTopK];
    float sel_w[TPC][kMaxTopK];
    int xe[TPC];                         // xp: exponent of each owned token row
    int pos[TPC][kMaxTopK];              // xp: grouped row of each owned slot (-1: none)
};

// bulk copy of `bytes` from this CTA's shared memory to a CTA of the
// cluster; completion is counted on that CTA's mbarrier (cluster addresses)
__device__ __forceinline__ void bulk_to_peer(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "r"(smem_u32(src)), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

constexpr int kNone = 0x7fffffff;

// (score desc, expert asc) order; unfilled slots (kNone) rank last
__device__ __forceinline__ bool ranks_before(float s, int e, float s2, int e2)
{
    return e2 == kNone || s > s2 || (s == s2 && e < e2);
}

// Insert (cs, cl, ce) into the sorted top-K (bs, bl, be); every slot's update
// reads only the old slots.
template <int K>
__device__ __forceinline__ void insert(float (&bs)[K], float (&bl)[K], int (&be)[K], float cs, float cl,
                                       int ce)
{
    if (ce == kNone) return;
    bool gt[K];
#pragma unroll
    for (int j = 0; j < K; ++j) gt[j] = ranks_before(cs, ce, bs[j], be[j]);
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
        const bool from_prev = gt[j - 1], take = gt[j];
        bs[j] = from_prev ? bs[j - 1] : (take ? cs : bs[j]);
        bl[j] = from_prev ? bl[j - 1] : (take ? cl : bl[j]);
        be[j] = from_prev ? be[j - 1] : (take ? ce : be[j]);
    }
    if (gt[0]) { bs[0] = cs; bl[0] = cl; be[0] = ce; }
}

// shared memory: [A tiles: kbpc x 16 KB][B tiles: kbpc x b_tile][staged
// partial logits: 128 x EP fp32][receive buffer: MAXR slots x TPC rows x EP
// fp32][Ctl]
__host__ __device__ inline size_t stage_offset(int kbpc, int EP) { return (size_t)kbpc * (A_TILE + b_tile_bytes(EP)); }
// staged and received rows are EP + 4 floats apart: rows land 4 banks apart,
// so per-row 16-byte stores and per-expert reads of 8 rows do not conflict
__host__ __device__ constexpr int row_stride(int EP) { return EP + 4; }
__host__ __device__ inline size_t recv_offset(int kbpc, int EP) { return stage_offset(kbpc, EP) + (size_t)128 * row_stride(EP) * 4; }
__host__ __device__ inline size_t ctl_offset(int kbpc, int EP)
{
    return recv_offset(kbpc, EP) + (size_t)MAXR * TPC * row_stride(EP) * 4;
}
// token rows owned by CTA q
__host__ __device__ inline int owned_rows(int q, int tpc, int T)
{
    const int lo = q * tpc, hi = lo + tpc < T ? lo + tpc : T;
    return hi > lo ? hi - lo : 0;
}

// XP: also write the grouped fp16 rows (a separate instantiation, so that the
// routing-only code is not touched by it)
template <int KMAX, bool XP>
__global__ void __launch_bounds__(THREADS, 1)
route_small_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                   const Params p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int EP = p.EP, E = p.E, R = p.R;
    const int kbpc = (p.kblocks + R - 1) / R;
    const uint32_t rank = cluster_rank();
    const int kb0 = (int)rank * p.kblocks / R, kb1 = ((int)rank + 1) * p.kblocks / R, nkb = kb1 - kb0;
    uint8_t *a_tiles = smem;
    uint8_t *b_tiles = smem + (size_t)kbpc * A_TILE;
    float *stage = reinterpret_cast<float *>(smem + stage_offset(kbpc, EP));   // [128][EP]
    float *recv = reinterpret_cast<float *>(smem + recv_offset(kbpc, EP));     // [MAXR][TPC][EP]
    Ctl &c = *reinterpret_cast<Ctl *>(smem + ctl_offset(kbpc, EP));
    const int BT = b_tile_bytes(EP);
    const int mine_rows = owned_rows((int)rank, p.tpc, p.T);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ncols = EP <= 32 ? 32 : EP <= 64 ? 64 : EP <= 128 ? 128 : 256;

    // set-up that reads nothing the preceding kernels write
    if (threadIdx.x == 0) {
        mbar_init(&c.full, 1);
        mbar_init(&c.tfull, 1);
        mbar_init(&c.never, 1);
        mbar_init(&c.rx, 1);
        mbar_init(&c.mx, 1);
        // the bytes the peers will send: R slots of this CTA's token rows, and
        // R mask rows
        if (mine_rows > 0) mbar_expect_tx(&c.rx, (uint32_t)(R * mine_rows * row_stride(EP) * 4));
        mbar_expect_tx(&c.mx, (uint32_t)(R * EP * 4));
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    }
    for (int e = threadIdx.x; e < kMaxExperts; e += THREADS) c.mask[e] = 0u;
    if (warp == 1) tmem_alloc(&c.tmem_base, ncols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();                       // every CTA's mbarriers exist before anyone signals them
    pdl_wait();   // (the next kernel is released once this CTA's operands are in: see below)
    if (threadIdx.x == 0) {
        // ------------------------------------------------ TMA: every operand tile at once,
        // first, so that the zeroing below overlaps the round trip from HBM
        mbar_expect_tx(&c.full, (uint32_t)(nkb * (p.box_rows + EP) * BK * 2));
        for (int j = 0; j < nkb; ++j) {
            tma_load_2d(a_tiles + (size_t)j * A_TILE, &tm_x, &c.full, (kb0 + j) * BK, 0);
            tma_load_2d(b_tiles + (size_t)j * BT, &tm_w, &c.full, (kb0 + j) * BK, 0);
        }
    }
    if (p.status && rank == 0 && threadIdx.x == 0) *p.status = kDevOk;
    if (p.out_zero) {   // this CTA's share of the output rows
        float4 *o4 = reinterpret_cast<float4 *>(p.out_zero);
        const long long n4 = (long long)p.T * p.d / 4;
        const long long per = (n4 + R - 1) / R, lo = (long long)rank * per;
        const long long hi = lo + per < n4 ? lo + per : n4;
        for (long long i = lo + threadIdx.x; i < hi; i += THREADS) o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = (int)rank * THREADS + threadIdx.x; i < p.n_zero; i += R * THREADS) p.zero_words[i] = 0u;
    for (int e = threadIdx.x; e < kMaxExperts; e += THREADS) c.bias[e] = (e < E && p.bias) ? p.bias[e] : 0.f;
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_f16_mn(0, 128, EP);
        const bool ok = (p.expire_ns == 0 || mbar_wait(&c.never, 0, abort_flag, p.expire_ns)) &&
                        mbar_wait(&c.full, 0, abort_flag);
        if (ok) {
            tc_fence_after();
            for (int j = 0; j < nkb; ++j) {
                const uint32_t a0 = smem_u32(a_tiles + (size_t)j * A_TILE);
                const uint32_t b0 = smem_u32(b_tiles + (size_t)j * BT);
                const uint64_t da = sw128_desc(a0), db = sw128_desc(b0);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_f16(tmem, desc_step(da, kk * 32), desc_step(db, kk * 32), idesc, (j | kk) != 0);
            }
        } else {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            volatile int no_abort = 0;   // let the loads land before the CTA moves on
            mbar_wait(&c.full, 0, &no_abort);
        }
        umma_commit(&c.tfull);
    } else if (warp >= 2) {
        // ------------------------------------------------ partial logits -> shared memory
        const int quarter = warp & 3;
        if constexpr (XP) {
            // the exponents of this CTA's own token rows, while the operands
            // load and the MMAs run
            for (int i = warp - 2; i < mine_rows; i += 4) {
                const int e = fp16_row_exponent(p.x + (size_t)((int)rank * p.tpc + i) * p.d, p.d, lane);
                if (lane == 0) c.xe[i] = e;
            }
        }
        const bool ok = __all_sync(0xffffffffu, mbar_wait(&c.tfull, 0, abort_flag));
        if (!ok) {
            if (lane == 0) flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        } else if (quarter * 32 < p.T) {
            tc_fence_after();
            const int row = quarter * 32 + lane;   // token row
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
            for (int c0 = 0; c0 < EP; c0 += 32) {  // two TMEM loads per wait
                uint32_t v[2][16];
                tmem_ld16(taddr + c0, v[0]);   // warp-collective
                if (c0 + 16 < EP) tmem_ld16(taddr + c0 + 16, v[1]);
                tmem_ld_wait();
                if (row < p.T) {
                    uint4 *dst = reinterpret_cast<uint4 *>(stage + (size_t)row * row_stride(EP) + c0);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        if (c0 + 4 * q < EP)
                            dst[q] = make_uint4(v[q >> 2][(4 * q) & 15], v[q >> 2][(4 * q + 1) & 15],
                                                v[q >> 2][(4 * q + 2) & 15], v[q >> 2][(4 * q + 3) & 15]);
                }
            }
            fence_proxy_async_smem();          // the bulk copies read these rows
        }
        tc_fence_before();
    }
    __syncwarp();
    __syncthreads();
    // the operands are in and the logits computed: the next kernel of the
    // stream may start launching now (its reads from HBM no longer compete
    // with this kernel's)
    pdl_trigger();
    if (threadIdx.x < R) {
        // owner q = lane receives its token rows of this CTA's partials in slot `rank`
        const int q = threadIdx.x, n = owned_rows(q, p.tpc, p.T);
        if (n > 0)
            bulk_to_peer(peer_addr(recv + (size_t)rank * TPC * row_stride(EP), (uint32_t)q),
                         stage + (size_t)q * p.tpc * row_stride(EP), (uint32_t)(n * row_stride(EP) * 4),
                         peer_addr(&c.rx, (uint32_t)q));
        bulk_commit();
    }

    // ---- ranking of this CTA's tokens: sum of the R partials in rank order
    const int tbase = (int)rank * p.tpc;
    if (warp >= 2) {
        const int et = threadIdx.x - 64;      // 0..127
        const int tok = et >> 3, sub = et & 7;
        const int t = tbase + tok;
        bool got = true;
        if (mine_rows > 0 && !mbar_wait(&c.rx, 0, abort_flag)) {
            got = false;
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
        const bool mine = got && tok < p.tpc && t < p.T && !c.abort_flag;
        float bs[KMAX], bl[KMAX];
        int be[KMAX];
#pragma unroll
        for (int j = 0; j < KMAX; ++j) { bs[j] = -INFINITY; bl[j] = 0.f; be[j] = kNone; }
        auto logit_of = [&](int e) {
            float cl = 0.f;
#pragma unroll
            for (int q = 0; q < MAXR; ++q)
                if (q < R) cl += recv[((size_t)q * TPC + tok) * row_stride(EP) + e];
            return cl;
        };
        // softmax before rank: the token's max and denominator over all E,
        // each of its 8 threads over every 8th expert, combined by xor shuffles
        float lmax = -INFINITY, lden = 1.f;
        if (p.mode == 1) {
            if (mine)
                for (int e = sub; e < E; e += SUBS) lmax = fmaxf(lmax, logit_of(e));
#pragma unroll
            for (int o = 1; o < SUBS; o <<= 1) lmax = fmaxf(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
            lden = 0.f;
            if (mine)
                for (int e = sub; e < E; e += SUBS) lden += expf(logit_of(e) - lmax);
#pragma unroll
            for (int o = 1; o < SUBS; o <<= 1) lden += __shfl_xor_sync(0xffffffffu, lden, o);
        }
        if (mine) {
            // bl: the selected experts' logits (mode 0) or probabilities
            for (int e = sub; e < E; e += SUBS) {
                float cl = logit_of(e);
                if (p.mode == 1) cl = expf(cl - lmax) / lden;
                else if (p.mode == 2) cl = 1.0f / (1.0f + expf(-cl));
                float cs = cl + c.bias[e];
                if (isnan(cs)) cs = -INFINITY;        // keep the ranking a total order
                insert<KMAX>(bs, bl, be, cs, cl, e);
            }
        }
        // merge the 8 partial lists of a token (lanes 8i .. 8i+7 of a warp)
#pragma unroll
        for (int o = 1; o < SUBS; o <<= 1) {
            float os[KMAX], ol[KMAX];
            int oe[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                os[j] = __shfl_xor_sync(0xffffffffu, bs[j], o);
                ol[j] = __shfl_xor_sync(0xffffffffu, bl[j], o);
                oe[j] = __shfl_xor_sync(0xffffffffu, be[j], o);
            }
#pragma unroll
            for (int j = 0; j < KMAX; ++j) insert<KMAX>(bs, bl, be, os[j], ol[j], oe[j]);
        }
        if (mine && sub == 0) {
            float m = bl[0];
#pragma unroll
            for (int j = 1; j < KMAX; ++j) if (j < p.k) m = fmaxf(m, bl[j]);
            float w[KMAX], den = 0.f;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                w[j] = j < p.k ? (p.mode == 0 ? expf(bl[j] - m) : bl[j]) : 0.f;
                den += w[j];
            }
            if (p.mode != 0) den = 1.f;   // probabilities as they are
            const size_t ob = (size_t)t * p.k;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
                if (j < p.k) {
                    const int e = be[j] < E ? be[j] : 0;   // kNone only if E < k (rejected on the host)
                    p.topk_idx[ob + j] = e;
                    p.topk_w[ob + j] = w[j] / den;
                    c.sel_e[tok][j] = e;
                    c.sel_w[tok][j] = w[j] / den;
                    atomicOr(&c.mask[e], 1u << tok);
                }
            }
        }
    }
    fence_proxy_async_smem();                 // the bulk copies read the masks
    __syncwarp();
    __syncthreads();
    if (threadIdx.x < R) {
        // this CTA's masks into slot `rank` of CTA q = lane's table
        const int q = threadIdx.x;
        bulk_to_peer(peer_addr(&c.all_mask[rank][0], (uint32_t)q), c.mask, (uint32_t)(EP * 4),
                     peer_addr(&c.mx, (uint32_t)q));
        bulk_commit();
    }
    if (!mbar_wait(&c.mx, 0, abort_flag)) {
        flag_status(p.status, kDevTimeout);
        c.abort_flag = 1;
    }

    // ---- grouping
    for (int e = threadIdx.x; e < E; e += THREADS) {
        int tot = 0, pre = 0;
        for (int r = 0; r < R; ++r) {
            const int n = __popc(c.all_mask[r][e]);
            tot += n;
            pre += r < (int)rank ? n : 0;
        }
        c.tot[e] = tot;
        c.pre[e] = pre;
    }
    __syncthreads();
    if (warp == 0) {
        constexpr int PER = kMaxExperts / 32;
        int local = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            local += e < E ? c.tot[e] : 0;
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        int run = incl - local;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            if (e < E) { c.off[e] = run; run += c.tot[e]; }
        }
        if (lane == 31) c.off[E] = incl;
    }
    __syncthreads();
    if (rank == 0 && p.counts) {
        for (int e = threadIdx.x; e < E; e += THREADS) { p.counts[e] = c.tot[e]; p.offsets[e] = c.off[e]; }
        if (threadIdx.x == 0) p.offsets[E] = c.off[E];
    }
    // slot (owned token i, choice j) -> grouped row (routing only: no grouping outputs)
    for (int s = threadIdx.x; p.counts && s < p.tpc * p.k; s += THREADS) {
        const int i = s / p.k, j = s - i * p.k, t = tbase + i;
        if (XP) c.pos[i][j] = -1;
        if (t >= p.T || c.abort_flag) continue;
        const int e = c.sel_e[i][j];
        const int pos = c.off[e] + c.pre[e] + __popc(c.mask[e] & ((1u << i) - 1u));
        if (pos < 0 || pos >= p.T * p.k) {   // cannot happen with consistent masks
            flag_status(p.status, kDevCheckFailed);
            continue;
        }
        if (XP) c.pos[i][j] = pos;
        p.perm_tok[pos] = t;
        p.inv[(size_t)t * p.k + j] = pos;
        p.perm_w[pos] = c.sel_w[i][j];
    }
    if (threadIdx.x == 0 && *abort_flag) {
        // a wait above gave up early: the peers' copies into this CTA (sent
        // by every CTA on every path) land before it leaves (bounded)
        volatile int no_abort = 0;
        if (mine_rows > 0) mbar_wait(&c.rx, 0, &no_abort);
        mbar_wait(&c.mx, 0, &no_abort);
    }
    __syncthreads();
    if (XP && p.counts && !*abort_flag) {
        // the grouped fp16 rows of this CTA's tokens and their exponents; each
        // thread issues U loads before it converts and stores any
        constexpr int U = 8;
        const int vec = p.d / 8, n = mine_rows * p.k * vec;
        for (int w0 = threadIdx.x; w0 < n; w0 += THREADS * U) {
            uint4 u[U];
            int dst[U], ex[U];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int w = w0 + q * THREADS;
                dst[q] = -1;
                if (w < n) {
                    const int sj = w / vec, ch = w - sj * vec;
                    const int i = sj / p.k, j = sj - i * p.k, pos = c.pos[i][j];
                    if (pos >= 0) {
                        u[q] = __ldg(reinterpret_cast<const uint4 *>(p.x + (size_t)(tbase + i) * p.d) + ch);
                        dst[q] = pos * vec + ch;
                        ex[q] = c.xe[i];
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
                if (dst[q] < 0) continue;
                reinterpret_cast<uint4 *>(p.xp)[dst[q]] = bf16x8_to_fp16_scaled(u[q], ex[q]);
                if (dst[q] % vec == 0) p.xexp[dst[q] / vec] = ex[q];
            }
        }
    }
    if (threadIdx.x < R) bulk_wait_read();    // this CTA's outgoing copies have read their sources
    // no CTA leaves while a peer may still copy into it (no memory ordering needed)
    __syncwarp();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

constexpr size_t kSmemCap = 200 * 1024;

size_t smem_bytes(int kbpc, int EP) { return 1024 + ctl_offset(kbpc, EP) + sizeof(Ctl); }

int cluster_size(int d) { const int kb = d / BK; return kb < MAXR ? kb : MAXR; }

}  // namespace rsm

bool route_small_capable(int act_dt, int T, int d, int E, int k)
{
    using namespace rsm;
    if (act_dt != MOE_BF16 || T < 1 || T > 128 || d % BK != 0 || E > kMaxExperts || k > E ||
        !tc_gemm_available())
        return false;
    const int R = cluster_size(d);
    const int kbpc = (d / BK + R - 1) / R;
    const int EP = (E + 15) / 16 * 16;
    return (T + R - 1) / R <= TPC && kbpc <= MAXKB && smem_bytes(kbpc, EP) <= kSmemCap;
}

cudaError_t launch_route_small(const RouteTcArgs &a, cudaStream_t stream)
{
    using namespace rsm;
    if (!route_small_capable(MOE_BF16, a.T, a.d, a.E, a.k)) return cudaErrorInvalidValue;
    const int EP = (a.E + 15) / 16 * 16;
    const int R = cluster_size(a.d);
    const int kblocks = a.d / BK;
    const int kbpc = (kblocks + R - 1) / R;
    const size_t smem = smem_bytes(kbpc, EP);
    CUtensorMap m_x, m_w;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int box_rows = a.T;   // all token rows of a k-block in one box (T <= 128)
    if (!tc::make_map(&m_x, a.x, (uint64_t)a.T, a.d, box_rows, bf) ||
        !tc::make_map(&m_w, a.w_router, (uint64_t)a.E, a.d, EP, bf))
        return cudaErrorInvalidValue;
    cudaError_t err;
    static PerDeviceFlag attr_done;
    const int dev = current_device();
    if (!attr_done.done(dev)) {
        const int mx = (int)kSmemCap;
        if ((err = cudaFuncSetAttribute(route_small_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_small_kernel<8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx)) != cudaSuccess)
            return err;
        attr_done.mark(dev);
    }
    Params p{};
    p.T = a.T; p.d = a.d; p.E = a.E; p.EP = EP; p.k = a.k; p.R = R; p.kblocks = kblocks;
    p.mode = a.mode;
    p.box_rows = box_rows; p.tpc = (a.T + R - 1) / R;
    p.bias = a.bias; p.topk_idx = a.topk_idx; p.topk_w = a.topk_w;
    p.counts = a.counts; p.offsets = a.offsets; p.perm_tok = a.perm_tok; p.inv = a.inv;
    p.perm_w = a.perm_w; p.status = a.status; p.out_zero = a.out_zero;
    p.zero_words = a.zero_words; p.n_zero = a.n_zero;
    p.expire_ns = a.expire_ns;
    p.x = static_cast<const uint16_t *>(a.x);
    // grouped rows: fp16 only (the bf16 decode kernels gather x themselves)
    if (a.xp && (!a.xp_fp16 || !a.counts || !a.xexp)) return cudaErrorInvalidValue;
    p.xp = static_cast<uint16_t *>(a.xp);
    p.xexp = a.xexp;
    auto kern = p.xp ? (a.k == 1 ? route_small_kernel<1, true> : a.k == 2 ? route_small_kernel<2, true>
                        : a.k <= 4 ? route_small_kernel<4, true> : route_small_kernel<8, true>)
                     : (a.k == 1 ? route_small_kernel<1, false> : a.k == 2 ? route_small_kernel<2, false>
                        : a.k <= 4 ? route_small_kernel<4, false> : route_small_kernel<8, false>);
    err = launch_pdl_cluster(kern, dim3(R), dim3(THREADS), smem, stream, R, m_x, m_w, p);
    if (err != cudaSuccess) return err;
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.ev_routed && (err = cudaEventRecord(a.ev_routed, stream)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace moe
