// route_tc.cu -- router projection + SelectedSoftmax on tcgen05, and the
// token-grouping scatter that follows it (bf16 activations).
//
// SelectedSoftmax ("New Community Model: ZONOS3-Mini (Zyphra) - #1271",
// §Framework change): rank experts by router logit plus selection bias, keep
// the top k, weight them by the softmax of their unbiased logits; ties in the
// ranking score go to the lower expert index.  Scoring modes 1 and 2 (same
// section): rank by softmax-over-all-experts / sigmoid probability plus the
// bias and weigh by that probability (no renormalisation).
//
// route_tc_kernel: one CTA per tile of 128 tokens.  Warp 0 streams the x tile
// [128 x 64] and the router tile [EP x 64] (E rows padded to a multiple of 16,
// TMA zero-fills the padding) through a ring of up to 8 stages (as many as fit
// in 192 KB for this EP); warp 1 issues
// tcgen05.mma M=128, N=EP, accumulating the logits [128 tokens x EP] in TMEM
// (fp32); warps 2-5 each own 32 tokens -- thread = token: it reads its logit
// row from TMEM, keeps a sorted top-k in registers, and writes indices and
// softmax weights.  The same threads record, per expert, a 128-bit mask of the
// tile's tokens that chose it: the tile's per-expert counts are the mask
// popcounts and a token's stable rank within the tile is the popcount of the
// mask bits below it.
//
// scatter_kernel: one CTA per token tile.  Exclusive scan over (expert, tile)
// of the tile counts gives every slot its grouped row
//   row = offset[e] + sum_{tiles b' < b} count[b'][e] + rank,
// i.e. a stable sort by expert with tokens ascending -- the same permutation
// as the single-CTA grouping kernel.  It writes perm_tok, inv and the
// per-row routing weight, and optionally copies x rows into grouped order for
// the grouped GEMMs.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tc_gemm.h"

namespace moe {
namespace rtc {

using namespace sm100;

constexpr int BM = 128, BK = 64, MAXST = 8;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB x tile
constexpr int RING_BYTES = 192 * 1024;          // stages of A_BYTES + EP * 128
constexpr int THREADS = 192;

__host__ __device__ constexpr int stage_bytes(int EP) { return (A_BYTES + EP * BK * 2 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int num_stages(int EP)
{
    return RING_BYTES / stage_bytes(EP) < MAXST ? RING_BYTES / stage_bytes(EP) : MAXST;
}

struct Params {
    int T, d, E, EP, k;
    int mode;             // scoring: 0 SelectedSoftmax, 1 softmax before rank, 2 sigmoid before rank
    const float *bias;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *rank;        // [T*k] stable rank of the slot within its token tile
    int32_t *tile_cnt;    // [ntiles][E]
    float *out_zero;      // optional [T, d] rows to zero
    uint32_t *zero_words;
    int n_zero;
    uint32_t *status;
    uint32_t expire_ns;   // > 0: the producer's first wait gives up after this long (test hook)
};

struct Ctl {
    uint64_t full[MAXST], empty[MAXST], tfull, epi;
    uint64_t never;                  // nothing arrives here (test hook)
    uint32_t tmem_base;
    int abort_flag;
    float bias[kMaxExperts];
    uint32_t mask[kMaxExperts][4];   // tokens of this tile that chose expert e
};

// Sorted top-K insertion of (score cs, logit cl, expert ce) into slots
// (bs, bl, be), ordered by score descending then expert ascending.  Experts
// arrive in ascending order, so a newcomer never precedes an equal score;
// unfilled slots (be == kNone) take anything.  Every slot's update reads only
// the old slots, so the K updates of one expert are independent.
constexpr int kNone = 0x7fffffff;
template <int K>
__device__ __forceinline__ void topk_insert(float (&bs)[K], float (&bl)[K], int (&be)[K], float cs,
                                            float cl, int ce)
{
    bool gt[K];
#pragma unroll
    for (int j = 0; j < K; ++j) gt[j] = cs > bs[j] || be[j] == kNone;
#pragma unroll
    for (int j = K - 1; j > 0; --j) {
        const bool from_prev = gt[j - 1], take = gt[j];
        bs[j] = from_prev ? bs[j - 1] : (take ? cs : bs[j]);
        bl[j] = from_prev ? bl[j - 1] : (take ? cl : bl[j]);
        be[j] = from_prev ? be[j - 1] : (take ? ce : be[j]);
    }
    if (gt[0]) { bs[0] = cs; bl[0] = cl; be[0] = ce; }
}

// KMAX: compile-time bound on k (1, 2, 4 or 8) so the top-k insertion is as
// short as the k it serves.
template <int KMAX>
__global__ void __launch_bounds__(THREADS, 1)
route_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                const Params p)
{
    pdl_enter();
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int b_bytes = p.EP * BK * 2;
    const int SLOT = stage_bytes(p.EP), STAGES = num_stages(p.EP);
    Ctl &c = *reinterpret_cast<Ctl *>(smem + RING_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E, EP = p.EP;
    const int t0 = blockIdx.x * BM;
    const int kblocks = p.d / BK;
    const uint32_t ncols = EP <= 32 ? 32 : EP <= 64 ? 64 : EP <= 128 ? 128 : 256;

    if (p.status && blockIdx.x == 0 && threadIdx.x == 0) *p.status = kDevOk;
    for (int i = blockIdx.x * THREADS + threadIdx.x; i < p.n_zero; i += gridDim.x * THREADS)
        p.zero_words[i] = 0u;
    if (p.out_zero) {
        const int ntok = min(BM, p.T - t0);
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = threadIdx.x * 4; i < ntok * p.d; i += THREADS * 4)
            *reinterpret_cast<float4 *>(p.out_zero + (size_t)t0 * p.d + i) = z;
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&c.full[s], 1); mbar_init(&c.empty[s], 1); }
        mbar_init(&c.tfull, 1);
        mbar_init(&c.epi, 128);
        mbar_init(&c.never, 1);
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    for (int e = threadIdx.x; e < kMaxExperts; e += THREADS) {
        c.bias[e] = (e < E && p.bias) ? p.bias[e] : 0.f;
        c.mask[e][0] = c.mask[e][1] = c.mask[e][2] = c.mask[e][3] = 0u;
    }
    if (warp == 1) tmem_alloc(&c.tmem_base, ncols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = c.tmem_base;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        bool ok = p.expire_ns == 0 || mbar_wait(&c.never, 0, abort_flag, p.expire_ns);
        int kb = 0;
        for (; ok && kb < kblocks; ++kb) {
            const int s = kb % STAGES;
            const uint32_t ph = (kb / STAGES) & 1u;
            if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
            mbar_expect_tx(&c.full[s], A_BYTES + b_bytes);
            tma_load_2d(smem + s * SLOT, &tm_x, &c.full[s], kb * BK, t0);
            tma_load_2d(smem + s * SLOT + A_BYTES, &tm_w, &c.full[s], kb * BK, 0);
        }
        if (!ok) {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            for (int j = (kb >= STAGES ? kb - STAGES : 0); j < kb; ++j) {
                volatile int no_abort = 0;
                mbar_wait(&c.full[j % STAGES], (j / STAGES) & 1u, &no_abort);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        const uint32_t idesc = idesc_f16_mn(0, BM, EP);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
            const int s = kb % STAGES;
            const uint32_t ph = (kb / STAGES) & 1u;
            if (!mbar_wait(&c.full[s], ph, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t a0 = smem_u32(smem + s * SLOT);
            const uint32_t b0 = a0 + A_BYTES;
            const uint64_t da = sw128_desc(a0), db = sw128_desc(b0);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
                umma_f16(tmem, desc_step(da, kk * 32), desc_step(db, kk * 32), idesc,
                         (kb | kk) != 0);
            umma_commit(&c.empty[s]);
        }
        if (ok) {
            umma_commit(&c.tfull);
        } else {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            umma_commit(&c.tfull);   // drains the MMAs in flight; the epilogue sees the abort
        }
    } else if (warp >= 2) {
        // ------------------------------------------------ thread = token epilogue
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;        // token row within the tile (TMEM lane)
        const int t = t0 + r;
        const bool valid = t < p.T;
        bool ok = mbar_wait(&c.tfull, 0, abort_flag);
        if (!ok) {
            if (lane == 0) flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
        ok = __all_sync(0xffffffffu, ok);   // tcgen05.ld below is warp-collective
        uint32_t epi_phase = 0;
        {
            if (ok) tc_fence_after();
            float bs[KMAX], bl[KMAX];
            int be[KMAX];
#pragma unroll
            for (int j = 0; j < KMAX; ++j) { bs[j] = -INFINITY; bl[j] = 0.f; be[j] = kNone; }
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16);
            // this token's logits, 32 TMEM columns at a time: f(e, logit)
            auto for_each_logit = [&](auto &&f) {
                for (int c0 = 0; ok && c0 < EP; c0 += 32) {
                    uint32_t v[2][16];
                    tmem_ld16(taddr + c0, v[0]);
                    if (c0 + 16 < EP) tmem_ld16(taddr + c0 + 16, v[1]);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int e = c0 + q;
                        if (e < E) f(e, __uint_as_float(v[q >> 4][q & 15]));
                    }
                }
            };
            // softmax before rank: max, then the denominator in expert order
            float lmax = -INFINITY, lden = 1.f;
            if (p.mode == 1) {
                for_each_logit([&](int, float l) { lmax = fmaxf(lmax, l); });
                lden = 0.f;
                for_each_logit([&](int, float l) { lden += expf(l - lmax); });
            }
            // bl: the selected experts' logits (mode 0) or probabilities
            for_each_logit([&](int e, float cl) {
                if (p.mode == 1) cl = expf(cl - lmax) / lden;
                else if (p.mode == 2) cl = 1.0f / (1.0f + expf(-cl));
                float cs = cl + c.bias[e];
                if (isnan(cs)) cs = -INFINITY;   // keep the ranking a total order
                topk_insert<KMAX>(bs, bl, be, cs, cl, e);
            });
            float wsel[KMAX];
            if (ok && valid) {
                float m = bl[0];
#pragma unroll
                for (int j = 1; j < KMAX; ++j) if (j < p.k) m = fmaxf(m, bl[j]);
                float den = 0.f;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    wsel[j] = j < p.k ? (p.mode == 0 ? expf(bl[j] - m) : bl[j]) : 0.f;
                    den += wsel[j];
                }
                const size_t base = (size_t)t * p.k;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < p.k) {
                        wsel[j] = p.mode == 0 ? wsel[j] / den : wsel[j];
                        p.topk_idx[base + j] = be[j];
                        p.topk_w[base + j] = wsel[j];
                        if (p.rank) atomicOr(&c.mask[be[j]][r >> 5], 1u << (r & 31));
                    }
                }
            }
            // wait for every token's mask bits, then ranks and tile counts
            // (a bounded barrier: a thread that gave up above still arrives)
            if (!bounded_bar(&c.epi, epi_phase, abort_flag)) ok = false;
            if (ok && valid && p.rank) {
                const size_t base = (size_t)t * p.k;
#pragma unroll
                for (int j = 0; j < KMAX; ++j) {
                    if (j < p.k) {
                        const uint32_t *mk = c.mask[be[j]];
                        int rk = 0;
                        for (int w = 0; w < (r >> 5); ++w) rk += __popc(mk[w]);
                        rk += __popc(mk[r >> 5] & ((1u << (r & 31)) - 1u));
                        p.rank[base + j] = rk;
                    }
                }
            }
            for (int e = threadIdx.x - 64; ok && p.tile_cnt && e < E; e += 128)
                p.tile_cnt[(size_t)blockIdx.x * E + e] =
                    __popc(c.mask[e][0]) + __popc(c.mask[e][1]) + __popc(c.mask[e][2]) + __popc(c.mask[e][3]);
        }
        tc_fence_before();
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, ncols);
    }
}

}  // namespace rtc

// Grouped rows of the slots of token tile `blockIdx.x` (tiles of `tile_tokens`
// tokens, as produced by either router): part blockIdx.y of gridDim.y handles
// every gridDim.y-th slot of the tile.  See the file header.
__global__ void __launch_bounds__(256)
scatter_kernel(const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w,
               const int32_t *__restrict__ rank, const int32_t *__restrict__ tile_cnt, int ntiles,
               int tile_tokens, int T, int k, int E, int32_t *__restrict__ counts,
               int32_t *__restrict__ offsets, int32_t *__restrict__ perm_tok,
               int32_t *__restrict__ inv, float *__restrict__ perm_w,
               const uint16_t *__restrict__ x, int d, uint16_t *__restrict__ xp, int xp_fp16,
               int32_t *__restrict__ xexp, uint32_t *__restrict__ status)
{
    pdl_enter();
    __shared__ int tot[kMaxExperts], pre[kMaxExperts], off[kMaxExperts + 1];
    __shared__ int part_tot[8][kMaxExperts], part_pre[8][kMaxExperts];
    if (upstream_failed(status)) return;
    const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nslots_all = T * k;
    // per-expert totals over all tiles and over the tiles before this one:
    // warp w sums tiles w, w+8, ...; lane owns experts lane, lane+32, ...
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        int s_tot = 0, s_pre = 0;
        if (e < E) {
            int bb = warp;
            for (; bb + 24 < ntiles; bb += 32) {   // four independent loads in flight
                const int c0 = __ldcg(tile_cnt + (size_t)bb * E + e);
                const int c1 = __ldcg(tile_cnt + (size_t)(bb + 8) * E + e);
                const int c2 = __ldcg(tile_cnt + (size_t)(bb + 16) * E + e);
                const int c3 = __ldcg(tile_cnt + (size_t)(bb + 24) * E + e);
                s_tot += c0 + c1 + c2 + c3;
                s_pre += (bb < b ? c0 : 0) + (bb + 8 < b ? c1 : 0) + (bb + 16 < b ? c2 : 0) +
                         (bb + 24 < b ? c3 : 0);
            }
            for (; bb < ntiles; bb += 8) {
                const int c0 = __ldcg(tile_cnt + (size_t)bb * E + e);
                s_tot += c0;
                s_pre += bb < b ? c0 : 0;
            }
        }
        if (e < E) { part_tot[warp][e] = s_tot; part_pre[warp][e] = s_pre; }
    }
    __syncthreads();
    if (threadIdx.x < E) {
        int s_tot = 0, s_pre = 0;
#pragma unroll
        for (int w = 0; w < 8; ++w) { s_tot += part_tot[w][threadIdx.x]; s_pre += part_pre[w][threadIdx.x]; }
        tot[threadIdx.x] = s_tot;
        pre[threadIdx.x] = s_pre;
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (E + 31) / 32;
        int local = 0;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) local += tot[e];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int j = 0; j < per; ++j) {
            const int e = lane * per + j;
            if (e < E) { off[e] = run; run += tot[e]; }
        }
        if (lane == 31) off[E] = incl;
    }
    __syncthreads();
    if (b == 0 && blockIdx.y == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) { counts[e] = tot[e]; offsets[e] = off[e]; }
        if (threadIdx.x == 0) offsets[E] = off[E];
    }
    const int t0 = b * tile_tokens;
    const int nslots = min(tile_tokens, T - t0) * k;
    const int part = blockIdx.y, nparts = gridDim.y;
    const int nwarps = nparts * (blockDim.x / 32), gw = part * (blockDim.x / 32) + warp;
    // warp gw owns slots gw, gw + nwarps, ...: in batches of 32, one slot per
    // lane resolves its grouped row (all loads in parallel), then the warp
    // copies the batch's x rows two at a time
    for (int b0 = 0; gw + b0 * nwarps < nslots; b0 += 32) {
        const int i = gw + (b0 + lane) * nwarps;
        int pos = -1, tok = 0;
        if (i < nslots) {
            const size_t slot = (size_t)t0 * k + i;
            const int e = __ldcg(topk_idx + slot);
            pos = (e >= 0 && e < E) ? off[e] + pre[e] + __ldcg(rank + slot) : -1;
            tok = (int)(slot / k);
            if (pos < 0 || pos >= nslots_all) {   // cannot happen with consistent routing
                flag_status(status, kDevCheckFailed);
                pos = -1;
            } else {
                perm_tok[pos] = tok;
                inv[slot] = pos;
                perm_w[pos] = __ldcg(topk_w + slot);
            }
        }
        if (!xp) continue;
        const int vec = d / 8;
        for (int j = 0; j < 32; j += 2) {
            const int p0 = __shfl_sync(0xffffffffu, pos, j), q0 = __shfl_sync(0xffffffffu, tok, j);
            const int p1 = __shfl_sync(0xffffffffu, pos, j + 1), q1 = __shfl_sync(0xffffffffu, tok, j + 1);
            if (p0 < 0 && p1 < 0) continue;
            const uint4 *s0 = reinterpret_cast<const uint4 *>(x + (size_t)q0 * d);
            const uint4 *s1 = reinterpret_cast<const uint4 *>(x + (size_t)q1 * d);
            uint4 *d0 = reinterpret_cast<uint4 *>(xp + (size_t)(p0 < 0 ? 0 : p0) * d);
            uint4 *d1 = reinterpret_cast<uint4 *>(xp + (size_t)(p1 < 0 ? 0 : p1) * d);
            // fp16 rows: each row scaled by 2^-e (see fp16_row_exponent), e kept per grouped row
            int e0 = 0, e1 = 0;
            if (xp_fp16) {
                if (p0 >= 0) e0 = fp16_row_exponent(x + (size_t)q0 * d, d, lane);
                if (p1 >= 0) e1 = fp16_row_exponent(x + (size_t)q1 * d, d, lane);
                if (lane == 0) {
                    if (p0 >= 0) xexp[p0] = e0;
                    if (p1 >= 0) xexp[p1] = e1;
                }
            }
            constexpr int U = 4;   // 2 rows x 4 x 16 bytes per lane in flight
            for (int c0 = lane; c0 < vec; c0 += 32 * U) {
                uint4 v[2][U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
                    if (c < vec) {
                        if (p0 >= 0) v[0][u] = __ldg(s0 + c);
                        if (p1 >= 0) v[1][u] = __ldg(s1 + c);
                    }
                }
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if ((r ? p1 : p0) < 0) continue;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + 32 * u;
                        if (c >= vec) continue;
                        uint4 w4 = v[r][u];
                        if (xp_fp16)   // bf16 -> fp16 rows for the fp16 (Q8_0) tensor-core path
                            w4 = bf16x8_to_fp16_scaled(w4, r ? e1 : e0);
                        (r ? d1 : d0)[c] = w4;
                    }
                }
            }
        }
    }
}

namespace rtc {

constexpr size_t smem_bytes()
{
    return 1024 + (size_t)RING_BYTES + sizeof(Ctl);
}

}  // namespace rtc

cudaError_t launch_scatter(const RouteTcArgs &a, int ntiles, int tile_tokens, cudaStream_t stream)
{
    // enough CTAs that every SM gets a few warps of slots
    const int slots_per_tile = tile_tokens * a.k;
    int parts = (2 * device_sm_count() + ntiles - 1) / ntiles;
    const int max_parts = (slots_per_tile + 7) / 8;   // >= 1 slot per warp
    if (parts > max_parts) parts = max_parts;
    if (parts < 1) parts = 1;
    launch_pdl(scatter_kernel, dim3(ntiles, parts), dim3(256), 0, stream,
        a.topk_idx, a.topk_w, a.rank, a.tile_cnt, ntiles, tile_tokens, a.T, a.k, a.E, a.counts,
        a.offsets, a.perm_tok, a.inv, a.perm_w, static_cast<const uint16_t *>(a.x), a.d,
        static_cast<uint16_t *>(a.xp), a.xp_fp16, a.xexp, a.status);
    return cudaGetLastError();
}

bool route_tc_capable(int act_dt, int d, int E)
{
    return act_dt == MOE_BF16 && d % 64 == 0 && E <= kMaxExperts && tc_gemm_available();
}

int route_tc_tiles(int T) { return (T + 127) / 128; }

cudaError_t launch_route_tc(const RouteTcArgs &a, cudaStream_t stream)
{
    using namespace rtc;
    const int EP = (a.E + 15) / 16 * 16;
    CUtensorMap m_x, m_w;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!tc::make_map(&m_x, a.x, (uint64_t)a.T, a.d, BM, bf) ||
        !tc::make_map(&m_w, a.w_router, (uint64_t)a.E, a.d, EP, bf))
        return cudaErrorInvalidValue;
    cudaError_t err;
    const size_t smem = smem_bytes();
    static PerDeviceFlag attr_done;
    const int dev = current_device();
    if (!attr_done.done(dev)) {
        if ((err = cudaFuncSetAttribute(route_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_tc_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(route_tc_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return err;
        attr_done.mark(dev);
    }
    Params p{};
    p.T = a.T; p.d = a.d; p.E = a.E; p.EP = EP; p.k = a.k; p.bias = a.bias; p.mode = a.mode;
    p.topk_idx = a.topk_idx; p.topk_w = a.topk_w; p.rank = a.rank; p.tile_cnt = a.tile_cnt;
    p.out_zero = a.out_zero; p.zero_words = a.zero_words; p.n_zero = a.n_zero; p.status = a.status;
    p.expire_ns = a.expire_ns;
    const int ntiles = route_tc_tiles(a.T);
    auto kern = a.k == 1 ? route_tc_kernel<1> : a.k == 2 ? route_tc_kernel<2>
              : a.k <= 4 ? route_tc_kernel<4> : route_tc_kernel<8>;
    launch_pdl(kern, dim3(ntiles), dim3(THREADS), smem, stream, m_x, m_w, p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.ev_routed && (err = cudaEventRecord(a.ev_routed, stream)) != cudaSuccess) return err;
    if (!a.counts) return cudaSuccess;   // routing only (moe_route)
    return launch_scatter(a, ntiles, BM, stream);
}

}  // namespace moe
