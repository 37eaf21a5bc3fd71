// decode_fused.cu -- the decode expert FFN in ONE persistent launch on
// tcgen05: gate/up, SwiGLU, down and the routing-weighted combine, weights
// streamed by TMA, for batches whose experts hold enough 128-row weight tiles
// that no K split is needed (the ZONOS3-Mini-shaped decode step: ~50 active
// experts x 4 tiles of F x 8 tiles of d).
//
// At decode sizes an expert holds a handful of token rows, and the layer's
// cost is reading the active experts' weights once from HBM ("Zyphra-ZONOS2-
// 4bit", §Performance notes: batch-1 MoE reads ~1/16 of the experts; batching
// touches more distinct experts until the read is bandwidth bound).  The
// contraction runs on the tensor cores with the operands swapped: a 128-row
// weight tile is the M operand (TMA, 128-byte swizzle, a ring of 16 KB
// stages), the expert's token rows (a chunk of <= 32, padded to 16 or 32) are
// the N operand, gathered into shared memory by four warps, and fp32
// accumulators live in TMEM.
//
// Work items are claimed from a ticket counter:
//   tickets [0, n_gu)      gate/up items (chunk, 128-row tile of F, whole K):
//                          the ring alternates gate and up tiles of the same
//                          rows into a pair of accumulators; the epilogue
//                          writes h = SiLU(G) * U (bf16);
//   tickets [n_gu, n_all)  down items (chunk, 128-row tile of d, whole K):
//                          the epilogue adds w * y into out.
// A down item depends on h of its chunk, F tile by F tile: its weight tiles
// stream into the ring as soon as it is claimed, and only the token-row
// gather of each stage waits for the F tile of h it reads (a per-(chunk, F
// tile) flag that reaches 4, one per epilogue warp).  Tickets are claimed in
// increasing order and gate/up items wait on nothing, so every gate/up item a
// down item waits for was claimed earlier by a running CTA and completes: no
// deadlock, whatever the residency.  A CTA claims its next ticket a ring's
// depth before its current item ends, so items are handed out as CTAs free
// up (balance) while the next weights still stream without a gap.  The
// gate/up -> down boundary is no longer a kernel boundary: down weights
// stream while the last gate/up items finish.
//
// The combine: k = 1 stores w * y; k = 2 adds w * y into out (zeroed by the
// router): exactly two additions onto zero per element, whose result does not
// depend on their order -- bitwise reproducible.
//
// CTA: warp 0 = ticket claims + TMA producer, warp 1 = MMA issuer (+ TMEM
// owner), warps 2-5 = epilogue (TMEM lane quarter = warp % 4), warps 6-9 =
// token-row gatherers (ring stage s by warp 6 + s % 4).  Items reach every
// role through a small queue in shared memory.  All waits -- mbarriers, the
// h flags -- are bounded (see sm100.cuh); a wait that gives up records
// MOE_ERR_TIMEOUT in the status word, raises the CTA's abort flag, lets its
// own copies and MMAs land, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tc_gemm.h"

namespace moe {
namespace dfu {

using namespace sm100;

// Tuning (compile-time): ring depth, resident CTAs per SM.
#ifndef MOE_DFU_STAGES
#define MOE_DFU_STAGES 4
#endif
#ifndef MOE_DFU_CTAS_PER_SM
#define MOE_DFU_CTAS_PER_SM 2
#endif

constexpr int BM = 128, BK = 64, STAGES = MOE_DFU_STAGES;
constexpr int CTAS_PER_SM = MOE_DFU_CTAS_PER_SM;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB weight tile
constexpr int NTMAX = 32;                       // token rows per chunk
constexpr int B_BYTES = NTMAX * BK * 2;         // 4 KB token tile (16 or 32 rows used)
constexpr int SLOT = A_BYTES + B_BYTES;         // 20 KB per stage, 1024-aligned
constexpr int THREADS = 320;
constexpr int NPAIR = 4;                        // accumulator pairs of 2 x 32 TMEM columns
constexpr int TMEM_COLS = 64 * NPAIR;
constexpr int QN = 8;                           // item queue depth
constexpr int kQueueConsumers = 1 + 4 + 4;      // MMA thread, epilogue warps, gather warps
static_assert(STAGES >= 4, "four gather warps: warp 6 + w fills the ring stages s with s % 4 == w");

enum Kind { GATEUP = 0, DOWN = 1, END = 2 };

struct Params {
    const int32_t *offsets;   // [E+1]
    int E, rows, d, F, k;
    int nc_max;               // bound on the chunk count (flag arrays are sized by it)
    int spec_kb;              // k-blocks of every expert's gate/up tiles to prefetch into L2
                              // before the routing is known (0: none)
    const uint16_t *x;        // [T, d] bf16
    const int32_t *perm_tok;  // [rows] grouped row -> token
    const float *perm_w;      // [rows] routing weight of each grouped row
    uint16_t *h;              // [rows, F] bf16
    float *out;               // [T, d] fp32 (zeroed beforehand when k == 2)
    uint32_t *flags;          // zeroed by the router: see flag_layout()
    uint32_t *status;
    uint32_t expire_ns;       // > 0: the producer's first wait gives up after this long (test hook)
};

// Flag words (all zero at launch): h ready per (chunk, F tile), then the
// ticket counter.
struct FlagLayout {
    int ready, ticket, total;
};
__host__ __device__ inline FlagLayout flag_layout(int nc_max, int F)
{
    FlagLayout f;
    f.ready = 0;
    f.ticket = nc_max * (F / BM);
    f.total = f.ticket + 1;
    return f;
}

struct Item {
    int kind, e, c, row0, nrows, nt, tile, kb0, nkb, nst;
};

struct Ctl {
    uint64_t full_w[STAGES], full_x[STAGES], empty[STAGES];
    uint64_t tfull[NPAIR], tempty[NPAIR], qfull[QN], qempty[QN], drain;
    uint64_t never;                     // nothing arrives here (test hook)
    uint32_t tmem_base;
    int abort_flag;
    int n_gu, n_all;
    int chunk_start[kMaxExperts + 1];   // first chunk of expert e; [E] = chunk count
    int off[kMaxExperts + 1];
    Item queue[QN];
};

__device__ __forceinline__ Item decode_ticket(const Ctl &c, const Params &p, int t)
{
    Item it{};
    if (t >= c.n_all) { it.kind = END; return it; }
    const int FT = p.F / BM, DT = p.d / BM;
    int q, kbt;
    if (t < c.n_gu) {
        it.kind = GATEUP; kbt = p.d / BK;
        it.c = t / FT; it.tile = t - it.c * FT;
    } else {
        it.kind = DOWN; kbt = p.F / BK;
        q = t - c.n_gu;
        it.c = q / DT; it.tile = q - it.c * DT;
    }
    int lo = 0, hi = p.E - 1;   // largest e with chunk_start[e] <= c (empty experts share starts)
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (c.chunk_start[mid] <= it.c) lo = mid;
        else hi = mid - 1;
    }
    it.e = lo;
    const int lc = it.c - c.chunk_start[lo];
    const int rows_e = c.off[lo + 1] - c.off[lo];
    it.row0 = c.off[lo] + lc * NTMAX;
    it.nrows = min(NTMAX, rows_e - lc * NTMAX);
    it.nt = it.nrows <= 16 ? 16 : 32;
    it.kb0 = 0;
    it.nkb = kbt;
    it.nst = it.kind == GATEUP ? 2 * it.nkb : it.nkb;
    return it;
}

// Weight matrix (0 gate / 1 up for gate/up items) and k-block of ring stage
// `kbl` of an item: gate/up stages alternate gate and up tiles of one k-block.
__device__ __forceinline__ void stage_of(const Item &it, int kbl, int &m, int &kb)
{
    if (it.kind == GATEUP) { m = kbl & 1; kb = it.kb0 + (kbl >> 1); }
    else { m = 0; kb = it.kb0 + kbl; }
}

// SiLU(z) = z * sigmoid(z) with the fast exponential and an approximate
// divide (relative error ~1e-6, below the bf16 rounding of h that follows).
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait until *flag >= target (one thread).  Gives up on the CTA's
// abort flag, on an error another CTA recorded in the status word, or after
// kTimeoutNs.
__device__ __noinline__ bool wait_flag_ge(const uint32_t *flag, uint32_t target,
                                          volatile int *abort_flag, const uint32_t *status)
{
    if (ld_acquire_u32(flag) >= target) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(96);   // one poll per ~L2 round trip per waiting warp
        if (ld_acquire_u32(flag) >= target) return true;
        if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (status && *(volatile const uint32_t *)status) return false;
            if (globaltimer() - t0 > kTimeoutNs) return false;
        }
    }
}

// h = SiLU(g) * u, rounded to bf16
__device__ __forceinline__ uint16_t swiglu_bf16(float g, float u)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(silu_f(g) * u));
}

// One epilogue warp's share of an h tile is written: count it in the tile's
// ready flag (4 = the whole 128-row tile), after the warp's stores.
__device__ __forceinline__ void publish(uint32_t *ready, int lane)
{
    __threadfence();
    __syncwarp();
    if (lane == 0) {
        __threadfence();
        atomicAdd(ready, 1u);
    }
}

// The routing-weighted combine of one output element: k = 1 stores
// w * y; k = 2 adds it onto the zeroed output (two additions onto zero: the
// result does not depend on their order).
__device__ __forceinline__ void combine_out(const Params &p, int tok, int col, float w, float y)
{
    float *o = p.out + (size_t)tok * p.d + col;
    if (p.k == 1) *o = w * y;
    else atomicAdd(o, w * y);
}

__device__ __forceinline__ void record_abort(Ctl &c, uint32_t *status)
{
    flag_status(status, kDevTimeout);
    c.abort_flag = 1;
}

__global__ void __launch_bounds__(THREADS, CTAS_PER_SM)
decode_fused_kernel(const __grid_constant__ CUtensorMap tm_wg, const __grid_constant__ CUtensorMap tm_wu,
                 const __grid_constant__ CUtensorMap tm_wd, const Params p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Ctl &c = *reinterpret_cast<Ctl *>(smem + STAGES * SLOT);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    // set-up that reads nothing the preceding kernels write (barriers, TMEM,
    // tensor-map prefetch) overlaps their tail under programmatic dependent launch
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&c.full_w[s], 1);      // the producer's expect_tx arrival + the tile's bytes
            mbar_init(&c.full_x[s], 32);     // the gather warp's 32 lanes
            mbar_init(&c.empty[s], 1);       // the MMA commit
        }
        for (int b = 0; b < NPAIR; ++b) { mbar_init(&c.tfull[b], 1); mbar_init(&c.tempty[b], 128); }
        for (int q = 0; q < QN; ++q) { mbar_init(&c.qfull[q], 1); mbar_init(&c.qempty[q], kQueueConsumers); }
        mbar_init(&c.drain, 1);
        mbar_init(&c.never, 1);
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wg)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wu)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_wd)) : "memory");
    }
    if (warp == 0 && lane == 0 && p.spec_kb > 0) {
        // while the routing is still being computed: the first spec_kb k-blocks
        // of every expert's gate and up tiles into L2 (weights only; which of
        // them the batch uses is not known yet), k-block by k-block
        const int FT = p.F / BM;
        const int n = p.spec_kb * p.E * FT * 2;
        for (int i = blockIdx.x; i < n; i += gridDim.x) {
            const int m = i & 1, q = i >> 1;
            const int kb = q / (p.E * FT), r = q - kb * (p.E * FT);
            tma_prefetch_l2_2d(m ? &tm_wu : &tm_wg, kb * BK, r * BM);   // row r*BM = e*F + ft*BM
        }
    }
    if (warp == 1) tmem_alloc(&c.tmem_base, TMEM_COLS);
    tc_fence_before();
    pdl_enter();
    if (upstream_failed(p.status)) {   // (synchronises the CTA)
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(c.tmem_base, TMEM_COLS);
        }
        return;
    }
    const FlagLayout fl = flag_layout(p.nc_max, p.F);
    // the first ticket's round trip overlaps the chunk table
    int first_ticket = 0;
    if (threadIdx.x == 0) first_ticket = (int)atomicAdd(p.flags + fl.ticket, 1u);
    // per-expert chunks of <= 32 rows, numbered across experts
    for (int e = threadIdx.x; e <= E; e += THREADS) c.off[e] = p.offsets[e];
    __syncthreads();
    const bool offsets_ok = debug_offsets_ok(c.off, E, p.rows, p.status);
    if (warp == 0) {
        constexpr int PER = kMaxExperts / 32;
        int local[PER], sum = 0;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            local[j] = e < E ? (c.off[e + 1] - c.off[e] + NTMAX - 1) / NTMAX : 0;
            sum += local[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - sum;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
            const int e = lane * PER + j;
            if (e < E) c.chunk_start[e] = run;
            run += local[j];
        }
        if (lane == 31) {
            const int nc = incl < p.nc_max ? incl : p.nc_max;   // (consistent routing: incl <= nc_max)
            c.chunk_start[E] = nc;
            c.n_gu = offsets_ok ? nc * (p.F / BM) : 0;
            c.n_all = offsets_ok ? c.n_gu + nc * (p.d / BM) : 0;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = c.tmem_base;
    volatile int *abort_flag = &c.abort_flag;
    const int FT = p.F / BM;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ tickets + TMA producer (weights)
        uint32_t it_k = 0, qi = 0;
        bool ok = p.expire_ns == 0 || mbar_wait(&c.never, 0, abort_flag, p.expire_ns);
        int t = first_ticket;
        while (ok) {
            const Item it = decode_ticket(c, p, t);
            const uint32_t qs = qi % QN, qph = (qi / QN) & 1u;
            if (!mbar_wait(&c.qempty[qs], qph ^ 1u, abort_flag)) { ok = false; break; }
            c.queue[qs] = it;
            mbar_arrive(&c.qfull[qs]);
            ++qi;
            if (it.kind == END) break;
            // the next ticket is claimed a ring's depth before this item's last
            // stage: late enough that items go to the CTAs that free up first,
            // early enough that the claim's round trip overlaps the copies
            int t_next = 0;
            const int claim_at = it.nst > STAGES ? it.nst - STAGES : 0;
            const int wrow = it.kind == GATEUP ? it.e * p.F + it.tile * BM : it.e * p.d + it.tile * BM;
            if (it.kind == DOWN)   // the tiles beyond the ring's depth head for L2 now: a
                                   // down item may wait for h with its ring full
                for (int kbl = STAGES; kbl < it.nst; ++kbl) tma_prefetch_l2_2d(&tm_wd, kbl * BK, wrow);
            for (int kbl = 0; kbl < it.nst; ++kbl, ++it_k) {
                if (kbl == claim_at) t_next = (int)atomicAdd(p.flags + fl.ticket, 1u);
                const int s = it_k % STAGES;
                const uint32_t ph = (it_k / STAGES) & 1u;
                if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                mbar_expect_tx(&c.full_w[s], A_BYTES);
                int m, kb;
                stage_of(it, kbl, m, kb);
                const CUtensorMap *wmap = it.kind == DOWN ? &tm_wd : (m ? &tm_wu : &tm_wg);
                tma_load_2d(smem + s * SLOT, wmap, &c.full_w[s], kb * BK, wrow);
            }
            if (!ok) break;
            t = t_next;
        }
        if (!ok) {
            record_abort(c, p.status);
            // let the weight tiles in flight land before the CTA frees its memory
            for (uint32_t j = (it_k >= STAGES ? it_k - STAGES : 0); j < it_k; ++j) {
                volatile int no_abort = 0;
                mbar_wait(&c.full_w[j % STAGES], (j / STAGES) & 1u, &no_abort);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t it_k = 0, qi = 0, li = 0;
        bool ok = true;
        for (;; ++li) {
            const uint32_t qs = qi % QN, qph = (qi / QN) & 1u;
            if (!mbar_wait(&c.qfull[qs], qph, abort_flag)) { ok = false; break; }
            const Item it = c.queue[qs];
            mbar_arrive(&c.qempty[qs]);
            ++qi;
            if (it.kind == END) break;
            const uint32_t acc = li % NPAIR, aph = (li / NPAIR) & 1u;
            if (!mbar_wait(&c.tempty[acc], aph ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t idesc = idesc_f16_mn(0, BM, it.nt);
            for (int kbl = 0; kbl < it.nst; ++kbl, ++it_k) {
                const int s = it_k % STAGES;
                const uint32_t ph = (it_k / STAGES) & 1u;
                if (!mbar_wait(&c.full_w[s], ph, abort_flag) || !mbar_wait(&c.full_x[s], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                int m, kb;
                stage_of(it, kbl, m, kb);
                const uint32_t d_tmem = tmem + acc * 64 + m * 32;
                const uint32_t a0 = smem_u32(smem + s * SLOT);
                const uint32_t b0 = a0 + A_BYTES;
                const bool first = kb == it.kb0;   // first k-block of this accumulator
                const uint64_t da = sw128_desc(a0), db = sw128_desc(b0);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_f16(d_tmem, desc_step(da, kk * 32), desc_step(db, kk * 32), idesc,
                             (!first || kk > 0) ? 1u : 0u);
                umma_commit(&c.empty[s]);
            }
            if (!ok) break;
            umma_commit(&c.tfull[acc]);
        }
        if (!ok) {
            record_abort(c, p.status);
            umma_commit(&c.drain);   // the MMAs issued so far complete before TMEM is freed
            volatile int no_abort = 0;
            mbar_wait(&c.drain, 0, &no_abort);
        }
    } else if (warp >= 6) {
        // ------------------------------------------------ token-row gatherers (4 warps)
        // warp 6 + w fills the ring stages s with s % 4 == w; lane j copies the
        // 128-byte K slice of the chunk's j-th row (x through perm_tok for
        // gate/up items, h for down items), zeros for the padding rows of a
        // 16/32-row tile, in the 128-byte-swizzled layout the MMA reads
        const int sw = warp - 6;
        uint32_t it_k = 0, qi = 0;
        bool ok = true;
        for (;;) {
            const uint32_t qs = qi % QN, qph = (qi / QN) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&c.qfull[qs], qph, abort_flag))) { ok = false; break; }
            const Item it = c.queue[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.qempty[qs]);
            ++qi;
            if (it.kind == END) break;
            const bool has = lane < it.nrows;
            const uint16_t *src;
            if (it.kind == GATEUP) {
                int tok = has ? p.perm_tok[it.row0 + lane] : 0;
                if (has && !debug_index_ok(tok, p.rows / p.k, p.status)) tok = 0;   // (debug builds)
                src = p.x + (size_t)tok * p.d;
            }
            else
                src = p.h + (size_t)(has ? it.row0 + lane : 0) * p.F;
            int ready_tile = -1;   // down: last F tile of h seen complete
            for (int kbl = 0; kbl < it.nst; ++kbl, ++it_k) {
                const int s = it_k % STAGES;
                if ((s & 3) != sw) continue;
                const uint32_t ph = (it_k / STAGES) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&c.empty[s], ph ^ 1u, abort_flag))) { ok = false; break; }
                int m, kb;
                stage_of(it, kbl, m, kb);
                if (it.kind == DOWN && (kb * BK) / BM != ready_tile) {
                    // the F tile of h this k-block reads: all 4 epilogue quarters written
                    ready_tile = (kb * BK) / BM;
                    bool got = true;
                    if (lane == 0)
                        got = wait_flag_ge(p.flags + fl.ready + it.c * FT + ready_tile, 4u, abort_flag,
                                           p.status);
                    if (!__shfl_sync(0xffffffffu, got, 0)) { ok = false; break; }
                    __syncwarp();
                }
                if (lane < it.nt) {
                    const int kx = kb * BK;
                    uint4 v[8];
                    if (it.kind == GATEUP) {
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            v[q] = has ? __ldg(reinterpret_cast<const uint4 *>(src + kx) + q) : make_uint4(0u, 0u, 0u, 0u);
                    } else {
#pragma unroll
                        for (int q = 0; q < 8; ++q)   // h written by other CTAs of this launch: L2
                            v[q] = has ? __ldcg(reinterpret_cast<const uint4 *>(src + kx) + q) : make_uint4(0u, 0u, 0u, 0u);
                    }
                    uint8_t *dst = smem + s * SLOT + A_BYTES + lane * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4 *>(dst + ((q ^ (lane & 7)) << 4)) = v[q];
                }
                fence_proxy_async_smem();
                mbar_arrive(&c.full_x[s]);
            }
            if (!ok) break;
        }
        if (!ok && lane == 0) record_abort(c, p.status);
    } else if (warp >= 2) {
        // ------------------------------------------------ epilogue (4 warps)
        const int quarter = warp & 3;   // TMEM lanes 32*quarter .. +31 (warp % 4 rule)
        uint32_t qi = 0, li = 0;
        bool ok = true;
        for (;; ++li) {
            const uint32_t qs = qi % QN, qph = (qi / QN) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait(&c.qfull[qs], qph, abort_flag))) { ok = false; break; }
            const Item it = c.queue[qs];
            __syncwarp();
            if (lane == 0) mbar_arrive(&c.qempty[qs]);
            ++qi;
            if (it.kind == END) break;
            const uint32_t acc = li % NPAIR, aph = (li / NPAIR) & 1u;
            // warp-uniform outcome: tcgen05.ld below is warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&c.tfull[acc], aph, abort_flag))) { ok = false; break; }
            tc_fence_after();
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * 64;
            const int wr = it.tile * BM + quarter * 32 + lane;   // weight row = output column
            // accumulators -> registers (column j = token row j of the chunk)
            uint32_t a0[32], a1[32];
            tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&a0[0]));
            if (it.nt > 16) tmem_ld16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&a0[16]));
            if (it.kind == GATEUP) {
                tmem_ld16(taddr + 32, *reinterpret_cast<uint32_t(*)[16]>(&a1[0]));
                if (it.nt > 16) tmem_ld16(taddr + 48, *reinterpret_cast<uint32_t(*)[16]>(&a1[16]));
            }
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&c.tempty[acc]);   // the accumulators are in registers now
            if (it.kind == GATEUP) {
                // h = SiLU(G) * U (bf16), then this quarter of the F tile is ready
                uint16_t *dst = p.h + (size_t)it.row0 * p.F + wr;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j < it.nrows)
                        dst[(size_t)j * p.F] = swiglu_bf16(__uint_as_float(a0[j]), __uint_as_float(a1[j]));
                publish(p.flags + fl.ready + it.c * FT + it.tile, lane);
                continue;
            }
            // down: token and routing weight of row j, held by lane j
            int tok_l = lane < it.nrows ? p.perm_tok[it.row0 + lane] : 0;
            float w_l = lane < it.nrows ? p.perm_w[it.row0 + lane] : 0.f;
            if (lane < it.nrows && !debug_index_ok(tok_l, p.rows / p.k, p.status)) { tok_l = 0; w_l = 0.f; }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const int tok = __shfl_sync(0xffffffffu, tok_l, j);
                const float w = __shfl_sync(0xffffffffu, w_l, j);
                if (j < it.nrows) combine_out(p, tok, wr, w, __uint_as_float(a0[j]));
            }
        }
        if (!ok && lane == 0) record_abort(c, p.status);
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

constexpr size_t smem_bytes() { return 1024 + (size_t)STAGES * SLOT + sizeof(Ctl); }

}  // namespace dfu

// Whole-K items keep every CTA busy once the batch has about half a wave of
// (expert, F tile) units and an item streams at most 512 KB (both matrices):
// larger items leave long tails when the last ones run alone.
bool decode_fused_fits(int T, int d, int E, int k, int F, int num_sms)
{
    const long long rows = (long long)T * k;
    const long long n_exp = E < rows ? E : rows;
    return k <= 2 && rows <= kDecodeTcMaxRows && d % dfu::BM == 0 && F % dfu::BM == 0 &&
           n_exp * (F / dfu::BM) * 2 >= (long long)num_sms * dfu::CTAS_PER_SM &&
           2LL * dfu::BM * d * 2 <= (512 << 10);
}

// Speculative L2 prefetch before the routing is known: when a batch is
// expected to touch most experts (uniform routing: 1 - (1 - k/E)^T >= 1/2),
// the first k-blocks of every expert's gate and up tiles, up to ~32 MB --
// about what HBM delivers while the router ranks and groups the tokens after
// its own operands are in.  Bytes of experts the batch does not use are read
// for nothing, at a time HBM would otherwise idle.
int decode_fused_spec_kb(int T, int d, int E, int k, int F)
{
    const double p_active = 1.0 - pow(1.0 - (double)k / E, (double)T);
    if (p_active < 0.5) return 0;
    const long long per_kb = (long long)E * (F / dfu::BM) * 2 * dfu::A_BYTES;   // one k-block, all tiles
    long long kb = (32LL << 20) / per_kb;
    if (kb > d / dfu::BK) kb = d / dfu::BK;
    return (int)(kb < 0 ? 0 : kb);
}

int decode_fused_max_chunks(int T, int E, int k)
{
    const long long rows = (long long)T * k;
    return (int)((E < rows ? E : rows) + rows / dfu::NTMAX + 1);
}

int decode_fused_flag_words(int T, int E, int k, int F)
{
    return dfu::flag_layout(decode_fused_max_chunks(T, E, k), F).total;
}

cudaError_t launch_decode_fused(const DecodeFusedArgs &a, cudaStream_t stream)
{
    using namespace dfu;
    const int rows = a.T * a.k;
    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap m_wg, m_wu, m_wd;
    if (!tc::make_map(&m_wg, a.w_gate, (uint64_t)a.E * a.F, a.d, BM, bf) ||
        !tc::make_map(&m_wu, a.w_up, (uint64_t)a.E * a.F, a.d, BM, bf) ||
        !tc::make_map(&m_wd, a.w_down, (uint64_t)a.E * a.d, a.F, BM, bf))
        return cudaErrorInvalidValue;

    cudaError_t err;
    const size_t smem = smem_bytes();
    static PerDeviceFlag attr_done;
    const int dev = current_device();
    if (!attr_done.done(dev)) {
        if ((err = cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)smem)) != cudaSuccess)
            return err;
        attr_done.mark(dev);
    }

    Params p{};
    p.offsets = a.offsets; p.E = a.E; p.rows = rows; p.d = a.d; p.F = a.F; p.k = a.k;
    p.nc_max = decode_fused_max_chunks(a.T, a.E, a.k);
    p.spec_kb = decode_fused_spec_kb(a.T, a.d, a.E, a.k, a.F);
    p.x = static_cast<const uint16_t *>(a.x); p.perm_tok = a.perm_tok; p.perm_w = a.perm_w;
    p.h = a.h; p.out = a.out; p.flags = a.flags; p.status = a.status;
    p.expire_ns = a.expire_ns;

    // grid: every CTA slot, or the items there can be at most
    const long long max_items = (long long)p.nc_max * (a.F / BM + a.d / BM);
    const long long slots = (long long)a.num_sms * CTAS_PER_SM;
    const long long g = max_items < slots ? max_items : slots;
    launch_pdl(decode_fused_kernel, dim3((unsigned)(g < 1 ? 1 : g)), dim3(THREADS), smem, stream, m_wg,
               m_wu, m_wd, p);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.ev_done && (err = cudaEventRecord(a.ev_done, stream)) != cudaSuccess) return err;
    return cudaSuccess;
}

}  // namespace moe
