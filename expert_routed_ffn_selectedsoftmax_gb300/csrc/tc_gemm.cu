// tc_gemm.cu -- grouped expert GEMMs on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA) for prefill-sized batches.
//
// The expert FFN is SwiGLU ("zonos2.cpp internals", §Recommended: expert
// stacks ffn_{gate,up,down}_exps; "New Community Model: ZONOS3-Mini (Zyphra) -
// #1271", §Summary): with many rows per expert it is a set of dense
// contractions, one group per expert, of the rows routed to that expert.
//
// Kernel GATEUP: C = Xp_e . [W_g[e]; W_u[e]]^T over tiles of 128 grouped rows
//   x (128 gate + 128 up columns); the epilogue reads both halves from TMEM
//   and writes h = SiLU(G) * U as 16-bit values, so G and U never reach HBM.
// Kernel DOWN: C = H_e . W_d[e]^T over tiles of 128 rows x 256 model columns;
//   the epilogue scales each row by its routing weight and adds it into
//   out[token] (fp32; a plain store when k == 1; with k > 2 it stores the row
//   and a combine kernel adds each token's k rows in slot order).
//
// Per CTA (persistent, one per SM): warp 0 issues TMA loads of the A (rows)
// and B (weights) tiles into a shared-memory ring (128-byte swizzle); warp 1
// issues tcgen05.mma (M=128, N=256, K=16, fp32 accumulators in TMEM, two
// accumulator buffers of 256 columns); warps 2-9 drain the accumulators, two
// warps per 32-lane TMEM quarter, each taking half of the tile's columns
// (with one warp per scheduler the drain was latency-bound and as slow as
// the mainloop of a tile).  In steady state a 16-bit k-block takes about as
// long as its four MMAs at the tensor pipe's sustained rate (~0.36 us per
// 128x256x64 on every SM at once).
// Tiles are (expert, n-tile, m-tile), m fastest, so CTAs running at the same
// time share weight tiles through L2.  Rows of a tile past the end of the
// expert's group are computed on neighbouring rows (or TMA zero fill) and
// dropped in the epilogue.
//
// Q8_0 weights ("zonos2.cpp internals", §Quantization: 8-bit blocks of 32
// values with one fp16 scale): the B stage holds the int8 tile as loaded by
// TMA; eight converter warps (10-17) turn it into fp16 in the 128-byte-swizzled
// layout -- int8 -> fp16 exactly via the 1024+q bit trick, times the block's
// fp16 scale -- in one of CVT converted-B buffers, and the MMA runs kind::f16
// with fp16 operands (the grouped rows and h are fp16 on this path).
//
// Affine 4-bit weights (the experts of the MLX build, "Zyphra-ZONOS2-4bit",
// §How this was quantized: 4 bits, groups of 64, affine): the B stage holds
// this CTA's packed 128-row tiles (codes, fp16 scales and biases; one
// contiguous copy each) and the same converter warps turn them into fp16,
// scale * q + bias rounded once (q4_word_fp16x8), on the Q8_0 path's fp16
// operands and pairs.
//
// CTA pairs (PAIR, used for Q8_0 and 4-bit): two CTAs of a cluster share one tile of
// 256 grouped rows x 256 columns through tcgen05.mma.cta_group::2 (M = 256):
// each CTA loads its own 128 rows of A and one half of B (GATEUP: the gate
// rows in the even CTA, the up rows in the odd one; DOWN: columns 0-127 /
// 128-255) and converts only that half, and the even CTA's MMA thread
// multiplies the whole tile, reading both CTAs' shared memory; each CTA's
// TMEM receives its own 128 rows.  Halving the per-CTA B part halves the
// converters' work per k-block and leaves room for four converted buffers.
// The odd CTA's loads count their bytes on the even CTA's "stage full"
// barrier (16-bit B) or its converter warps arrive there once its part of B
// is converted (Q8_0); the MMA commits are multicast to the "stage empty" /
// "accumulator full" barriers of both CTAs, and both CTAs' epilogue warps
// arrive on the even CTA's "accumulator empty" barrier.
//
// Every wait on an mbarrier is bounded (2 s of %globaltimer); on timeout the
// waiting role sets the status word, raises a CTA-wide abort flag that the
// other roles poll, waits (bounded) for its own copies or MMAs in flight, and
// the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tc_gemm.h"

// Tuning (compile-time): which grouped GEMMs run as CTA pairs (when clusters
// of two fit on the device): 0 none, 1 Q8_0 weights only, 2 all.  Measured on
// the ZONOS2 Q8_0 prefill layer, pairs with 4 converted buffers took 238 us
// per layer against 249 us for single CTAs; on the ZONOS3-Mini bf16 prefill
// layer (Zipf-skewed experts) single CTAs took 111 us against 114 us, since
// 256-row units pad more rows of small experts.
#ifndef MOE_GEMM_PAIR
#define MOE_GEMM_PAIR 1
#endif

namespace moe {
namespace tc {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int SC_BYTES = BN * (BK / 32) * 2;  // 1 KB (fp16 scales of a 256-row int8 tile)
constexpr int TMEM_COLS = 512;                // 2 accumulators x 256 fp32 columns
constexpr int kMaxStages = 6;

#ifndef MOE_GEMM_CONV_WARPS
#define MOE_GEMM_CONV_WARPS 8
#endif
constexpr int kConvWarps = MOE_GEMM_CONV_WARPS;   // Q8_0 converter warps (4 or 8)
// Q8_0: converted fp16 B buffers and ring stages, pair and single-CTA kernels
#ifndef MOE_GEMM_PAIR_Q8_CVT
#define MOE_GEMM_PAIR_Q8_CVT 4
#endif
#ifndef MOE_GEMM_Q8_CVT
#define MOE_GEMM_Q8_CVT 2
#endif
#ifndef MOE_GEMM_PAIR_Q8_STAGES
#define MOE_GEMM_PAIR_Q8_STAGES 5
#endif
#ifndef MOE_GEMM_Q8_STAGES
#define MOE_GEMM_Q8_STAGES 4
#endif
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;

// Weight storage of a variant: 16-bit, 8-bit planes with a scale per 32 values
// (Q8_0) or per 16 (Q6_K, repacked), 4-bit tiles, or fp8 planes (E4M3 codes;
// each row's fp32 scale multiplies its sums in the epilogue) -- all but the
// first through converter warps.
enum WKind { W16 = 0, WQ8 = 1, WQ4 = 2, WQ6 = 3, WF8 = 4 };

// Per-variant shared-memory layout: a ring of STAGES stages {A, this CTA's
// part of B (16-bit), of Bq (int8) + its scales, or its packed 4-bit tiles},
// then (converted kinds) CVT converted fp16 B buffers, then the control block.
template <int WQ, bool PAIR> struct Cfg {
    static constexpr bool Q8 = WQ != W16;           // converted weights (Q8_0 or 4-bit)
    static constexpr int CL = PAIR ? 2 : 1;
    static constexpr int BNL = BN / CL;             // B rows held by this CTA
    static constexpr int B_BYTES = BNL * BK * 2;    // 16-bit B (this CTA's rows)
    // packed B (4-bit: room for the larger, Q4_K, tiles)
    static constexpr int BQ_BYTES = WQ == WQ4 ? (BNL / kQ4TileRows) * kQ4KTileBytes : BNL * BK;
    // 8-bit planes' scales: per k-block of 64 columns, NSB blocks of BN/2 rows
    static constexpr int NSB = WQ == WQ6 ? 4 : 2;
    // (only the kinds with fp16 scale planes, Q8_0 and Q6_K, load scales)
    static constexpr int SCL_BYTES = (WQ == WQ8 || WQ == WQ6) ? SC_BYTES * (NSB / 2) / CL : 0;
    static constexpr int STAGE = Q8 ? (A_BYTES + BQ_BYTES + SCL_BYTES + 1023) / 1024 * 1024
                                    : A_BYTES + B_BYTES;
    static constexpr int STAGES = Q8 ? (PAIR ? MOE_GEMM_PAIR_Q8_STAGES : MOE_GEMM_Q8_STAGES) : (PAIR ? 6 : 4);
    static constexpr int CVT = Q8 ? (PAIR ? MOE_GEMM_PAIR_Q8_CVT : MOE_GEMM_Q8_CVT) : 0;
    static constexpr int NCVT = CVT > 0 ? CVT : 1;   // (index arithmetic of the 16-bit variants)
    static constexpr int THREADS = Q8 ? 64 + kEpiThreads + 32 * kConvWarps : 64 + kEpiThreads;
    static constexpr size_t CTL = (size_t)STAGES * STAGE + (size_t)CVT * B_BYTES;
    static_assert(STAGES <= kMaxStages && CVT <= 4, "ring deeper than the control block");
};

enum Mode { GATEUP = 0, DOWN = 1 };
// down-epilogue staging: per epilogue warp 32 rows x 16 fp32 columns, rows
// padded to 20 floats (80 B: 16-byte aligned, and 8 consecutive rows fall in
// distinct banks)
constexpr int kStgRow = 20;
constexpr size_t kStgBytes = (size_t)kEpiWarps * 32 * kStgRow * 4;

struct Params {
    const int32_t *offsets;   // [E+1] grouped-row offsets
    int E;
    int K;                    // reduction length (d for GATEUP, F for DOWN)
    int n_tiles;              // N / BN   (GATEUP: F / 128, DOWN: d / 256)
    int F, d, k;
    int rows;                 // grouped rows (T * k)
    uint16_t *h;              // GATEUP output [rows, F] (bf16 or fp16 bits)
    const int32_t *perm_tok;  // DOWN epilogue
    const float *perm_w;
    float *out;
    float *y;                 // DOWN, k > 2: [rows, d] weighted outputs per grouped row
    uint32_t *status;
    int h_fp16;               // GATEUP: write h as fp16 (else bf16)
    const uint8_t *q4[3];     // 4-bit: packed tiles of W_g, W_u, W_d
    int gpr;                  // 4-bit: affine groups per tile row (1 affine 4-bit, 2 Q4_K)
    const int32_t *xexp;      // fp16 rows (Q8_0, 4-bit): row r of the grouped x is scaled by 2^-xexp[r];
                              // h is written scaled by 2^-2 xexp[r], undone in the down epilogue
    float *out_zero;          // GATEUP: `out` to zero for the down kernel's adds, or null
    long long zero4;          // float4 elements of out_zero
    uint32_t expire_ns;       // > 0: the producer's first wait gives up after this long (test hook)
    const float *wsc[3];      // fp8: fp32 row scales of W_g, W_u, W_d
};

// (16-byte aligned size: the down epilogue's float4 staging rows follow it)
struct alignas(16) SmemCtl {
    uint64_t full[kMaxStages], empty[kMaxStages], tfull[2], tempty[2], drain, cfull[4], cempty[4];
    uint64_t never;   // nothing arrives here (test hook)
    uint32_t tmem_base;
    int abort_flag;
    uint32_t fail;
    int n_tiles_total;
    int tile_start[kMaxExperts + 1];
    int mtiles[kMaxExperts];
    int off[kMaxExperts + 1];
};

// SiLU(z) = z * sigmoid(z), with the fast exponential and an approximate
// divide (relative error ~1e-6, far below the 16-bit rounding of h that
// follows; for z < -87, 1 + e^-z overflows and the result is the correct -0).
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// unit -> (expert, m-group, n-tile); tile_start is an exclusive scan over
// experts of mtiles[e] * n_tiles, mtiles[e] the number of CL-row-tile groups
// of expert e; units are m-group fastest, so CTAs running at the same time
// share weight tiles through L2.
__device__ __forceinline__ void decode_tile(const SmemCtl &c, int E, int tile, int &e, int &mt, int &nt)
{
    int lo = 0, hi = E - 1;   // largest e with tile_start[e] <= tile
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (c.tile_start[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    e = lo;
    const int local = tile - c.tile_start[e];
    const int m = c.mtiles[e];
    nt = local / m;
    mt = local - nt * m;
}

// Bounded wait of a whole warp for a barrier phase (warp-uniform result).
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
}

// Arrival of one warp (lane 0, after the warp's prior work) on the barrier
// `bar` of cluster CTA 0 (PAIR) or of this CTA.
template <bool PAIR>
__device__ __forceinline__ void warp_arrive(uint64_t *bar, int lane)
{
    __syncwarp();
    if (lane == 0) {
        if (PAIR) mbar_arrive_cluster(peer_addr(bar, 0));
        else mbar_arrive(bar);
    }
}

// tm_s0/tm_s1 (Q8 only): the B matrices' fp16 scale planes [cols/32, rows],
// box {128 rows, 2 blocks}.
template <int MODE, int WQ, bool PAIR>
__global__ void __launch_bounds__(Cfg<WQ, PAIR>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b0,
                    const __grid_constant__ CUtensorMap tm_b1,
                    const __grid_constant__ CUtensorMap tm_s0,
                    const __grid_constant__ CUtensorMap tm_s1, const Params p)
{
    using C = Cfg<WQ, PAIR>;
    constexpr bool Q8 = C::Q8;   // converted weights (Q8_0 or 4-bit)
    constexpr int CL = C::CL, STAGES = C::STAGES, BNL = C::BNL;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sCvt = smem + STAGES * C::STAGE;   // Q8: converted fp16 B buffers
    SmemCtl &c = *reinterpret_cast<SmemCtl *>(smem + C::CTL);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;
    const uint32_t rank = PAIR ? cluster_rank() : 0u;
    const int cid = blockIdx.x / CL, nclusters = gridDim.x / CL;

    // ---- set-up that reads nothing the preceding kernels write (barriers,
    // TMEM, tensor-map prefetch): under programmatic dependent launch it
    // overlaps the tail of the kernel before
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&c.full[s], 1); mbar_init(&c.empty[s], 1); }
        for (int b = 0; b < 2; ++b) { mbar_init(&c.tfull[b], 1); mbar_init(&c.tempty[b], CL * kEpiWarps); }
        for (int b = 0; b < 4; ++b) { mbar_init(&c.cfull[b], CL * kConvWarps); mbar_init(&c.cempty[b], 1); }
        mbar_init(&c.drain, 1);
        mbar_init(&c.never, 1);
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b0)) : "memory");
        if (MODE == GATEUP)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b1)) : "memory");
    }
    if (warp == 1) {
        if (PAIR) tmem_alloc_pair(&c.tmem_base, TMEM_COLS);
        else tmem_alloc(&c.tmem_base, TMEM_COLS);
    }
    tc_fence_before();
    pdl_enter();
    // ---- status of the kernels before, and the tile table from the
    // grouped-row offsets (harmless arithmetic when the status says failed)
    if (threadIdx.x == 0) c.fail = p.status ? *(volatile const uint32_t *)p.status : 0u;
    for (int e = threadIdx.x; e <= E; e += C::THREADS) c.off[e] = p.offsets[e];
    __syncthreads();
    if (!debug_offsets_ok(c.off, E, p.rows, p.status) && threadIdx.x == 0) c.fail = 1u;   // no tiles run
    if (threadIdx.x < 32) {
        // exclusive scan of mtiles_e * n_tiles over experts (E <= 256: 8 per lane)
        int local[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            int m = 0;
            if (e < E) {
                const int rows = c.off[e + 1] - c.off[e];
                m = (rows + BM * CL - 1) / (BM * CL);   // groups of CL m-tiles
                c.mtiles[e] = m;
            }
            local[j] = m * p.n_tiles;
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
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            if (e < E) c.tile_start[e] = run;
            run += local[j];
        }
        if (lane == 31) { c.n_tiles_total = incl; c.tile_start[E] = incl; }
    }
    tc_fence_before();
    // the peer's arrivals and commits target this CTA's barriers: every
    // barrier of the cluster is initialised before anyone proceeds
    if (PAIR) cluster_sync_all();
    else __syncthreads();
    tc_fence_after();
    // both CTAs of a pair take the same decision (the peer's flag is read
    // before the final cluster barrier, so it is still resident)
    const bool run = (c.fail | (PAIR ? ld_cluster_u32(peer_addr(&c.fail, rank ^ 1u)) : 0u)) == 0u;

    const uint32_t tmem = c.tmem_base;
    const int total = run ? c.n_tiles_total : 0;
    const int kblocks = p.K / BK;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t it = 0;   // global k-block counter across tiles
        bool ok = p.expire_ns == 0 || mbar_wait(&c.never, 0, abort_flag, p.expire_ns);
        for (int tile = cid; tile < total && ok; tile += nclusters) {
            int e, mt, nt;
            decode_tile(c, E, tile, e, mt, nt);
            mt = mt * CL + (int)rank;
            const int arow = c.off[e] + mt * BM;
            // this CTA's B rows: GATEUP (non-pair: gate then up; pair: gate in
            // CTA 0, up in CTA 1), DOWN 256 (non-pair) or 128 rows of W_d
            const int grow = e * p.F + nt * (BN / 2);
            const int drow = e * p.d + nt * BN + (int)rank * BNL;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                uint8_t *st = smem + s * C::STAGE;
                uint8_t *sb = st + A_BYTES;
                uint8_t *sc = st + A_BYTES + C::BQ_BYTES;   // Q8 scales
                if (PAIR && !Q8) {
                    // both CTAs' A and B parts count on CTA 0's stage barrier
                    if (rank == 0) mbar_expect_tx(&c.full[s], 2 * (A_BYTES + C::B_BYTES));
                    const uint32_t bar0 = peer_addr(&c.full[s], 0);
                    tma_load_2d_pair(st, &tm_a, bar0, kb * BK, arow);
                    if (MODE == GATEUP) tma_load_2d_pair(sb, rank ? &tm_b1 : &tm_b0, bar0, kb * BK, grow);
                    else tma_load_2d_pair(sb, &tm_b0, bar0, kb * BK, drow);
                    continue;
                }
                const uint32_t tb = (uint32_t)q4_tile_bytes(p.gpr);   // (4-bit)
                mbar_expect_tx(&c.full[s], A_BYTES + (WQ == WQ4 ? (BNL / kQ4TileRows) * tb
                                                      : Q8 ? C::BQ_BYTES + C::SCL_BYTES : C::B_BYTES));
                tma_load_2d(st, &tm_a, &c.full[s], kb * BK, arow);
                if constexpr (WQ == WQ4) {
                    // this CTA's packed 128-row tiles of k-block kb, one copy each
                    const int groups = p.K / 64;
                    if (MODE == GATEUP) {
                        if (PAIR) {
                            bulk_load(sb, p.q4[rank] + q4_tile_offset(grow, kb, groups, p.gpr), tb, &c.full[s]);
                        } else {
                            bulk_load(sb, p.q4[0] + q4_tile_offset(grow, kb, groups, p.gpr), tb, &c.full[s]);
                            bulk_load(sb + tb, p.q4[1] + q4_tile_offset(grow, kb, groups, p.gpr), tb, &c.full[s]);
                        }
                    } else {
#pragma unroll
                        for (int t = 0; t < BNL / kQ4TileRows; ++t)
                            bulk_load(sb + t * tb, p.q4[2] + q4_tile_offset(drow + t * kQ4TileRows, kb, groups, p.gpr),
                                      tb, &c.full[s]);
                    }
                    continue;
                }
                if (MODE == GATEUP) {
                    if (PAIR) {
                        const CUtensorMap *bm = rank ? &tm_b1 : &tm_b0;
                        tma_load_2d(sb, bm, &c.full[s], kb * BK, grow);
                        if (C::SCL_BYTES > 0) tma_load_2d(sc, rank ? &tm_s1 : &tm_s0, &c.full[s], grow, kb * C::NSB);
                    } else {
                        constexpr int half_b = (Q8 ? C::BQ_BYTES : C::B_BYTES) / 2;
                        tma_load_2d(sb, &tm_b0, &c.full[s], kb * BK, grow);
                        tma_load_2d(sb + half_b, &tm_b1, &c.full[s], kb * BK, grow);
                        if (C::SCL_BYTES > 0) {
                            tma_load_2d(sc, &tm_s0, &c.full[s], grow, kb * C::NSB);
                            tma_load_2d(sc + C::SCL_BYTES / 2, &tm_s1, &c.full[s], grow, kb * C::NSB);
                        }
                    }
                } else {
                    tma_load_2d(sb, &tm_b0, &c.full[s], kb * BK, drow);   // BNL-row box
                    if (C::SCL_BYTES > 0) {
                        tma_load_2d(sc, &tm_s0, &c.full[s], drow, kb * C::NSB);
                        if (!PAIR) tma_load_2d(sc + C::SCL_BYTES / 2, &tm_s0, &c.full[s], drow + BN / 2, kb * C::NSB);
                    }
                }
            }
        }
        if (!ok) {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            // let loads already issued land before the CTA exits
            if (PAIR && !Q8 && rank != 0) {
                // their bytes count on CTA 0's barriers: give them time
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {}
            } else {
                for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
                    volatile int no_abort = 0;
                    mbar_wait(&c.full[j % STAGES], (j / STAGES) & 1u, &no_abort, 1000000ull);
                }
            }
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ------------------------------------------------ MMA issuer (CTA 0 of a pair)
        // fp16 operands on the Q8_0 and 4-bit paths (grouped rows and h are fp16), else bf16
        const uint32_t idesc = idesc_f16_mn(Q8 ? 1 : 0, BM * CL, BN);
        uint32_t it = 0, local_tile = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += nclusters, ++local_tile) {
            const uint32_t acc = local_tile & 1u;
            const uint32_t acc_ph = (local_tile >> 1) & 1u;
            if (!mbar_wait(&c.tempty[acc], acc_ph ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * BN;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait(&c.full[s], ph, abort_flag)) { ok = false; break; }
                const int cb = Q8 ? it % C::NCVT : 0;
                if (Q8 && !mbar_wait(&c.cfull[cb], (it / C::NCVT) & 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + s * C::STAGE);
                const uint32_t b0 = Q8 ? smem_u32(sCvt + cb * C::B_BYTES) : a0 + A_BYTES;
                const uint64_t da = sw128_desc(a0), db = sw128_desc(b0);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    if (PAIR)
                        umma_f16_pair(d_tmem, desc_step(da, kk * 32), desc_step(db, kk * 32), idesc,
                                      (kb | kk) != 0);
                    else
                        umma_f16(d_tmem, desc_step(da, kk * 32), desc_step(db, kk * 32), idesc,
                                 (kb | kk) != 0);
                }
                // frees the stage (and the converted buffer) in both CTAs of a
                // pair once these MMAs have read them
                if (PAIR) {
                    umma_commit_pair_mc(&c.empty[s], 3);
                    if (Q8) umma_commit_pair_mc(&c.cempty[cb], 3);
                } else {
                    umma_commit(&c.empty[s]);
                    if (Q8) umma_commit(&c.cempty[cb]);
                }
            }
            if (!ok) break;
            // accumulator ready for the epilogue warps of both CTAs
            if (PAIR) umma_commit_pair_mc(&c.tfull[acc], 3);
            else umma_commit(&c.tfull[acc]);
        }
        if (!ok) {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            // wait for MMAs in flight before TMEM is freed
            if (PAIR) umma_commit_pair(&c.drain);
            else umma_commit(&c.drain);
            volatile int no_abort = 0;
            mbar_wait(&c.drain, 0, &no_abort);
        }
    } else if (Q8 && warp >= 2 + kEpiWarps) {
        // ------------------------------------------------ Q8_0 converters (kConvWarps warps)
        // lane -> (row in an 8-row pass, 16-byte column chunk of the int8 row);
        // converter warp cw converts rows [cw*BNL/kConvWarps, (cw+1)*BNL/kConvWarps)
        // of this CTA's B rows
        const int cw = warp - 2 - kEpiWarps;
        const int rsub = lane >> 2, q = lane & 3;
        const Q4Fix fx(q4_zero_code(p.gpr));   // (4-bit weights only)
        uint32_t it = 0;
        bool ok = true;
        for (int tile = cid; tile < total && ok; tile += nclusters) {
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const int cb = it % C::NCVT;
                if (!warp_wait(&c.full[s], (it / STAGES) & 1u, abort_flag)) { ok = false; break; }
                if (!warp_wait(&c.cempty[cb], ((it / C::NCVT) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                const uint8_t *bq = smem + s * C::STAGE + A_BYTES;
                const __half *scl = reinterpret_cast<const __half *>(bq + C::BQ_BYTES);
                uint8_t *bo = sCvt + cb * C::B_BYTES;
                if constexpr (WQ == WQ4) {
                    // lane: row rsub of an 8-row pass, values 16q .. 16q+15 (two words)
#pragma unroll
                    for (int pass = 0; pass < BNL / 8 / kConvWarps; ++pass) {
                        const int r = cw * (BNL / kConvWarps) + pass * 8 + rsub;
                        const uint8_t *t = bq + (r / kQ4TileRows) * q4_tile_bytes(p.gpr);
                        const int rr = r % kQ4TileRows;
                        // values 16q .. 16q+15 lie in group q / 2 of two (Q4_K), else in the one group
                        const int gi = (p.gpr - 1) * (q >> 1) * kQ4TileRows + rr;
                        const uint2 v = *reinterpret_cast<const uint2 *>(t + rr * 32 + q * 8);
                        const __half2 sc2 = __half2half2(reinterpret_cast<const __half *>(t + kQ4ScaleOff)[gi]);
                        const __half2 bi2 = __half2half2(reinterpret_cast<const __half *>(t + q4_bias_off(p.gpr))[gi]);
                        *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q) ^ (r & 7)) << 4)) =
                            q4_word_fp16x8(v.x, sc2, bi2, fx);
                        *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q + 1) ^ (r & 7)) << 4)) =
                            q4_word_fp16x8(v.y, sc2, bi2, fx);
                    }
                    fence_proxy_async_smem();
                    warp_arrive<PAIR>(&c.cfull[cb], lane);
                    continue;
                }
                if constexpr (WQ == WF8) {
                    // E4M3 codes widened to fp16 exactly (the row scales act in the epilogue)
#pragma unroll
                    for (int pass = 0; pass < BNL / 8 / kConvWarps; ++pass) {
                        const int r = cw * (BNL / kConvWarps) + pass * 8 + rsub;
                        const uint4 v = *reinterpret_cast<const uint4 *>(bq + r * 64 + q * 16);
                        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                        uint32_t o[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) o[i] = e4m3x2_to_f16x2((uint16_t)(w[i >> 1] >> (16 * (i & 1))));
                        *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q) ^ (r & 7)) << 4)) =
                            make_uint4(o[0], o[1], o[2], o[3]);
                        *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q + 1) ^ (r & 7)) << 4)) =
                            make_uint4(o[4], o[5], o[6], o[7]);
                    }
                    fence_proxy_async_smem();
                    warp_arrive<PAIR>(&c.cfull[cb], lane);
                    continue;
                }
#pragma unroll
                for (int pass = 0; pass < BNL / 8 / kConvWarps; ++pass) {
                    const int r = cw * (BNL / kConvWarps) + pass * 8 + rsub;
                    // scale of (row r, values 16q .. 16q+15): boxes of [NSB blocks][128
                    // rows], a block 32 columns (Q8_0) or 16 (Q6_K)
                    const int blk = C::NSB == 4 ? q : q >> 1;
                    const __half sv = scl[(r >> 7) * (128 * C::NSB) + blk * 128 + (r & 127)];
                    const uint4 v = *reinterpret_cast<const uint4 *>(bq + r * 64 + q * 16);
                    uint4 lo, hi;
                    dequant16(v, __half2half2(sv), lo, hi);
                    *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q) ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q + 1) ^ (r & 7)) << 4)) = hi;
                }
                fence_proxy_async_smem();
                warp_arrive<PAIR>(&c.cfull[cb], lane);
            }
        }
        if (!ok) {
            if (lane == 0) flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
    } else if (warp >= 2 && warp < 2 + kEpiWarps) {
        // ------------------------------------------------ epilogue (8 warps)
        const int quarter = warp & 3;         // TMEM lanes this warp may access
        const int row_in_tile = quarter * 32 + lane;
        const int chalf = (warp - 2) >> 2;    // which half of the tile's columns
        if (MODE == GATEUP && p.out_zero && run) {
            // the down kernel accumulates into `out`: zero this CTA's share of
            // it while the first tile's operands stream in
            float4 *o4 = reinterpret_cast<float4 *>(p.out_zero);
            const long long per = (p.zero4 + gridDim.x - 1) / gridDim.x;
            const long long lo = (long long)blockIdx.x * per;
            const long long hi = lo + per < p.zero4 ? lo + per : p.zero4;
            for (long long i = lo + (threadIdx.x - 64); i < hi; i += kEpiThreads)
                o4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        uint32_t local_tile = 0;
        for (int tile = cid; tile < total; tile += nclusters, ++local_tile) {
            const uint32_t acc = local_tile & 1u;
            const uint32_t acc_ph = (local_tile >> 1) & 1u;
            // warp-uniform outcome: tcgen05.ld below is warp-collective
            if (!warp_wait(&c.tfull[acc], acc_ph, abort_flag)) {
                if (lane == 0) flag_status(p.status, kDevTimeout);
                c.abort_flag = 1;
                break;
            }
            tc_fence_after();
            int e, mt, nt;
            decode_tile(c, E, tile, e, mt, nt);
            mt = mt * CL + (int)rank;
            const int rows_e = c.off[e + 1] - c.off[e];
            const bool valid = mt * BM + row_in_tile < rows_e;
            const int grow = c.off[e] + mt * BM + row_in_tile;
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            if (MODE == GATEUP) {
                // this thread: h columns [chalf*64, chalf*64 + 64) of its row
                constexpr int HC = BN / 4;
                uint16_t *hrow = p.h + (size_t)grow * p.F + nt * (BN / 2) + chalf * HC;
                const uint32_t tg = tbase + chalf * HC, tu = tg + BN / 2;
                // fp16 rows (Q8_0): the accumulators are G / s and U / s for this
                // row's scale s; h / s^2 = (G/s) * sigmoid(G) * (U/s) is what fp16
                // holds (its magnitude is bounded by the weights, whatever x is)
                const float sx = (p.xexp && valid) ? ldexpf(1.f, p.xexp[grow]) : 1.f;
                // fp8: the row scales of this thread's gate and up columns
                const float *gsc = nullptr, *usc = nullptr;
                if constexpr (WQ == WF8) {
                    const size_t r0 = (size_t)e * p.F + nt * (BN / 2) + chalf * HC;
                    gsc = p.wsc[0] + r0;
                    usc = p.wsc[1] + r0;
                }
                bool out_of_range = false;
#pragma unroll 1
                for (int cc = 0; cc < HC; cc += 32) {
                    uint32_t g[2][16], u[2][16];
                    tmem_ld16(tg + cc, g[0]);
                    tmem_ld16(tg + cc + 16, g[1]);
                    tmem_ld16(tu + cc, u[0]);
                    tmem_ld16(tu + cc + 16, u[1]);
                    tmem_ld_wait();
                    uint32_t packed[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int hi = j >> 3, i0 = (2 * j) & 15;
                        float g0 = __uint_as_float(g[hi][i0]), g1 = __uint_as_float(g[hi][i0 + 1]);
                        float u0 = __uint_as_float(u[hi][i0]), u1 = __uint_as_float(u[hi][i0 + 1]);
                        if constexpr (WQ == WF8) {
                            const int cj = cc + 2 * j;
                            g0 *= __ldg(gsc + cj); g1 *= __ldg(gsc + cj + 1);
                            u0 *= __ldg(usc + cj); u1 *= __ldg(usc + cj + 1);
                        }
                        if (p.h_fp16) {
                            const float h0 = __fdividef(g0 * u0, 1.0f + __expf(-sx * g0));
                            const float h1 = __fdividef(g1 * u1, 1.0f + __expf(-sx * g1));
                            out_of_range |= !(fabsf(h0) <= 65504.f) || !(fabsf(h1) <= 65504.f);
                            __half2 v = __floats2half2_rn(h0, h1);
                            packed[j] = *reinterpret_cast<uint32_t *>(&v);
                        } else {
                            const float h0 = silu_f(g0) * u0, h1 = silu_f(g1) * u1;
                            __nv_bfloat162 v = __floats2bfloat162_rn(h0, h1);
                            packed[j] = *reinterpret_cast<uint32_t *>(&v);
                        }
                    }
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(hrow + cc);
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                                packed[4 * q + 3]);
                    }
                }
                // an h beyond fp16's range (weights too large for it) is not silent
                if (__any_sync(0xffffffffu, out_of_range && valid) && lane == 0)
                    flag_status(p.status, kDevCheckFailed);
            } else {
                int tok = 0;
                float wgt = 0.f;
                if (valid) {
                    tok = p.perm_tok[grow];
                    wgt = p.perm_w[grow];
                    if (!debug_index_ok(tok, p.rows / p.k, p.status)) { tok = 0; wgt = 0.f; }   // (debug builds)
                    // fp16 rows (Q8_0): h was held as h / s^2
                    if (p.xexp) wgt *= ldexpf(1.f, 2 * p.xexp[grow]);
                }
                // this warp: output columns [chalf*128, chalf*128 + 128) of its 32
                // rows, in chunks of 16 columns.  A chunk is transposed through
                // shared memory so that each store / reduction instruction of the
                // warp covers 8 rows x 64 contiguous bytes (lane l: row l/4 + 8i,
                // columns 4(l%4)..+3) instead of 32 rows x 16 bytes.
                float *stg = reinterpret_cast<float *>(smem + C::CTL + sizeof(SmemCtl)) +
                             (warp - 2) * 32 * kStgRow;
                const uint32_t tv = tbase + chalf * (BN / 2);
                // fp8: the row scales of this warp's output columns
                const float *dsc = WQ == WF8 ? p.wsc[2] + (size_t)e * p.d + nt * BN + chalf * (BN / 2) : nullptr;
#pragma unroll 1
                for (int cc = 0; cc < BN / 2; cc += 16) {
                    uint32_t v[16];
                    tmem_ld16(tv + cc, v);
                    tmem_ld_wait();
                    if constexpr (WQ == WF8) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * __ldg(dsc + cc + i));
                    }
                    float4 *srow = reinterpret_cast<float4 *>(stg + lane * kStgRow);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        srow[j] = make_float4(wgt * __uint_as_float(v[4 * j]), wgt * __uint_as_float(v[4 * j + 1]),
                                              wgt * __uint_as_float(v[4 * j + 2]), wgt * __uint_as_float(v[4 * j + 3]));
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int r = (lane >> 2) + 8 * i;          // row within the warp's 32
                        const int rt = __shfl_sync(0xffffffffu, tok, r);
                        const int rg = __shfl_sync(0xffffffffu, grow, r);
                        const bool rv = __shfl_sync(0xffffffffu, valid ? 1 : 0, r) != 0;
                        const float4 val = *reinterpret_cast<const float4 *>(stg + r * kStgRow + (lane & 3) * 4);
                        if (rv) {
                            const size_t col = (size_t)(nt * BN + chalf * (BN / 2) + cc + (lane & 3) * 4);
                            if (p.k > 2) {
                                // the grouped row's weighted output; the combine kernel
                                // adds each token's k rows in slot order
                                *reinterpret_cast<float4 *>(p.y + (size_t)rg * p.d + col) = val;
                            } else {
                                // k = 1: the only contribution; k = 2: two additions
                                // onto zero, whose result does not depend on their order
                                float *o = p.out + (size_t)rt * p.d + col;
                                if (p.k == 1) *reinterpret_cast<float4 *>(o) = val;
                                else red_add_v4(o, val.x, val.y, val.z, val.w);
                            }
                        }
                    }
                    __syncwarp();
                }
            }
            tc_fence_before();
            warp_arrive<PAIR>(&c.tempty[acc], lane);
        }
    }

    // no CTA leaves while its peer may still read its shared memory, arrive
    // on its barriers or (CTA 0) have MMAs writing its TMEM
    if (PAIR) cluster_sync_all();
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (PAIR) tmem_dealloc_pair(tmem, TMEM_COLS);
        else tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int WQ, bool PAIR> constexpr size_t smem_bytes()
{
    // ring (+ converted B buffers), control block, down-epilogue staging
    return 1024 + Cfg<WQ, PAIR>::CTL + sizeof(SmemCtl) + kStgBytes;
}
static_assert(sizeof(SmemCtl) % 16 == 0, "the staging rows after the control block take float4 stores");
static_assert(smem_bytes<W16, true>() <= 232448 && smem_bytes<WQ8, true>() <= 232448 &&
                  smem_bytes<W16, false>() <= 232448 && smem_bytes<WQ8, false>() <= 232448 &&
                  smem_bytes<WQ4, true>() <= 232448 && smem_bytes<WQ4, false>() <= 232448 &&
                  smem_bytes<WQ6, true>() <= 232448 && smem_bytes<WQ6, false>() <= 232448 &&
                  smem_bytes<WF8, true>() <= 232448 && smem_bytes<WF8, false>() <= 232448,
              "shared memory per CTA");

// ------------------------------------------------------------------- host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (!f) {
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn.store(f);
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// 2-D row-major [rows, cols] int8 tensor, box {64 cols, box_rows}, no swizzle
// (the GEMM converters read it row by row) or 64-byte swizzle (the decode
// converters: one row per lane).
bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                 bool swizzle64)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The fp16 scale plane [cols/group, rows] of an 8-bit packed buffer (at
// align256(rows * cols)), box {box_rows rows, 64/group blocks}: the scales of
// one k-block of a weight tile.
bool make_scale_map(CUtensorMap *m, const void *packed, uint64_t rows, uint64_t cols, int group,
                    uint32_t box_rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    const void *base = static_cast<const char *>(packed) + align_up((size_t)(rows * cols), 256);
    cuuint64_t dims[2] = {rows, cols / (uint64_t)group};
    cuuint64_t strides[1] = {rows * 2};
    cuuint32_t box[2] = {box_rows, (cuuint32_t)(64 / group)};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D row-major [rows, cols] 16-bit tensor, box {64 cols, box_rows}, 128B swizzle.
bool make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
              CUtensorMapDataType dt)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tc

bool tc_gemm_available() { return tc::encode_fn() != nullptr; }
bool tc_gemm_supports(moe_dtype w_dt) { return w_dt == MOE_BF16 || is_conv(w_dt); }

bool tc_gemm_prefer(int T, int d, int E, int k, int F)
{
    (void)d; (void)F;
    // grouped GEMMs pay off once experts hold whole 128-row tiles on average
    return (long long)T * k >= 64LL * E && T >= 512;
}

template <int WQ, bool PAIR>
static cudaError_t set_smem_attrs()
{
    using namespace tc;
    static PerDeviceFlag done;
    const int dev = current_device();
    if (done.done(dev)) return cudaSuccess;
    const int smem = (int)smem_bytes<WQ, PAIR>();
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(grouped_gemm_kernel<GATEUP, WQ, PAIR>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grouped_gemm_kernel<DOWN, WQ, PAIR>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return err;
    done.mark(dev);
    return cudaSuccess;
}

// Clusters of two CTAs (pair kernels) that can be resident at once (0 if the
// query fails).
template <int MODE, int WQ>
static int max_active_pairs()
{
    using namespace tc;
    static PerDeviceInt cached;
    const int dev = current_device();
    int n = cached.get(dev);
    if (n >= 0) return n;
    // the query needs the kernel's dynamic shared-memory limit raised first
    if (set_smem_attrs<WQ, true>() != cudaSuccess) {
        cudaGetLastError();
        cached.put(dev, 0);
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * device_sm_count());
    cfg.blockDim = dim3(Cfg<WQ, true>::THREADS);
    cfg.dynamicSmemBytes = smem_bytes<WQ, true>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_kernel<MODE, WQ, true>, &cfg) != cudaSuccess)
        n = 0;
    cudaGetLastError();   // clear a failed query
    cached.put(dev, n);
    return n;
}

bool tc_gemm_pairs(moe_dtype w_dt)
{
    const bool q8 = is_q8p(w_dt) || is_fp8(w_dt), q4 = is_q4(w_dt);
    if (MOE_GEMM_PAIR == 0 || (MOE_GEMM_PAIR == 1 && !q8 && !q4)) return false;
    if constexpr (MOE_GEMM_PAIR >= 2) {
        if (!q8 && !q4)
            return max_active_pairs<tc::GATEUP, tc::W16>() > 0 && max_active_pairs<tc::DOWN, tc::W16>() > 0;
    }
    if (q4) return max_active_pairs<tc::GATEUP, tc::WQ4>() > 0 && max_active_pairs<tc::DOWN, tc::WQ4>() > 0;
    if (w_dt == MOE_Q6_K)
        return max_active_pairs<tc::GATEUP, tc::WQ6>() > 0 && max_active_pairs<tc::DOWN, tc::WQ6>() > 0;
    if (is_fp8(w_dt))
        return max_active_pairs<tc::GATEUP, tc::WF8>() > 0 && max_active_pairs<tc::DOWN, tc::WF8>() > 0;
    return q8 && max_active_pairs<tc::GATEUP, tc::WQ8>() > 0 && max_active_pairs<tc::DOWN, tc::WQ8>() > 0;
}

template <int WQ, bool PAIR>
static cudaError_t launch_gemms(const TcArgs &a, tc::Params p, const CUtensorMap &m_xp,
                                const CUtensorMap &m_wg, const CUtensorMap &m_wu,
                                const CUtensorMap &m_h, const CUtensorMap &m_wd,
                                const CUtensorMap &m_sg, const CUtensorMap &m_su,
                                const CUtensorMap &m_sd, cudaStream_t stream)
{
    using namespace tc;
    constexpr int CL = Cfg<WQ, PAIR>::CL;
    cudaError_t err;
    if ((err = set_smem_attrs<WQ, PAIR>()) != cudaSuccess) return err;
    const int rows = a.T * a.k;
    // upper bound on units: every expert could own a ragged group of CL m-tiles
    const long long max_groups = rows / (BM * CL) + (a.E < rows ? a.E : rows);
    auto grid_for = [&](long long units, int max_clusters) {
        long long cl = units < max_clusters ? units : max_clusters;
        return dim3((unsigned)((cl < 1 ? 1 : cl) * CL));
    };
    const size_t smem = smem_bytes<WQ, PAIR>();
    const dim3 block(Cfg<WQ, PAIR>::THREADS);

    p.K = a.d; p.n_tiles = a.F / (BN / 2);
    const dim3 g1 = grid_for(max_groups * p.n_tiles, PAIR ? max_active_pairs<GATEUP, WQ>() : a.num_sms);
    if (PAIR)
        err = launch_pdl_cluster(grouped_gemm_kernel<GATEUP, WQ, PAIR>, g1, block, smem, stream, CL,
                                 m_xp, m_wg, m_wu, m_sg, m_su, p);
    else
        err = launch_pdl(grouped_gemm_kernel<GATEUP, WQ, PAIR>, g1, block, smem, stream, m_xp, m_wg,
                         m_wu, m_sg, m_su, p);
    if (err != cudaSuccess || (err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.ev_gateup && (err = cudaEventRecord(a.ev_gateup, stream)) != cudaSuccess) return err;

    p.K = a.F; p.n_tiles = a.d / BN;
    p.expire_ns = 0;   // (the hook acts on the gate/up kernel only)
    const dim3 g2 = grid_for(max_groups * p.n_tiles, PAIR ? max_active_pairs<DOWN, WQ>() : a.num_sms);
    if (PAIR)
        err = launch_pdl_cluster(grouped_gemm_kernel<DOWN, WQ, PAIR>, g2, block, smem, stream, CL, m_h,
                                 m_wd, m_wd, m_sd, m_sd, p);
    else
        err = launch_pdl(grouped_gemm_kernel<DOWN, WQ, PAIR>, g2, block, smem, stream, m_h, m_wd, m_wd,
                         m_sd, m_sd, p);
    if (err != cudaSuccess || (err = cudaGetLastError()) != cudaSuccess || a.k <= 2) return err;
    return launch_combine_rows(a.y, a.d, a.inv, a.T, a.k, a.out, a.status, a.num_sms, stream);
}

cudaError_t launch_tc_experts(const TcArgs &a, cudaStream_t stream)
{
    using namespace tc;
    const bool q8 = is_q8p(a.w_dt), q4 = is_q4(a.w_dt), f8 = is_fp8(a.w_dt);
    const bool f16 = q8 || q4 || f8;   // fp16 operands (converted weights)
    const int g8 = q8_group(a.w_dt);   // values per scale of the 8-bit planes
    if (!f16 && a.w_dt != MOE_BF16) return cudaErrorNotSupported;
    const int rows = a.T * a.k;
    cudaError_t err = cudaSuccess;
    if (!a.xp_ready &&
        (err = launch_gather_rows(a.x, a.d, a.perm_tok, rows, a.xp, f16 ? 1 : 0, a.xexp, a.T, a.status,
                                   a.num_sms, stream)) !=
            cudaSuccess)
        return err;
    if (a.ev_gathered && (err = cudaEventRecord(a.ev_gathered, stream)) != cudaSuccess) return err;

    // pairs of CTAs when clusters of two can be resident, else single CTAs
    const bool pair = tc_gemm_pairs(a.w_dt);

    // activations: bf16, or fp16 on the Q8_0 and 4-bit paths
    const CUtensorMapDataType act = f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t gu_rows = (uint64_t)a.E * a.F, d_rows = (uint64_t)a.E * a.d;
    const uint32_t wd_box = (uint32_t)(pair ? BN / 2 : BN);   // each CTA of a pair: 128 rows of W_d
    CUtensorMap m_xp, m_wg, m_wu, m_h, m_wd;
    bool ok = make_map(&m_xp, a.xp, rows, a.d, BM, act) && make_map(&m_h, a.h, rows, a.F, BM, act);
    if (q4) {
        m_wg = m_wu = m_wd = m_xp;   // unused: the 4-bit tiles are contiguous copies
    } else if (q8 || f8) {
        ok = ok && make_map_u8(&m_wg, a.w_gate, gu_rows, a.d, BN / 2) &&
             make_map_u8(&m_wu, a.w_up, gu_rows, a.d, BN / 2) &&
             make_map_u8(&m_wd, a.w_down, d_rows, a.F, wd_box);
    } else {
        ok = ok && make_map(&m_wg, a.w_gate, gu_rows, a.d, BN / 2, act) &&
             make_map(&m_wu, a.w_up, gu_rows, a.d, BN / 2, act) &&
             make_map(&m_wd, a.w_down, d_rows, a.F, wd_box, act);
    }
    if (!ok) return cudaErrorInvalidValue;

    // 8-bit packed buffers: int8 plane, then the fp16 scale plane [cols/g8, rows]
    // at align256(rows * cols); maps with box {128 rows, 64/g8 blocks}
    auto scale_map = [g8](CUtensorMap *m, const void *packed, uint64_t r, uint64_t cols) {
        return make_scale_map(m, packed, r, cols, g8, (uint32_t)(BN / 2));
    };
    CUtensorMap m_sg = m_xp, m_su = m_xp, m_sd = m_xp;   // unused unless Q8_0
    if (q8 && !(scale_map(&m_sg, a.w_gate, gu_rows, a.d) && scale_map(&m_su, a.w_up, gu_rows, a.d) &&
                scale_map(&m_sd, a.w_down, d_rows, a.F)))
        return cudaErrorInvalidValue;

    Params p{};
    p.offsets = a.offsets; p.E = a.E; p.F = a.F; p.d = a.d; p.k = a.k; p.rows = a.T * a.k;
    p.h = static_cast<uint16_t *>(a.h); p.perm_tok = a.perm_tok; p.perm_w = a.perm_w;
    p.out = a.out; p.y = a.y; p.status = a.status; p.h_fp16 = f16 ? 1 : 0;
    p.xexp = f16 ? a.xexp : nullptr;
    p.q4[0] = static_cast<const uint8_t *>(a.w_gate);
    p.q4[1] = static_cast<const uint8_t *>(a.w_up);
    p.q4[2] = static_cast<const uint8_t *>(a.w_down);
    p.gpr = q4_gpr(a.w_dt);
    p.out_zero = a.zero_out ? a.out : nullptr;
    p.zero4 = (long long)a.T * a.d / 4;
    p.expire_ns = a.expire_ns;
    if (f8) {   // the fp32 row scales follow each E4M3 plane at align256(rows * cols)
        auto rs = [](const void *w, uint64_t r, int cols) {
            return reinterpret_cast<const float *>(static_cast<const char *>(w) + align_up((size_t)r * cols, 256));
        };
        p.wsc[0] = rs(a.w_gate, gu_rows, a.d);
        p.wsc[1] = rs(a.w_up, gu_rows, a.d);
        p.wsc[2] = rs(a.w_down, d_rows, a.F);
        return pair ? launch_gemms<WF8, true>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream)
                    : launch_gemms<WF8, false>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream);
    }
    if (q4)
        return pair ? launch_gemms<WQ4, true>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream)
                    : launch_gemms<WQ4, false>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream);
    if (a.w_dt == MOE_Q6_K)
        return pair ? launch_gemms<WQ6, true>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream)
                    : launch_gemms<WQ6, false>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream);
    if (q8)
        return pair ? launch_gemms<WQ8, true>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream)
                    : launch_gemms<WQ8, false>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream);
    if constexpr (MOE_GEMM_PAIR >= 2) {
        if (pair)
            return launch_gemms<W16, true>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream);
    }
    return launch_gemms<W16, false>(a, p, m_xp, m_wg, m_wu, m_h, m_wd, m_sg, m_su, m_sd, stream);
}

}  // namespace moe
