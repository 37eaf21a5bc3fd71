// decode_tc.cu -- expert FFN for decode-sized batches on tcgen05, weights
// streamed by TMA.
//
// At decode sizes an expert holds a handful of token rows, and the layer's
// cost is reading the active experts' weights once from HBM ("Zyphra-ZONOS2-
// 4bit", §Performance notes: batch-1 MoE reads ~1/16 of the experts; batching
// touches more distinct experts until the read is bandwidth bound).  The
// contraction is still dense -- [rows x K] . [K x weight rows] per expert --
// so it runs on the tensor cores with the operands swapped: a 128-row weight
// tile is the M operand (TMA, 128-byte swizzle, an 8-deep ring of 16 KB
// stages per SM), the expert's token rows (padded to 16 or 32) are the N
// operand, and fp32 accumulators live in TMEM.  This keeps the instruction
// count per weight byte near zero, which the CUDA-core version could not.
//
// Two schedules, chosen per kernel by how many work units the batch has:
//  * whole K (enough units to keep every SM streaming in one wave): GATEUP
//    item = (expert, chunk of <= 32 token rows, 128-row tile of F), its ring
//    stages alternating between the gate and the up tile of the same rows
//    into two accumulators; the epilogue writes h = SiLU(G) * U (bf16)
//    directly.  DOWN item = (expert, chunk, 128-row tile of d); the epilogue
//    adds w * y into out[token] (a plain store when k = 1; with k = 2 each
//    element receives exactly two additions onto zero, whose fp32 result does
//    not depend on their order).
//  * split K (small batches, or k > 2): K is split so that every SM streams
//    several items; partial sums go to fp32 scratch and are reduced in split
//    order, so results are bitwise reproducible.
//      GATEUP item = (expert, chunk, matrix, 128-row tile, K split) -> partials
//      Pgu[s][m][row][f]; swiglu: h = SiLU(sum_s G) * sum_s U (bf16);
//      DOWN item -> partials Pd[s][row][o]; combine: out[t] =
//      sum_j w[t,j] * sum_s Pd[s][inv[t,j]] (fp32).
// (An equal split of every layer's k-blocks across CTAs with a fix-up of the
// items cut at range boundaries measured slower on these shapes: the
// fix-ups land at the end of every CTA's range.)
// Both operands of every ring stage arrive by TMA, so the MMA thread only
// waits for data and the epilogue only reads TMEM and stores partials.
//
// CTA: warp 0 = TMA producer, warp 1 = MMA issuer (+ TMEM owner), warps 2-5
// stage the B operand of the next item and drain the accumulator of the
// previous one.  All mbarrier waits are bounded (see sm100.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"
#include "tc_gemm.h"

namespace moe {
namespace dtc {

using namespace sm100;

// Tuning (compile-time): ring depth, resident CTAs per SM, target item count.
#ifndef MOE_DTC_STAGES
#define MOE_DTC_STAGES 4
#endif
#ifndef MOE_DTC_CTAS_PER_SM
#define MOE_DTC_CTAS_PER_SM 2
#endif
#ifndef MOE_DTC_TARGET_ITEMS
#define MOE_DTC_TARGET_ITEMS 304
#endif

constexpr int BM = 128, BK = 64, STAGES = MOE_DTC_STAGES;
constexpr int CTAS_PER_SM = MOE_DTC_CTAS_PER_SM;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB weight tile
constexpr int NTMAX = 32;                       // token rows per item
constexpr int B_BYTES = NTMAX * BK * 2;         // 4 KB token tile (16 or 32 rows used)
constexpr int SLOT = A_BYTES + B_BYTES;         // 20 KB per stage, 1024-aligned
constexpr int KBMAX = 8;                        // k-blocks per item (bf16; kbmax_of)
constexpr int THREADS = 192;
constexpr int THREADS_GATHER = 320;             // + 4 warps that gather the token rows
// 4-bit weights (W4: affine 4-bit or Q4_K, both as packed tiles with one or
// two affine groups per tile row, p.gpr): a stage holds two parts -- k-blocks kb and kb+1 of
// the item's matrix, or (whole-K gate/up items) the gate and the up tile of one
// k-block -- so the waits, commits and loop overheads of the MMA issuer and the
// converters are paid once per two weight tiles.  Layout: two token tiles of 4 KB
// (only one for a gate/up pair, which shares it) and two packed weight tiles
// (q4_tile_offset: 128 x 64 codes, then their fp16 scales and biases; the two
// k-blocks of one row tile are adjacent, one contiguous copy).  Four converter
// warps turn each weight tile into the fp16 A operand of the MMA and store it in
// tensor memory (row i in TMEM lane i, 32 columns per tile, NCVT4 buffers of two
// tiles after the accumulators), so the converted weights never pass through
// shared memory; the MMA issuer waits only for the converters, which have seen
// the stage's copies land.  The MMAs then run
// on fp16 operands: each weight is scale * q + bias rounded once to fp16
// (relative error 2^-11, a quarter of a bf16 rounding), the token rows are
// fp16 rows of x scaled by 2^-xexp[r] (exact for bf16 digits), and h is kept
// in fp16 as h * 2^-2 xexp[r], undone in the down epilogue or the combine.
#ifndef MOE_DTC_STAGES4
#define MOE_DTC_STAGES4 5
#endif
#ifndef MOE_DTC_NCVT4
#define MOE_DTC_NCVT4 2
#endif
constexpr int STAGES4 = MOE_DTC_STAGES4;
constexpr int SLOT4 = 18432;                    // 2 x 4096 + 2 x 5120, 1024-aligned
constexpr int WT_OFF4 = 2 * 4096;               // the two weight tiles (4608 or 5120 bytes each)
static_assert(WT_OFF4 + 2 * kQ4KTileBytes <= SLOT4 && SLOT4 % 1024 == 0, "W4 stage layout");
constexpr int NCVT4 = MOE_DTC_NCVT4;
constexpr int THREADS_W4 = 320;                 // + 4 converter warps
// 8-bit planes (Q8_0, and Q6_K repacked: int8 q plane + fp16 scales per 32 or
// 16 values) take the same converter path: a stage holds two parts, each an
// int8 tile of 128 rows x 64 columns (TMA, 64-byte swizzle, so that the
// converter lanes -- one row each -- read distinct banks) and its scales
// ([64 / group][128] fp16, TMA), beside the fp16 token tiles; the converters
// dequantise q * scale with one rounding to fp16 (dequant16) into the
// A operand in tensor memory.
// Ring depths of the converted kinds: in cluster mode the CTA also holds the
// 16 KB reduction buffer, so its ring is one stage shorter than outside it (a
// deeper 8-bit ring there would leave one CTA per SM).  The extra stage
// outside cluster mode lets the producer run a stage further ahead of the
// converters, whose stage is freed only once the MMAs have read its token
// rows.
#ifndef MOE_DTC_STAGES8
#define MOE_DTC_STAGES8 3
#endif
#ifndef MOE_DTC_STAGES8_WIDE
#define MOE_DTC_STAGES8_WIDE 4
#endif
#ifndef MOE_DTC_STAGES4_WIDE
#define MOE_DTC_STAGES4_WIDE 5
#endif
#ifndef MOE_DTC_STAGES_WIDE
#define MOE_DTC_STAGES_WIDE 4
#endif
constexpr int STAGES8 = MOE_DTC_STAGES8;            // cluster mode
constexpr int STAGES8W = MOE_DTC_STAGES8_WIDE;      // outside cluster mode
constexpr int STAGES4W = MOE_DTC_STAGES4_WIDE;
constexpr int STAGESW = MOE_DTC_STAGES_WIDE;        // bf16 outside cluster mode
constexpr int WT_OFF8 = 2 * 4096;               // two int8 tiles of 8 KB
constexpr int Q8_TILE = 8192;
constexpr int SC_OFF8 = WT_OFF8 + 2 * Q8_TILE;  // two scale boxes of up to 1 KB
constexpr int SC8_MAX = 1024;
constexpr int SLOT8 = SC_OFF8 + 2 * SC8_MAX;    // 26 KB
static_assert(SLOT8 % 1024 == 0, "8-bit stage layout");
constexpr int cmax(int a, int b) { return a > b ? a : b; }
constexpr int kStagesMax = cmax(cmax(cmax(STAGES, STAGESW), STAGES4), cmax(STAGES4W, cmax(STAGES8, STAGES8W)));
// ring of weight kind K: 0 bf16, 1 4-bit tiles, 2 8-bit planes (CL: cluster mode)
template <int K, bool CL = false> struct Ring {
    static constexpr int NST = K == 0 ? (CL ? STAGES : STAGESW) : K == 1 ? (CL ? STAGES4 : STAGES4W)
                                                                : (CL ? STAGES8 : STAGES8W);
    static constexpr int SLOTB = K == 0 ? SLOT : K == 1 ? SLOT4 : SLOT8;
    static constexpr int B_OFF = K == 0 ? A_BYTES : 0;  // token tile
    static constexpr int CTL = NST * SLOTB;
    // TMEM: NACC accumulators of 32 columns, then (converted kinds) NCVT4 A buffers of 32
    static constexpr uint32_t TMEM_COLS = K == 0 ? 128 : 256;
};
constexpr int NACC = 4;                         // TMEM accumulators of 32 columns
constexpr uint32_t A_COL4 = NACC * 32;          // W4: first column of the converted A buffers
static_assert(A_COL4 + NCVT4 * 64 <= 256, "W4 accumulators and A buffers fit in 256 TMEM columns");
constexpr int kTargetItems = MOE_DTC_TARGET_ITEMS;   // ~1 item per CTA: 2 CTAs per SM on a 152-SM GB300
// Cluster mode (CL): the CS CTAs of a cluster take the CS K splits of one
// unit (chunk, 128-row tile), gate/up items covering both matrices; each
// epilogue parks its fp32 accumulators in shared memory, and CTA rank r sums
// rows [r * 128 / CS, (r + 1) * 128 / CS) over the cluster in rank order
// (distributed shared memory) and writes h, or w * y into out -- no partial
// sums in global memory and no reduction kernel.  Chunks of at most 16 token
// rows keep the reduction buffer at 16 KB.
constexpr int NTCL = 16;
constexpr int RED_BYTES = 2 * NTCL * BM * 4;    // [gate, up][16 token columns][128 rows] fp32
#ifndef MOE_DTC_CLUSTER_MAX
#define MOE_DTC_CLUSTER_MAX 8
#endif
constexpr int kClusterMax = 8;                  // (register arrays of the reduction)
constexpr int kClusterUse = MOE_DTC_CLUSTER_MAX;   // largest cluster the launcher picks (0: no cluster mode)

enum Mode { GATEUP = 0, DOWN = 1 };

struct Params {
    const int32_t *offsets;
    int E;
    int K, R, n_mats, KS, kb_total, rows_total, rtiles;
    float *P;            // partial outputs [KS][n_mats][rows_total][R]
    uint32_t *status;
    // GATHER: the token rows come from x[perm_tok[row]] (no grouped copy)
    const uint16_t *xg;  // [T, K] bf16
    const int32_t *perm_tok;
    int fused;           // GATEUP: gate + up tiles per item, h written directly
    uint16_t *h;         //   h [rows_total, R] bf16
    int direct;          // DOWN: w * y added into out directly
    float *out;          //   out [T, R] fp32 (zeroed beforehand when k > 1)
    const float *perm_w;
    int k;
    uint32_t expire_ns;  // > 0: the producer's first wait gives up after this long (test hook)
    const int32_t *xexp; // W4: token row r holds x * 2^-xexp[r] (fp16); h is h * 2^-2 xexp[r]
    int T;               // tokens (debug builds: range of perm_tok)
    const uint8_t *w4[2];  // W4: packed tiles of the matrix (GATEUP: gate, up; DOWN: down)
    int groups;            // W4: K / 64, tiles per row tile
    int gpr;               // W4: affine groups per tile row (1 affine 4-bit, 2 Q4_K)
    int cl;                // cluster mode: CTAs per cluster (= KS); 0 otherwise
    const float *wsc[2];   // fp8: fp32 row scales of the matrices (GATEUP: gate, up; DOWN: down)
};

struct Ctl {
    uint64_t full[kStagesMax], empty[kStagesMax], tfull[NACC], tempty[NACC], drain;
    uint64_t cfull[NCVT4], cempty[NCVT4];   // W4: converted buffers
    uint64_t never;      // nothing arrives here (test hook)
    uint64_t rfull, rfree;   // cluster mode: partials of every CTA parked / read by every CTA
    uint32_t tmem_base;
    int abort_flag;
    int n_items;
    int unit_start[kMaxExperts + 1];
    int off[kMaxExperts + 1];
};

constexpr int kCtlBytes = (int)((sizeof(Ctl) + 15) / 16 * 16);   // the reduction buffer follows

struct Item {
    int e, nc, m, rt, s;
    int row0, nrows, nt, kb0, nkb;
};

// CL: cluster mode (16-row chunks; gate/up items of both matrices over a K split)
template <bool CL>
__device__ __forceinline__ Item decode_item(const Ctl &c, const Params &p, int item)
{
    constexpr int CH = CL ? NTCL : NTMAX;
    int lo = 0, hi = p.E - 1;   // largest e with unit_start[e] <= item
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (c.unit_start[mid] <= item) lo = mid;
        else hi = mid - 1;
    }
    Item it;
    it.e = lo;
    const int units = p.n_mats * p.rtiles * p.KS;
    int local = item - c.unit_start[lo];
    it.nc = local / units;
    local -= it.nc * units;
    it.m = local / (p.rtiles * p.KS);
    local -= it.m * (p.rtiles * p.KS);
    it.rt = local / p.KS;
    it.s = local - it.rt * p.KS;
    const int rows_e = c.off[lo + 1] - c.off[lo];
    it.row0 = c.off[lo] + it.nc * CH;
    it.nrows = min(CH, rows_e - it.nc * CH);
    it.nt = it.nrows <= 16 ? 16 : 32;
    it.kb0 = it.s * p.kb_total / p.KS;
    it.nkb = (it.s + 1) * p.kb_total / p.KS - it.kb0;
    // stages alternate gate / up tiles of each k-block (whole K outside cluster mode)
    if (p.fused) {
        if (CL) it.nkb *= 2;
        else { it.kb0 = 0; it.nkb = 2 * p.kb_total; }
    }
    return it;
}

// Weight matrix and k-block of stage `kbl` of an item.
__device__ __forceinline__ void stage_of(const Params &p, const Item &it, int kbl, int &m, int &kb)
{
    if (p.fused) { m = kbl & 1; kb = it.kb0 + (kbl >> 1); }   // (kb0 = 0 outside cluster mode)
    else { m = it.m; kb = it.kb0 + kbl; }
}

// W4 stages of an item, the parts (1 or 2) of stage st, and part j's matrix,
// k-block and token tile.
template <bool CL>
__device__ __forceinline__ int w4_stages(const Params &p, const Item &it)
{
    return p.fused ? (CL ? it.nkb / 2 : p.kb_total) : (it.nkb + 1) / 2;
}
__device__ __forceinline__ int w4_parts(const Params &p, const Item &it, int st)
{
    return p.fused ? 2 : min(2, it.nkb - 2 * st);
}
template <bool CL>
__device__ __forceinline__ void w4_part(const Params &p, const Item &it, int st, int j, int &m, int &kb, int &tt)
{
    if (p.fused) { m = j; kb = CL ? it.kb0 + st : st; tt = 0; }
    else { m = it.m; kb = it.kb0 + 2 * st + j; tt = j; }
}

// SiLU(z) = z * sigmoid(z) with the fast exponential and an approximate
// divide (relative error ~1e-6, below the bf16 rounding of h that follows).
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// The scaled SwiGLU of the fp16 (W4) path: with g = g' 2^e and u = u' 2^e,
// h * 2^-2e = g' * sigmoid(g' 2^e) * u' -- no 2^-e factor that could overflow.
__device__ __forceinline__ float swiglu_scaled(float g, float u, int e)
{
    return __fdividef(g, 1.0f + __expf(-ldexpf(g, e))) * u;
}

// Warp 0: items per expert (chunks x n_mats x row tiles x K splits), their
// exclusive prefix sums and the item count (0 when the offsets are bad).
template <bool CL>
__device__ __forceinline__ void build_units(Ctl &c, const Params &p, bool offsets_ok, int lane)
{
    constexpr int CH = CL ? NTCL : NTMAX;
    const int E = p.E;
    const int units = p.n_mats * p.rtiles * p.KS;
    int local[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int e = lane * 8 + j;
        int n = 0;
        if (e < E) n = (c.off[e + 1] - c.off[e] + CH - 1) / CH;
        local[j] = n * units;
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
        if (e < E) c.unit_start[e] = run;
        run += local[j];
    }
    if (lane == 31) { c.n_items = offsets_ok ? incl : 0; c.unit_start[E] = incl; }
}

// tm_w0/tm_w1: weight matrices (box 64 x 128 rows); tm_b16/tm_b32: the token
// rows (grouped x for GATEUP, h for DOWN) with boxes of 16 and 32 rows.
// GATHER: the token rows are not loaded by TMA but gathered from x through
// perm_tok by warps 6-9 (stage s by warp 6 + s % 4, lane = token row), written
// into the 128-byte-swizzled layout the MMA expects.
// W4 (affine 4-bit weights): tm_w0/tm_w1 are unused; each stage's weight tile
// is one contiguous copy from p.w4[m], converted to fp16 by warps 6-9.
// WQ: the weight storage, fixed at compile time: 0 bf16; 1 affine 4-bit and
// 2 Q4_K tiles (1 or 2 affine groups per tile row); 3 Q8_0 and 4 Q6_K 8-bit
// planes (a scale per 32 or 16 values); 5 fp8 planes (E4M3 codes widened to
// fp16 exactly; each row's fp32 scale, p.wsc, multiplies its sums in the
// epilogue).  tm_s0/tm_s1: the 8-bit planes' scale maps (GATEUP: gate, up;
// DOWN: down), unused otherwise.
template <int MODE, bool GATHER, int WQ, bool CL = false>
__global__ void __launch_bounds__(GATHER || WQ ? THREADS_GATHER : THREADS, CTAS_PER_SM)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                 const __grid_constant__ CUtensorMap tm_b16, const __grid_constant__ CUtensorMap tm_b32,
                 const __grid_constant__ CUtensorMap tm_s0, const __grid_constant__ CUtensorMap tm_s1,
                 const Params p)
{
    constexpr bool Q8P = WQ == 3 || WQ == 4;   // 8-bit planes with fp16 scale planes
    constexpr bool FP8 = WQ == 5;              // fp8 planes: row scales applied to the sums
    constexpr bool P8 = Q8P || FP8;            // 8-bit tiles by TMA
    constexpr bool W4 = WQ != 0;               // converted weights (4- or 8-bit): fp16 A in TMEM
    static_assert(!(GATHER && W4), "converted weights take the token rows by TMA");
    using RG = Ring<P8 ? 2 : (W4 ? 1 : 0), CL>;
    constexpr int GPR = WQ == 2 ? 2 : 1;       // 4-bit tiles: affine groups per tile row
    constexpr int NSB8 = WQ == 4 ? 4 : 2;      // 8-bit planes: scale blocks per k-block
    constexpr int SCB8 = NSB8 * 128 * 2;       //   their bytes per 128-row tile
    constexpr int STAGES = RG::NST, SLOT = RG::SLOTB;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Ctl &c = *reinterpret_cast<Ctl *>(smem + RG::CTL);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    // set-up that reads nothing the preceding kernels write (barriers, TMEM,
    // tensor-map prefetch) overlaps their tail under programmatic dependent launch
    constexpr int NTHREADS = GATHER || W4 ? THREADS_GATHER : THREADS;
    if (threadIdx.x == 0) {
        // GATHER: a stage is full after the weight tile's bytes and the 32
        // arrivals of the warp that wrote its token rows
        // W4: the four converter warps release a stage
        for (int s = 0; s < STAGES; ++s) { mbar_init(&c.full[s], GATHER ? 33 : 1); mbar_init(&c.empty[s], 1); }
        for (int b = 0; b < NCVT4; ++b) { mbar_init(&c.cfull[b], 4); mbar_init(&c.cempty[b], 1); }
        for (int b = 0; b < NACC; ++b) { mbar_init(&c.tfull[b], 1); mbar_init(&c.tempty[b], 128); }
        mbar_init(&c.drain, 1);
        mbar_init(&c.never, 1);
        if (CL) { mbar_init(&c.rfull, 4 * p.cl); mbar_init(&c.rfree, 4 * p.cl); }
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        if (!W4 || P8)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w0)) : "memory");
        if (MODE == GATEUP && (!W4 || P8))
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w1)) : "memory");
        if (Q8P) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s0)) : "memory");
            if (MODE == GATEUP)
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_s1)) : "memory");
        }
        if (!GATHER) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b16)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b32)) : "memory");
        }
    }
    if (warp == 1) tmem_alloc(&c.tmem_base, RG::TMEM_COLS);
    tc_fence_before();
    if constexpr (MODE == DOWN) {
        // The grouping comes from the router, which completed before the
        // kernel preceding this one passed its dependency wait and let this
        // one start: the unit table is built now, while that kernel finishes
        // (offsets read from L2, never a stale L1 line).  (Streaming the
        // first weight tiles into L2 here as well measured slower: it takes
        // bandwidth from the gate/up kernel still running.)
        for (int e = threadIdx.x; e <= E; e += NTHREADS) c.off[e] = __ldcg(p.offsets + e);
        __syncthreads();
        const bool offsets_ok = debug_offsets_ok(c.off, E, p.rows_total, p.status);
        if (threadIdx.x < 32) build_units<CL>(c, p, offsets_ok, lane);
        pdl_enter();
        if (upstream_failed(p.status)) {   // (synchronises the CTA)
            if (warp == 1) {
                tc_fence_after();
                tmem_dealloc(c.tmem_base, RG::TMEM_COLS);
            }
            return;
        }
    } else {
        pdl_enter();
        // the offsets' loads are in flight with the status read below, whose
        // barrier also publishes them
        for (int e = threadIdx.x; e <= E; e += NTHREADS) c.off[e] = p.offsets[e];
        if (upstream_failed(p.status)) {   // (synchronises the CTA)
            if (warp == 1) {
                tc_fence_after();
                tmem_dealloc(c.tmem_base, RG::TMEM_COLS);
            }
            return;
        }
        const bool offsets_ok = debug_offsets_ok(c.off, E, p.rows_total, p.status);
        if (threadIdx.x < 32) build_units<CL>(c, p, offsets_ok, lane);
    }
    tc_fence_before();
    // cluster mode: peers arrive on this CTA's barriers -- all initialised first
    if (CL) cluster_sync_all();
    else __syncthreads();
    tc_fence_after();

    const uint32_t tmem = c.tmem_base;
    const int n_items = c.n_items;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer: weights + token rows
        uint32_t it_k = 0;
        bool ok = p.expire_ns == 0 || mbar_wait(&c.never, 0, abort_flag, p.expire_ns);
        for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item it = decode_item<CL>(c, p, item);
            const CUtensorMap *bmap = it.nt == 16 ? &tm_b16 : &tm_b32;
            const uint32_t bytes = A_BYTES + (GATHER ? 0 : it.nt * BK * 2);
            const int wrow = it.e * p.R + it.rt * BM;
            if constexpr (P8) {
                const int nst = w4_stages<CL>(p, it);
                for (int st = 0; st < nst; ++st, ++it_k) {
                    const int s = it_k % STAGES;
                    if (!mbar_wait(&c.empty[s], ((it_k / STAGES) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                    const int np = w4_parts(p, it, st), ntok = p.fused ? 1 : np;
                    mbar_expect_tx(&c.full[s], (uint32_t)(np * (Q8_TILE + (Q8P ? SCB8 : 0)) + ntok * it.nt * BK * 2));
                    uint8_t *sp = smem + s * SLOT;
                    for (int j = 0; j < np; ++j) {
                        int m, kb, tt;
                        w4_part<CL>(p, it, st, j, m, kb, tt);
                        const bool second = MODE == GATEUP && m == 1;
                        tma_load_2d(sp + WT_OFF8 + j * Q8_TILE, second ? &tm_w1 : &tm_w0, &c.full[s], kb * BK, wrow);
                        if (Q8P)
                            tma_load_2d(sp + SC_OFF8 + j * SC8_MAX, second ? &tm_s1 : &tm_s0, &c.full[s], wrow,
                                        kb * NSB8);
                    }
                    for (int j = 0; j < ntok; ++j) {
                        int m, kb, tt;
                        w4_part<CL>(p, it, st, j, m, kb, tt);
                        tma_load_2d(sp + tt * B_BYTES, bmap, &c.full[s], kb * BK, it.row0);
                    }
                }
                continue;
            }
            if constexpr (W4) {
                const int nst = w4_stages<CL>(p, it);
                for (int st = 0; st < nst; ++st, ++it_k) {
                    const int s = it_k % STAGES;
                    if (!mbar_wait(&c.empty[s], ((it_k / STAGES) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                    const int np = w4_parts(p, it, st), ntok = p.fused ? 1 : np;
                    const uint32_t tb = (uint32_t)q4_tile_bytes(GPR);
                    mbar_expect_tx(&c.full[s], (uint32_t)(np * tb + ntok * it.nt * BK * 2));
                    uint8_t *sp = smem + s * SLOT;
                    if (p.fused) {   // gate and up tiles of k-block kb0 + st (kb0 = 0 outside cluster mode)
                        const int kb = CL ? it.kb0 + st : st;
                        bulk_load(sp + WT_OFF4, p.w4[0] + q4_tile_offset(wrow, kb, p.groups, GPR), tb, &c.full[s]);
                        bulk_load(sp + WT_OFF4 + tb, p.w4[1] + q4_tile_offset(wrow, kb, p.groups, GPR), tb,
                                  &c.full[s]);
                    } else {         // k-blocks kb, kb + 1: adjacent tiles
                        bulk_load(sp + WT_OFF4, p.w4[it.m] + q4_tile_offset(wrow, it.kb0 + 2 * st, p.groups, GPR),
                                  np * tb, &c.full[s]);
                    }
                    for (int j = 0; j < ntok; ++j) {
                        int m, kb, tt;
                        w4_part<CL>(p, it, st, j, m, kb, tt);
                        tma_load_2d(sp + tt * B_BYTES, bmap, &c.full[s], kb * BK, it.row0);
                    }
                }
                continue;
            }
            for (int kbl = 0; kbl < it.nkb; ++kbl, ++it_k) {
                const int s = it_k % STAGES;
                const uint32_t ph = (it_k / STAGES) & 1u;
                if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                mbar_expect_tx(&c.full[s], bytes);
                int m, kb;
                stage_of(p, it, kbl, m, kb);
                const CUtensorMap *wmap = (MODE == GATEUP && m == 1) ? &tm_w1 : &tm_w0;
                const int kx = kb * BK;
                uint8_t *st = smem + s * SLOT;
                tma_load_2d(st, wmap, &c.full[s], kx, wrow);
                if (!GATHER) tma_load_2d(st + RG::B_OFF, bmap, &c.full[s], kx, it.row0);
            }
        }
        if (!ok) {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            for (uint32_t j = (it_k >= STAGES ? it_k - STAGES : 0); j < it_k; ++j) {
                volatile int no_abort = 0;
                mbar_wait(&c.full[j % STAGES], (j / STAGES) & 1u, &no_abort);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t it_k = 0, li = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x, ++li) {
            const Item it = decode_item<CL>(c, p, item);
            // accumulator slots: NACC of 32 columns, or (fused) NACC/2 pairs of
            // (gate, up) accumulators
            const uint32_t nslot = p.fused ? NACC / 2 : NACC;
            const uint32_t acc = li % nslot, aph = (li / nslot) & 1u;
            if (!mbar_wait(&c.tempty[acc], aph ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t idesc = idesc_f16_mn(W4 ? 1 : 0, BM, it.nt);
            if constexpr (W4) {
                const int nst = w4_stages<CL>(p, it);
                for (int st = 0; st < nst; ++st, ++it_k) {
                    const int s = it_k % STAGES, cb = it_k % NCVT4;
                    // the converters arrive after they have seen the stage land
                    if (!mbar_wait(&c.cfull[cb], (it_k / NCVT4) & 1u, abort_flag)) { ok = false; break; }
                    tc_fence_after();
                    const int np = w4_parts(p, it, st);
                    const uint32_t sp = smem_u32(smem + s * SLOT);
                    const uint32_t a_tm = tmem + A_COL4 + cb * 64;   // A in TMEM: K = 16 is 8 columns
                    for (int j = 0; j < np; ++j) {
                        int m, kb, tt;
                        w4_part<CL>(p, it, st, j, m, kb, tt);
                        const uint32_t d_tmem = tmem + (p.fused ? (acc * 2 + m) * 32 : acc * 32);
                        const uint64_t db = sw128_desc(sp + tt * B_BYTES);
                        const int first = p.fused ? kb - (CL ? it.kb0 : 0) : 2 * st + j;   // 0: first k-block of this accumulator
#pragma unroll
                        for (int kk = 0; kk < BK / 16; ++kk)
                            umma_f16_ts(d_tmem, a_tm + j * 32 + kk * 8, desc_step(db, kk * 32), idesc,
                                        (first | kk) != 0);
                    }
                    umma_commit(&c.empty[s]);
                    umma_commit(&c.cempty[cb]);
                }
                if (!ok) break;
                umma_commit(&c.tfull[acc]);
                continue;
            }
            for (int kbl = 0; kbl < it.nkb; ++kbl, ++it_k) {
                const int s = it_k % STAGES;
                const uint32_t ph = (it_k / STAGES) & 1u;
                if (!mbar_wait(&c.full[s], ph, abort_flag)) { ok = false; break; }
                tc_fence_after();
                int m, kb;
                stage_of(p, it, kbl, m, kb);
                const uint32_t d_tmem = tmem + (p.fused ? (acc * 2 + m) * 32 : acc * 32);
                const uint32_t a0 = smem_u32(smem + s * SLOT);
                const uint32_t b0 = smem_u32(smem + s * SLOT + RG::B_OFF);
                const int first = kb - it.kb0;   // 0: first k-block of this accumulator
                const uint64_t da = sw128_desc(a0), db = sw128_desc(b0);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_f16(d_tmem, desc_step(da, kk * 32), desc_step(db, kk * 32), idesc, (first | kk) != 0);
                umma_commit(&c.empty[s]);
            }
            if (!ok) break;
            umma_commit(&c.tfull[acc]);
        }
        if (!ok) {
            flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
            umma_commit(&c.drain);
            volatile int no_abort = 0;
            mbar_wait(&c.drain, 0, &no_abort);
        }
    } else if (W4 && warp >= 6) {
        // ------------------------------------------------ 4-bit converters (4 warps)
        // a warp may access only the TMEM lanes of its quadrant (warp % 4): warp w
        // converts rows 32 (w % 4) .. +31 of every weight tile, lane = row:
        // 64 codes -> scale * q + bias in fp16 -> 32 columns of its TMEM lane.
        // (q4_word_fp16x8: one packed word -> 8 fp16 weights, an exact fma and a rounded one)
        const int quad = warp & 3, row = quad * 32 + lane;
        const uint32_t t_lane = tmem + ((uint32_t)(quad * 32) << 16) + A_COL4;
        const Q4Fix fx(q4_zero_code(GPR));
        uint32_t it_k = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item it = decode_item<CL>(c, p, item);
            const int nst = w4_stages<CL>(p, it);
            for (int st = 0; st < nst; ++st, ++it_k) {
                const int s = it_k % STAGES, cb = it_k % NCVT4;
                if (!__all_sync(0xffffffffu, mbar_wait(&c.full[s], (it_k / STAGES) & 1u, abort_flag)) ||
                    !__all_sync(0xffffffffu, mbar_wait(&c.cempty[cb], ((it_k / NCVT4) & 1u) ^ 1u, abort_flag))) {
                    ok = false;
                    break;
                }
                const int np = w4_parts(p, it, st);
                if constexpr (P8) {
                    // 8-bit row (64 values, 64-byte swizzled: 16-byte chunk c at
                    // c ^ ((row >> 1) & 3)) -> fp16: int8 q * scale, one
                    // rounding (Q8_0, Q6_K), or E4M3 widened exactly (fp8)
                    for (int j = 0; j < np; ++j) {
                        const uint8_t *wt = smem + s * SLOT + WT_OFF8 + j * Q8_TILE + row * 64;
                        const __half *scp = reinterpret_cast<const __half *>(smem + s * SLOT + SC_OFF8 + j * SC8_MAX);
                        uint32_t o[32];   // column c: values 2c, 2c+1
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch) {   // values 16ch .. 16ch+15
                            const uint4 v = *reinterpret_cast<const uint4 *>(wt + ((ch ^ ((row >> 1) & 3)) << 4));
                            if constexpr (FP8) {
                                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    o[8 * ch + i] = e4m3x2_to_f16x2((uint16_t)(w[i >> 1] >> (16 * (i & 1))));
                            } else {
                                const __half2 sc2 = __half2half2(scp[(ch * NSB8 / 4) * 128 + row]);
                                uint4 lo, hi;
                                dequant16(v, sc2, lo, hi);
                                o[8 * ch + 0] = lo.x; o[8 * ch + 1] = lo.y; o[8 * ch + 2] = lo.z; o[8 * ch + 3] = lo.w;
                                o[8 * ch + 4] = hi.x; o[8 * ch + 5] = hi.y; o[8 * ch + 6] = hi.z; o[8 * ch + 7] = hi.w;
                            }
                        }
                        tmem_st16(t_lane + cb * 64 + j * 32, *reinterpret_cast<const uint32_t(*)[16]>(&o[0]));
                        tmem_st16(t_lane + cb * 64 + j * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&o[16]));
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&c.cfull[cb]);
                    continue;
                }
                constexpr int tb = q4_tile_bytes(GPR), g1 = GPR - 1;   // g1: the second group's index
                for (int j = 0; j < np; ++j) {
                    const uint8_t *wt = smem + s * SLOT + WT_OFF4 + j * tb;
                    const uint4 q0 = *reinterpret_cast<const uint4 *>(wt + row * 32);
                    const uint4 q1 = *reinterpret_cast<const uint4 *>(wt + row * 32 + 16);
                    // scale and bias of values 0-31 and of values 32-63 (the same with one group)
                    const __half *scp = reinterpret_cast<const __half *>(wt + kQ4ScaleOff);
                    const __half *bip = reinterpret_cast<const __half *>(wt + q4_bias_off(GPR));
                    const __half2 sc2[2] = {__half2half2(scp[row]), __half2half2(scp[g1 * BM + row])};
                    const __half2 bi2[2] = {__half2half2(bip[row]), __half2half2(bip[g1 * BM + row])};
                    const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    uint32_t o[32];   // column c: values 2c, 2c+1
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {   // values 8ch .. 8ch+7
                        const uint4 v = q4_word_fp16x8(w[ch], sc2[ch >> 2], bi2[ch >> 2], fx);
                        o[4 * ch + 0] = v.x; o[4 * ch + 1] = v.y; o[4 * ch + 2] = v.z; o[4 * ch + 3] = v.w;
                    }
                    tmem_st16(t_lane + cb * 64 + j * 32, *reinterpret_cast<const uint32_t(*)[16]>(&o[0]));
                    tmem_st16(t_lane + cb * 64 + j * 32 + 16, *reinterpret_cast<const uint32_t(*)[16]>(&o[16]));
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&c.cfull[cb]);
            }
        }
        if (!ok) {
            if (lane == 0) flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
    } else if (GATHER && warp >= 6) {
        // ------------------------------------------------ token-row gatherers (4 warps)
        // warp 6 + w fills the ring stages s with s % 4 == w;
        // lane j copies the 128-byte K slice of the item's j-th token row,
        // zeros for the padding rows of a 16/32-row tile
        const int sw = warp - 6;
        uint32_t it_k = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const Item it = decode_item<CL>(c, p, item);
            const bool has = lane < it.nrows;
            int tok = has ? p.perm_tok[it.row0 + lane] : 0;
            if (has && !debug_index_ok(tok, p.T, p.status)) tok = 0;   // (debug builds)
            const uint16_t *src = p.xg + (size_t)tok * p.K;
            for (int kbl = 0; kbl < it.nkb; ++kbl, ++it_k) {
                const int s = it_k % STAGES;
                if ((s & 3) != sw) continue;
                const uint32_t ph = (it_k / STAGES) & 1u;
                if (!__all_sync(0xffffffffu, mbar_wait(&c.empty[s], ph ^ 1u, abort_flag))) { ok = false; break; }
                if (lane < it.nt) {
                    int m, kb;
                    stage_of(p, it, kbl, m, kb);
                    const int kx = kb * BK;
                    uint4 v[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        v[q] = has ? __ldg(reinterpret_cast<const uint4 *>(src + kx) + q) : make_uint4(0u, 0u, 0u, 0u);
                    uint8_t *dst = smem + s * SLOT + RG::B_OFF + lane * 128;
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<uint4 *>(dst + ((q ^ (lane & 7)) << 4)) = v[q];
                }
                fence_proxy_async_smem();
                mbar_arrive(&c.full[s]);
            }
        }
        if (!ok) {
            if (lane == 0) flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------ epilogue (4 warps)
        const int quarter = warp & 3;
        uint32_t li = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < n_items; item += gridDim.x, ++li) {
            const Item it = decode_item<CL>(c, p, item);
            const uint32_t nslot = p.fused ? NACC / 2 : NACC;
            const uint32_t acc = li % nslot, aph = (li / nslot) & 1u;
            // warp-uniform outcome: tcgen05.ld below is warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&c.tfull[acc], aph, abort_flag))) { ok = false; break; }
            tc_fence_after();
            const int wr = it.rt * BM + quarter * 32 + lane;   // weight row = output column
            if constexpr (CL) {
                // park this split's accumulators (lane = row, 16 token columns;
                // gate/up: G then U) once every CTA has read the previous ones
                float *red = reinterpret_cast<float *>(smem + RG::CTL + kCtlBytes);
                if (!__all_sync(0xffffffffu, mbar_wait(&c.rfree, (li & 1u) ^ 1u, abort_flag))) { ok = false; break; }
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * (MODE == GATEUP ? 64 : 32);
                const int row = quarter * 32 + lane;
                uint32_t v[16];
#pragma unroll
                for (int mt = 0; mt < (MODE == GATEUP ? 2 : 1); ++mt) {
                    // fp8: this row's scale multiplies its partial sums
                    const float rs = FP8 ? p.wsc[mt][(size_t)it.e * p.R + it.rt * BM + row] : 1.f;
                    tmem_ld16(taddr + mt * 32, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) red[(mt * NTCL + q) * BM + row] = __uint_as_float(v[q]) * rs;
                }
                tc_fence_before();
                mbar_arrive(&c.tempty[acc]);
                fence_acq_rel_cluster();
                __syncwarp();
                const int CS = p.cl;
                if (lane < CS) mbar_arrive_release_cluster(peer_addr(&c.rfull, (uint32_t)lane));
                if (!__all_sync(0xffffffffu, mbar_wait_acquire_cluster(&c.rfull, li & 1u, abort_flag))) {
                    ok = false;
                    break;
                }
                // rows [rank * RS, +RS) of the tile: sum over the cluster in rank order
                const int RS = BM / CS, rank = (int)cluster_rank();
                uint32_t base[kClusterMax];
#pragma unroll
                for (int q = 0; q < kClusterMax; ++q) base[q] = q < CS ? peer_addr(red, (uint32_t)q) : 0u;
                for (int idx = quarter * 32 + lane; idx < RS * it.nrows; idx += 128) {
                    const int r = rank * RS + idx % RS, j = idx / RS;
                    float a[kClusterMax], b[kClusterMax];
#pragma unroll
                    for (int q = 0; q < kClusterMax; ++q) {
                        if (q < CS) {
                            a[q] = ld_cluster_f32(base[q] + 4u * (uint32_t)(j * BM + r));
                            if (MODE == GATEUP) b[q] = ld_cluster_f32(base[q] + 4u * (uint32_t)((NTCL + j) * BM + r));
                        }
                    }
                    float ga = a[0], ub = MODE == GATEUP ? b[0] : 0.f;
#pragma unroll
                    for (int q = 1; q < kClusterMax; ++q)
                        if (q < CS) { ga += a[q]; if (MODE == GATEUP) ub += b[q]; }
                    const int col = it.rt * BM + r;
                    if (MODE == GATEUP && W4) {
                        // fp16 h * 2^-2e (the scaled token rows of the 4-bit path)
                        const float hv = swiglu_scaled(ga, ub, p.xexp[it.row0 + j]);
                        if (!(fabsf(hv) <= 65504.f)) flag_status(p.status, kDevCheckFailed);   // h beyond fp16
                        p.h[(size_t)(it.row0 + j) * p.R + col] = __half_as_ushort(__float2half_rn(hv));
                    } else if (MODE == GATEUP) {
                        p.h[(size_t)(it.row0 + j) * p.R + col] = __bfloat16_as_ushort(__float2bfloat16_rn(silu_f(ga) * ub));
                    } else {
                        int tok = p.perm_tok[it.row0 + j];
                        float w = p.perm_w[it.row0 + j];
                        if (W4) w *= ldexpf(1.f, 2 * p.xexp[it.row0 + j]);   // undo h's scale
                        if (!debug_index_ok(tok, p.T, p.status)) { tok = 0; w = 0.f; }   // (debug builds)
                        float *o = p.out + (size_t)tok * p.R + col;
                        if (p.k == 1) *o = w * ga;
                        else atomicAdd(o, w * ga);
                    }
                }
                // (the peers' partials were read: the sums above consumed them)
                __syncwarp();
                if (lane < CS) mbar_arrive_cluster(peer_addr(&c.rfree, (uint32_t)lane));
                continue;
            }
            if (MODE == GATEUP && p.fused) {
                // lane = f; column j = token row j of the chunk; two halves of
                // 16 token columns (the second only for 32-row chunks)
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * 64;
                uint16_t *dst = p.h + (size_t)it.row0 * p.R + wr;
                // W4: lane j holds the scale exponent of token row j (fp16 h, scaled)
                const int e_l = (W4 && lane < it.nrows) ? p.xexp[it.row0 + lane] : 0;
                // fp8: this row's gate and up scales multiply its sums
                const float gs = FP8 ? p.wsc[0][(size_t)it.e * p.R + wr] : 1.f;
                const float us = FP8 ? p.wsc[1][(size_t)it.e * p.R + wr] : 1.f;
                bool out_of_range = false;
                for (int half = 0; half < it.nt / 16; ++half) {
                    uint32_t g[16], u[16];
                    tmem_ld16(taddr + half * 16, g);
                    tmem_ld16(taddr + 32 + half * 16, u);
                    tmem_ld_wait();
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int j = half * 16 + q;
                        if (W4) {
                            const int ej = __shfl_sync(0xffffffffu, e_l, j);
                            if (j < it.nrows) {
                                const float hv = swiglu_scaled(__uint_as_float(g[q]) * gs, __uint_as_float(u[q]) * us, ej);
                                out_of_range |= !(fabsf(hv) <= 65504.f);
                                dst[(size_t)j * p.R] = __half_as_ushort(__float2half_rn(hv));
                            }
                        } else if (j < it.nrows) {
                            const float hv = silu_f(__uint_as_float(g[q])) * __uint_as_float(u[q]);
                            dst[(size_t)j * p.R] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
                        }
                    }
                }
                if (W4 && out_of_range) flag_status(p.status, kDevCheckFailed);   // h beyond fp16
                tc_fence_before();
                mbar_arrive(&c.tempty[acc]);      // accumulators are read
                continue;
            }
            uint32_t v[32];
            const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * 32;
            tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
            if (it.nt > 16) tmem_ld16(taddr + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&c.tempty[acc]);          // accumulator is in registers now
            if constexpr (FP8) {                  // this row's scale multiplies its sums
                const float rs = p.wsc[MODE == GATEUP ? it.m : 0][(size_t)it.e * p.R + wr];
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * rs);
            }
            if (MODE == DOWN && p.direct) {
                // token and routing weight of row j, held by lane j
                int tok_l = lane < it.nrows ? p.perm_tok[it.row0 + lane] : 0;
                float w_l = lane < it.nrows ? p.perm_w[it.row0 + lane] : 0.f;
                if (lane < it.nrows && !debug_index_ok(tok_l, p.T, p.status)) { tok_l = 0; w_l = 0.f; }
                if (W4 && lane < it.nrows) w_l *= ldexpf(1.f, 2 * p.xexp[it.row0 + lane]);   // undo h's scale
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int tok = __shfl_sync(0xffffffffu, tok_l, j);
                    const float w = __shfl_sync(0xffffffffu, w_l, j);
                    if (j < it.nrows) {
                        float *o = p.out + (size_t)tok * p.R + wr;
                        if (p.k == 1) *o = w * __uint_as_float(v[j]);
                        else atomicAdd(o, w * __uint_as_float(v[j]));
                    }
                }
                continue;
            }
            float *dst = p.P + ((size_t)(it.s * p.n_mats + it.m) * p.rows_total + it.row0) * p.R + wr;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < it.nrows) dst[(size_t)j * p.R] = __uint_as_float(v[j]);
        }
        if (!ok) {
            if (lane == 0) flag_status(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
    }

    // cluster mode: no CTA leaves while a peer may still read its shared memory
    if (CL) cluster_sync_all();
    else __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, RG::TMEM_COLS);
    }
}

// The split-K reductions below give each group of 32 float4 columns a block
// of 32 x SL threads: warp sl sums splits sl, sl + SL, ... (loads unrolled so
// several are in flight), and the block adds the SL warps' sums in warp
// order.  The order depends only on (KS, SL), never on which tokens a row
// holds, so results are deterministic and permutation-equivariant.
constexpr int kSplitLanes = 8;

// h[row, f] = SiLU(sum_s G[s][row][f]) * sum_s U[s][row][f], bf16; with xexp
// (the fp16 rows of the 4-bit path) h * 2^-2 xexp[row] in fp16 instead
__global__ void __launch_bounds__(32 * kSplitLanes)
swiglu_reduce_kernel(const float *__restrict__ pgu, int KS, int rows, int F,
                     uint16_t *__restrict__ h, const int32_t *__restrict__ xexp, uint32_t *status)
{
    pdl_enter();
    if (upstream_failed(status)) return;
    __shared__ float4 sg[kSplitLanes][32], su[kSplitLanes][32];
    const int lane = threadIdx.x, sl = threadIdx.y, SL = blockDim.y;
    const long long total = (long long)rows * (F / 4);
    const size_t mat = (size_t)rows * F;
    for (long long base = blockIdx.x * 32LL; base < total; base += gridDim.x * 32LL) {
        const long long i = base + lane;
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
        if (i < total) {
            const size_t o = (size_t)i * 4;
#pragma unroll 4
            for (int s = sl; s < KS; s += SL) {
                const float4 a = __ldcg(reinterpret_cast<const float4 *>(pgu + (size_t)(2 * s) * mat + o));
                const float4 b = __ldcg(reinterpret_cast<const float4 *>(pgu + (size_t)(2 * s + 1) * mat + o));
                g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
                u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
            }
        }
        sg[sl][lane] = g;
        su[sl][lane] = u;
        __syncthreads();
        if (sl == 0 && i < total) {
            for (int w = 1; w < SL; ++w) {
                const float4 a = sg[w][lane], b = su[w][lane];
                g.x += a.x; g.y += a.y; g.z += a.z; g.w += a.w;
                u.x += b.x; u.y += b.y; u.z += b.z; u.w += b.w;
            }
            uint2 packed;
            if (xexp) {
                const int e = xexp[(size_t)i * 4 / F];
                const float h0 = swiglu_scaled(g.x, u.x, e), h1 = swiglu_scaled(g.y, u.y, e);
                const float h2 = swiglu_scaled(g.z, u.z, e), h3 = swiglu_scaled(g.w, u.w, e);
                if (!(fmaxf(fmaxf(fabsf(h0), fabsf(h1)), fmaxf(fabsf(h2), fabsf(h3))) <= 65504.f))
                    flag_status(status, kDevCheckFailed);   // h beyond fp16
                __half2 lo = __floats2half2_rn(h0, h1), hi = __floats2half2_rn(h2, h3);
                packed = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            } else {
                __nv_bfloat162 lo = __floats2bfloat162_rn(silu_f(g.x) * u.x, silu_f(g.y) * u.y);
                __nv_bfloat162 hi = __floats2bfloat162_rn(silu_f(g.z) * u.z, silu_f(g.w) * u.w);
                packed = make_uint2(*reinterpret_cast<uint32_t *>(&lo), *reinterpret_cast<uint32_t *>(&hi));
            }
            *reinterpret_cast<uint2 *>(h + (size_t)i * 4) = packed;
        }
        __syncthreads();
    }
}

// out[t, :] = sum_j w[t, j] * sum_s Pd[s][inv[t, j]][:]   (fixed order: see above);
// with xexp each weight also carries 2^2 xexp[row] (the scaled fp16 h)
__global__ void __launch_bounds__(32 * kSplitLanes)
combine_kernel(const float *__restrict__ pd, int KS, int rows_total, int d,
               const int32_t *__restrict__ inv, const float *__restrict__ topk_w,
               const int32_t *__restrict__ xexp, int T, int k, float *__restrict__ out,
               const uint32_t *status)
{
    pdl_enter();
    if (upstream_failed(status)) return;
    __shared__ float4 sy[kSplitLanes][kMaxTopK][32];
    const int lane = threadIdx.x, sl = threadIdx.y, SL = blockDim.y;
    const int vec = d / 4;
    const long long total = (long long)T * vec;
    for (long long base = blockIdx.x * 32LL; base < total; base += gridDim.x * 32LL) {
        const long long i = base + lane;
        const int t = (int)(i / vec), o = (int)(i - (long long)t * vec) * 4;
        if (i < total) {
            for (int j = 0; j < k; ++j) {
                const int r = inv[t * k + j];
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                for (int s = sl; s < KS; s += SL) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(pd + ((size_t)s * rows_total + r) * d + o));
                    y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
                }
                sy[sl][j][lane] = y;
            }
        }
        __syncthreads();
        if (sl == 0 && i < total) {
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int j = 0; j < k; ++j) {
                float4 y = sy[0][j][lane];
                for (int w = 1; w < SL; ++w) {
                    const float4 v = sy[w][j][lane];
                    y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
                }
                float wt = topk_w[t * k + j];
                if (xexp) wt *= ldexpf(1.f, 2 * xexp[inv[t * k + j]]);
                acc.x += wt * y.x; acc.y += wt * y.y; acc.z += wt * y.z; acc.w += wt * y.w;
            }
            *reinterpret_cast<float4 *>(out + (size_t)t * d + o) = acc;
        }
        __syncthreads();
    }
}

template <int K, bool CL = false> constexpr size_t smem_bytes()
{
    return 1024 + (size_t)Ring<K, CL>::CTL + kCtlBytes + (CL ? RED_BYTES : 0);
}
// two CTAs per SM (228 KB of shared memory, 1 KB reserved per CTA)
static_assert(2 * (smem_bytes<0, false>() + 1024) <= 233472 && 2 * (smem_bytes<0, true>() + 1024) <= 233472 &&
              2 * (smem_bytes<1, false>() + 1024) <= 233472 && 2 * (smem_bytes<1, true>() + 1024) <= 233472 &&
              2 * (smem_bytes<2, false>() + 1024) <= 233472 && 2 * (smem_bytes<2, true>() + 1024) <= 233472,
              "two CTAs per SM");

// Longest split-K item, in k-blocks, by weight storage: a converted kind's item
// pays more to start (its first loads, then the first conversion before any
// MMA), so its items are twice as long as bf16's (ZONOS2 decode T = 64: fp8
// 71.6 -> 69.4, Q8_0 77.7 -> 75.5, affine 4-bit 77.4 -> 74.3 us per layer; at
// T = 8, two waves of items instead of four, the 4-bit and Q8_0 layers are
// ~1 % slower; bf16 was 2 % slower at T = 8 with longer items).
int kbmax_of(int w_dt) { return w_dt == MOE_BF16 ? KBMAX : 2 * KBMAX; }

int choose_splits(int kb_total, long long units, int kbmax)
{
    long long ks = (kTargetItems + units - 1) / (units > 0 ? units : 1);
    const int min_ks = (kb_total + kbmax - 1) / kbmax;   // keep each split <= kbmax k-blocks
    if (ks < min_ks) ks = min_ks;
    if (ks > kb_total) ks = kb_total;
    if (ks < 1) ks = 1;
    return (int)ks;
}

}  // namespace dtc

bool decode_tc_capable(int act_dt, int w_dt, int d, int F, int E)
{
    return act_dt == MOE_BF16 && (w_dt == MOE_BF16 || is_conv(w_dt)) && d % 128 == 0 &&
           F % 128 == 0 && E <= kMaxExperts && tc_gemm_available();
}

void decode_tc_splits(int T, int d, int E, int k, int F, int w_dt, int *ks_gu, int *ks_d)
{
    const long long n_exp = (long long)(E < T * k ? E : T * k);
    const int kbmax = dtc::kbmax_of(w_dt);
    *ks_gu = dtc::choose_splits(d / dtc::BK, n_exp * 2 * (F / dtc::BM), kbmax);
    *ks_d = dtc::choose_splits(F / dtc::BK, n_exp * (d / dtc::BM), kbmax);
}

// Whole-K items stream at a few tens of GB/s per CTA: about 200 of them keep
// HBM busy.  Gate/up items (both matrices, the whole of d) are large, so they
// are used only when they also fit in one wave of the CTAs.
constexpr long long kWholeKMinUnits = 192;

bool decode_tc_gateup_fused(int T, int d, int E, int k, int F, int num_sms)
{
    (void)d;
    const long long n_exp = (long long)(E < T * k ? E : T * k);
    const long long units = n_exp * (F / dtc::BM);
    return units >= kWholeKMinUnits && units <= (long long)num_sms * dtc::CTAS_PER_SM;
}

bool decode_tc_down_direct(int T, int d, int E, int k, int F)
{
    (void)F;
    const long long n_exp = (long long)(E < T * k ? E : T * k);
    return k <= 2 && n_exp * (d / dtc::BM) >= kWholeKMinUnits;
}

// Cluster mode: CS CTAs per unit (CS = 8, 4 or 2) when the kernel's units
// (16-row chunks x 128-row tiles, an upper bound before routing) then fill at
// most one wave of CTAs and every K split keeps at least two k-blocks; 0
// otherwise.  bf16 and 4-bit weights.
static int cluster_size(long long units, int kb_total, int num_sms)
{
    // (allowing two or more waves of clusters measured slower: ZONOS2 decode T = 8
    // 51.3 -> 55.9 / 61.1 us per layer with two / three)
    const long long slots = (long long)num_sms * dtc::CTAS_PER_SM;
    for (int cs = dtc::kClusterUse; cs >= 2; cs /= 2)
        if (units * cs <= slots && kb_total / cs >= 2) return cs;
    return 0;
}
static long long cluster_chunks(int T, int E, int k)
{
    const long long rows = (long long)T * k, n_exp = E < rows ? E : rows;
    return n_exp + rows / dtc::NTCL;
}
int decode_tc_gateup_cluster(int T, int d, int E, int k, int F, int w_dt, int num_sms)
{
    if (!(w_dt == MOE_BF16 || is_conv(w_dt)) || decode_tc_gateup_fused(T, d, E, k, F, num_sms))
        return 0;
    return cluster_size(cluster_chunks(T, E, k) * (F / dtc::BM), d / dtc::BK, num_sms);
}
int decode_tc_down_cluster(int T, int d, int E, int k, int F, int w_dt, int num_sms)
{
    if (!(w_dt == MOE_BF16 || is_conv(w_dt)) || k > 2 || decode_tc_down_direct(T, d, E, k, F))
        return 0;
    return cluster_size(cluster_chunks(T, E, k) * (d / dtc::BM), F / dtc::BK, num_sms);
}
bool decode_tc_down_into_out(int T, int d, int E, int k, int F, int w_dt, int num_sms)
{
    return decode_tc_down_direct(T, d, E, k, F) || decode_tc_down_cluster(T, d, E, k, F, w_dt, num_sms) > 0;
}

namespace dtc {

// Dynamic shared memory of the kernels of weight storage WQ (CL: cluster mode).
template <int WQ, bool CL> constexpr size_t smem_of()
{
    return smem_bytes<WQ >= 3 ? 2 : (WQ ? 1 : 0), CL>();
}
template <int WQ> constexpr int threads_of(bool gather) { return WQ || gather ? THREADS_GATHER : THREADS; }

// One launch of decode_tc_kernel<MODE, GATHER, WQ, CL>: plain, or in
// clusters of `cluster` CTAs; the shared-memory attribute is set once per
// device and instantiation.
template <int MODE, bool GATHER, int WQ, bool CL>
static cudaError_t launch_one(dim3 grid, int cluster, cudaStream_t stream, const CUtensorMap &w0,
                              const CUtensorMap &w1, const CUtensorMap &b16, const CUtensorMap &b32,
                              const CUtensorMap &s0, const CUtensorMap &s1, const Params &p)
{
    static PerDeviceFlag attr_done;
    const int dev = current_device();
    const size_t smem = smem_of<WQ, CL>();
    auto kern = decode_tc_kernel<MODE, GATHER, WQ, CL>;
    cudaError_t err;
    if (!attr_done.done(dev)) {
        if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return err;
        attr_done.mark(dev);
    }
    const dim3 block(threads_of<WQ>(GATHER));
    if (CL) launch_pdl_cluster(kern, grid, block, smem, stream, cluster, w0, w1, b16, b32, s0, s1, p);
    else launch_pdl(kern, grid, block, smem, stream, w0, w1, b16, b32, s0, s1, p);
    return cudaGetLastError();
}

template <int WQ>
static cudaError_t launch_t(const DecodeTcArgs &a, cudaStream_t stream)
{
    constexpr bool conv = WQ != 0;               // converted weights (fp16 operands)
    constexpr bool q8p = WQ == 3 || WQ == 4;     // 8-bit planes with fp16 scale planes
    constexpr bool p8 = q8p || WQ == 5;          // 8-bit tiles (Q8_0, Q6_K, fp8)
    const int rows = a.T * a.k;
    int ks_gu, ks_d;
    decode_tc_splits(a.T, a.d, a.E, a.k, a.F, a.w_dt, &ks_gu, &ks_d);

    const CUtensorMapDataType bf = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    // token rows and h: fp16 when the weights are converted
    const CUtensorMapDataType rowt = conv ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : bf;
    const bool gather = a.x_gather != nullptr && !conv;   // token rows gathered from x in-kernel
    CUtensorMap m_wg, m_wu, m_wd, m_x16, m_x32, m_h16, m_h32, m_sg, m_su, m_sd;
    if (!tc::make_map(&m_h16, a.h, (uint64_t)rows, a.F, 16, rowt) ||
        !tc::make_map(&m_h32, a.h, (uint64_t)rows, a.F, 32, rowt))
        return cudaErrorInvalidValue;
    m_sg = m_su = m_sd = m_h16;   // unused unless 8-bit planes
    const uint64_t gu_rows = (uint64_t)a.E * a.F, d_rows = (uint64_t)a.E * a.d;
    if (p8) {
        const int g8 = WQ == 4 ? 16 : 32;
        if (!tc::make_map_u8(&m_wg, a.w_gate, gu_rows, a.d, BM, true) ||
            !tc::make_map_u8(&m_wu, a.w_up, gu_rows, a.d, BM, true) ||
            !tc::make_map_u8(&m_wd, a.w_down, d_rows, a.F, BM, true))
            return cudaErrorInvalidValue;
        if (q8p && (!tc::make_scale_map(&m_sg, a.w_gate, gu_rows, a.d, g8, BM) ||
                    !tc::make_scale_map(&m_su, a.w_up, gu_rows, a.d, g8, BM) ||
                    !tc::make_scale_map(&m_sd, a.w_down, d_rows, a.F, g8, BM)))
            return cudaErrorInvalidValue;
    } else if (conv) {
        m_wg = m_wu = m_wd = m_h16;   // unused: the 4-bit tiles are contiguous copies
    } else if (!tc::make_map(&m_wg, a.w_gate, gu_rows, a.d, BM, bf) ||
               !tc::make_map(&m_wu, a.w_up, gu_rows, a.d, BM, bf) ||
               !tc::make_map(&m_wd, a.w_down, d_rows, a.F, BM, bf)) {
        return cudaErrorInvalidValue;
    }
    if (gather) {
        m_x16 = m_wg;   // unused by the gathering kernel
        m_x32 = m_wg;
    } else if (!tc::make_map(&m_x16, a.xp, (uint64_t)rows, a.d, 16, rowt) ||
               !tc::make_map(&m_x32, a.xp, (uint64_t)rows, a.d, 32, rowt)) {
        return cudaErrorInvalidValue;
    }

    cudaError_t err;
    const long long n_exp = a.E < rows ? a.E : rows;
    auto grid_for = [&](long long max_items) {
        const long long slots = (long long)a.num_sms * CTAS_PER_SM;
        long long g = max_items < slots ? max_items : slots;
        return dim3((unsigned)(g < 1 ? 1 : g));
    };

    Params p{};
    p.offsets = a.offsets; p.E = a.E; p.rows_total = rows; p.status = a.status;
    p.cl = 0;
    p.xexp = conv ? a.xexp : nullptr;
    p.T = a.T;
    p.w4[0] = static_cast<const uint8_t *>(a.w_gate);
    p.w4[1] = static_cast<const uint8_t *>(a.w_up);
    p.groups = a.d / 64;
    p.gpr = q4_gpr(a.w_dt);
    // fp8: the row scales follow each E4M3 plane at align256(rows * cols)
    auto row_scales = [](const void *w, uint64_t r, int cols) {
        return reinterpret_cast<const float *>(static_cast<const char *>(w) + align_up((size_t)r * cols, 256));
    };
    if (WQ == 5) {
        p.wsc[0] = row_scales(a.w_gate, gu_rows, a.d);
        p.wsc[1] = row_scales(a.w_up, gu_rows, a.d);
    }
    // upper bound on items: chunks <= n_exp + rows / NTMAX
    const long long chunks = n_exp + rows / NTMAX;

    const bool fused = decode_tc_gateup_fused(a.T, a.d, a.E, a.k, a.F, a.num_sms);
    const bool direct = decode_tc_down_direct(a.T, a.d, a.E, a.k, a.F);
    const int cl_gu = decode_tc_gateup_cluster(a.T, a.d, a.E, a.k, a.F, a.w_dt, a.num_sms);
    const int cl_d = decode_tc_down_cluster(a.T, a.d, a.E, a.k, a.F, a.w_dt, a.num_sms);
    const long long chunks_cl = cluster_chunks(a.T, a.E, a.k);
    // grid of a cluster-mode launch: whole clusters, at most one wave
    auto grid_cl = [&](long long units, int cs) {
        const long long per = (long long)a.num_sms * CTAS_PER_SM / cs;
        return dim3((unsigned)((units < per ? units : per) * cs));
    };

    // gate/up: matrices W_g, W_u ([E*F, d]), K = d, token rows = grouped x
    p.K = a.d; p.R = a.F; p.kb_total = a.d / BK; p.rtiles = a.F / BM;
    if (fused) {
        p.n_mats = 1; p.KS = 1; p.fused = 1; p.h = a.h;   // an item covers both matrices
    } else if (cl_gu) {
        p.n_mats = 1; p.KS = cl_gu; p.fused = 1; p.h = a.h; p.cl = cl_gu;
    } else {
        p.n_mats = 2; p.KS = ks_gu; p.P = a.pgu;
    }
    p.expire_ns = a.expire_ns;   // (the gate/up kernel only)
    if (gather) {
        p.xg = static_cast<const uint16_t *>(a.x_gather);
        p.perm_tok = a.perm_tok;
    }
    const dim3 g_gu = cl_gu ? grid_cl(chunks_cl * p.rtiles, cl_gu) : grid_for(chunks * p.n_mats * p.rtiles * p.KS);
    err = cudaSuccess;
    if constexpr (!conv) {   // (only bf16 weights gather token rows in-kernel)
        if (gather && cl_gu)
            err = launch_one<GATEUP, true, WQ, true>(g_gu, cl_gu, stream, m_wg, m_wu, m_x16, m_x32, m_sg, m_su, p);
        else if (gather)
            err = launch_one<GATEUP, true, WQ, false>(g_gu, 0, stream, m_wg, m_wu, m_x16, m_x32, m_sg, m_su, p);
    }
    if (!gather && cl_gu)
        err = launch_one<GATEUP, false, WQ, true>(g_gu, cl_gu, stream, m_wg, m_wu, m_x16, m_x32, m_sg, m_su, p);
    else if (!gather)
        err = launch_one<GATEUP, false, WQ, false>(g_gu, 0, stream, m_wg, m_wu, m_x16, m_x32, m_sg, m_su, p);
    if (err != cudaSuccess) return err;
    // split-K reductions: blocks of 32 float4 columns x min(KS, 8) split lanes
    auto reduce_block = [](int ks) { return dim3(32, ks < kSplitLanes ? (ks < 1 ? 1 : ks) : kSplitLanes); };
    auto reduce_grid = [&](long long total, int ks) {
        long long blocks = (total + 31) / 32;
        const long long cap = (long long)a.num_sms * (64 / reduce_block(ks).y) * 4;
        if (blocks > cap) blocks = cap;
        return (int)(blocks < 1 ? 1 : blocks);
    };
    if (!fused && !cl_gu) {
        launch_pdl(swiglu_reduce_kernel, dim3(reduce_grid((long long)rows * (a.F / 4), ks_gu)), reduce_block(ks_gu),
                   0, stream, a.pgu, ks_gu, rows, a.F, a.h, p.xexp, a.status);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (a.ev_gateup && (err = cudaEventRecord(a.ev_gateup, stream)) != cudaSuccess) return err;

    // down: matrix W_d ([E*d, F]), K = F, token rows = h
    p.K = a.F; p.R = a.d; p.n_mats = 1; p.kb_total = a.F / BK; p.rtiles = a.d / BM;
    p.w4[0] = p.w4[1] = static_cast<const uint8_t *>(a.w_down);
    p.groups = a.F / 64;
    if (WQ == 5) p.wsc[0] = p.wsc[1] = row_scales(a.w_down, d_rows, a.F);
    p.fused = 0; p.h = nullptr;
    p.xg = nullptr;
    p.expire_ns = 0;
    p.cl = 0;
    if (direct) {
        p.KS = 1; p.direct = 1; p.out = a.out; p.perm_tok = a.perm_tok; p.perm_w = a.perm_w; p.k = a.k;
    } else if (cl_d) {
        p.KS = cl_d; p.cl = cl_d; p.direct = 0;
        p.out = a.out; p.perm_tok = a.perm_tok; p.perm_w = a.perm_w; p.k = a.k;
    } else {
        p.KS = ks_d; p.P = a.pd; p.perm_tok = nullptr;
    }
    if (cl_d)
        err = launch_one<DOWN, false, WQ, true>(grid_cl(chunks_cl * p.rtiles, cl_d), cl_d, stream, m_wd, m_wd,
                                                m_h16, m_h32, m_sd, m_sd, p);
    else
        err = launch_one<DOWN, false, WQ, false>(grid_for(chunks * p.rtiles * p.KS), 0, stream, m_wd, m_wd,
                                                 m_h16, m_h32, m_sd, m_sd, p);
    if (err != cudaSuccess) return err;
    if (direct || cl_d) return cudaSuccess;

    launch_pdl(combine_kernel, dim3(reduce_grid((long long)a.T * (a.d / 4), ks_d)), reduce_block(ks_d), 0, stream,
        a.pd, ks_d, rows, a.d, a.inv, a.topk_w, p.xexp, a.T, a.k, a.out, a.status);
    return cudaGetLastError();
}

}  // namespace dtc

cudaError_t launch_decode_tc(const DecodeTcArgs &a, cudaStream_t stream)
{
    switch (a.w_dt) {
    case MOE_BF16: return dtc::launch_t<0>(a, stream);
    case MOE_Q4_A64: return dtc::launch_t<1>(a, stream);
    case MOE_Q4_K: return dtc::launch_t<2>(a, stream);
    case MOE_Q8_0: return dtc::launch_t<3>(a, stream);
    case MOE_Q6_K: return dtc::launch_t<4>(a, stream);
    case MOE_FP8: return dtc::launch_t<5>(a, stream);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace moe
