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
//   out[token] (fp32; a plain store when k == 1).
//
// Per CTA (persistent, one per SM): warp 0 issues TMA loads of the A (rows)
// and B (weights) tiles into a 4-stage shared-memory ring (128-byte swizzle);
// warp 1 issues tcgen05.mma (M=128, N=256, K=16, fp32 accumulators in TMEM,
// two accumulator buffers of 256 columns); warps 2-5 drain the accumulators.
// Tiles are (expert, n-tile, m-tile), m fastest, so CTAs running at the same
// time share weight tiles through L2.  Rows of a tile past the end of the
// expert's group are computed on neighbouring rows (or TMA zero fill) and
// dropped in the epilogue.
//
// Q8_0 weights ("zonos2.cpp internals", §Quantization: 8-bit blocks of 32
// values with one fp16 scale): the B stage holds the int8 tile as loaded by
// TMA; four converter warps (6-9) turn it into fp16 in the 128-byte-swizzled
// layout -- int8 -> fp16 exactly via the 1024+q bit trick, times the block's
// fp16 scale -- in one of two converted-B buffers, and the MMA runs kind::f16
// with fp16 operands (the grouped rows and h are fp16 on this path).
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

namespace moe {
namespace tc {

using namespace sm100;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;          // 16 KB
constexpr int B_BYTES = BN * BK * 2;          // 32 KB (16-bit B tile)
constexpr int BQ_BYTES = BN * BK;             // 16 KB (int8 B tile)
constexpr int SC_BYTES = BN * (BK / 32) * 2;  // 1 KB (fp16 scales of the int8 tile)
constexpr int TMEM_COLS = 512;                // 2 accumulators x 256 fp32 columns

// Per-variant shared-memory layout: a ring of STAGES stages {A, B or Bq},
// then (Q8 only) two converted fp16 B buffers, then the control block.
template <bool Q8> struct Cfg {
    static constexpr int STAGE = Q8 ? (A_BYTES + BQ_BYTES + SC_BYTES + 1023) / 1024 * 1024
                                    : A_BYTES + B_BYTES;
    static constexpr int CVT = Q8 ? 2 : 0;
    static constexpr int THREADS = Q8 ? 320 : 192;
    static constexpr size_t CTL = (size_t)STAGES * STAGE + (size_t)CVT * B_BYTES;
};

enum Mode { GATEUP = 0, DOWN = 1 };

struct Params {
    const int32_t *offsets;   // [E+1] grouped-row offsets
    int E;
    int K;                    // reduction length (d for GATEUP, F for DOWN)
    int n_tiles;              // N / BN   (GATEUP: F / 128, DOWN: d / 256)
    int F, d, k;
    uint16_t *h;              // GATEUP output [rows, F] (bf16 or fp16 bits)
    const int32_t *perm_tok;  // DOWN epilogue
    const float *perm_w;
    float *out;
    uint32_t *status;
    int h_fp16;               // GATEUP: write h as fp16 (else bf16)
};

struct SmemCtl {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, cfull[2], cempty[2];
    uint32_t tmem_base;
    int abort_flag;
    int n_tiles_total;
    int tile_start[kMaxExperts + 1];
    int mtiles[kMaxExperts];
    int off[kMaxExperts + 1];
};

// Instruction descriptor for the M = 128, N = 256 tiles of this file.
__host__ __device__ constexpr uint32_t idesc_f16(int ab_fp16) { return idesc_f16_mn(ab_fp16, BM, BN); }

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

// tile -> (expert, m-tile, n-tile); tile_start is an exclusive scan over experts
__device__ __forceinline__ void decode_tile(const SmemCtl &c, int E, int n_tiles, int tile,
                                            int &e, int &mt, int &nt)
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
    (void)n_tiles;
}

// int8 x 16 (one uint4) -> fp16 x 16 scaled by s: (q ^ 0x80) placed in the
// mantissa of 1024.0 gives 1024 + 128 + q exactly; subtracting 1152 leaves q.
__device__ __forceinline__ void dequant16(const uint4 q, const __half2 s, uint4 &lo, uint4 &hi)
{
    const uint32_t w[4] = {q.x ^ 0x80808080u, q.y ^ 0x80808080u, q.z ^ 0x80808080u,
                           q.w ^ 0x80808080u};
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t a = __byte_perm(w[i], 0x64646464u, 0x4140);
        uint32_t b = __byte_perm(w[i], 0x64646464u, 0x4342);
        __half2 ha = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&a), bias), s);
        __half2 hb = __hmul2(__hsub2(*reinterpret_cast<__half2 *>(&b), bias), s);
        o[2 * i] = *reinterpret_cast<uint32_t *>(&ha);
        o[2 * i + 1] = *reinterpret_cast<uint32_t *>(&hb);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// tm_s0/tm_s1 (Q8 only): the B matrices' fp16 scale planes [cols/32, rows],
// box {rows of the tile, 2 blocks}.
template <int MODE, bool Q8>
__global__ void __launch_bounds__(Cfg<Q8>::THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b0,
                    const __grid_constant__ CUtensorMap tm_b1,
                    const __grid_constant__ CUtensorMap tm_s0,
                    const __grid_constant__ CUtensorMap tm_s1, const Params p)
{
    pdl_enter();
    using C = Cfg<Q8>;
    constexpr int THREADS = C::THREADS;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sCvt = smem + STAGES * C::STAGE;   // Q8: converted fp16 B buffers
    SmemCtl &c = *reinterpret_cast<SmemCtl *>(smem + C::CTL);

    if (upstream_failed(p.status)) return;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E;

    // ---- set-up: barriers, tile table, TMEM
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(&c.full[s], 1); mbar_init(&c.empty[s], 1); }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&c.tfull[b], 1); mbar_init(&c.tempty[b], 128);
            mbar_init(&c.cfull[b], 128); mbar_init(&c.cempty[b], 1);
        }
        mbar_init(&c.drain, 1);
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b0)) : "memory");
        if (MODE == GATEUP)
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_b1)) : "memory");
    }
    for (int e = threadIdx.x; e <= E; e += THREADS) c.off[e] = p.offsets[e];
    __syncthreads();
    if (threadIdx.x < 32) {
        // exclusive scan of mtiles_e * n_tiles over experts (E <= 256: 8 per lane)
        int local[8], sum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int e = lane * 8 + j;
            int m = 0;
            if (e < E) {
                const int rows = c.off[e + 1] - c.off[e];
                m = (rows + BM - 1) / BM;
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
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&c.tmem_base)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    const uint32_t tmem = c.tmem_base;
    const int total = c.n_tiles_total;
    const int kblocks = p.K / BK;
    volatile int *abort_flag = &c.abort_flag;

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t it = 0;   // global k-block counter across tiles
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            int e, mt, nt;
            decode_tile(c, E, p.n_tiles, tile, e, mt, nt);
            const int arow = c.off[e] + mt * BM;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait(&c.empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                mbar_expect_tx(&c.full[s], A_BYTES + (Q8 ? BQ_BYTES + SC_BYTES : B_BYTES));
                uint8_t *st = smem + s * C::STAGE;
                tma_load_2d(st, &tm_a, &c.full[s], kb * BK, arow);
                // B: 16-bit tiles are 128 B per row, int8 tiles 64 B per row
                constexpr int half_b = (Q8 ? BQ_BYTES : B_BYTES) / 2;
                uint8_t *sc = st + A_BYTES + BQ_BYTES;   // Q8: scales [2 blocks][rows]
                if (MODE == GATEUP) {
                    const int brow = e * p.F + nt * (BN / 2);
                    tma_load_2d(st + A_BYTES, &tm_b0, &c.full[s], kb * BK, brow);
                    tma_load_2d(st + A_BYTES + half_b, &tm_b1, &c.full[s], kb * BK, brow);
                    if (Q8) {
                        tma_load_2d(sc, &tm_s0, &c.full[s], brow, kb * 2);
                        tma_load_2d(sc + SC_BYTES / 2, &tm_s1, &c.full[s], brow, kb * 2);
                    }
                } else {
                    const int brow = e * p.d + nt * BN;
                    tma_load_2d(st + A_BYTES, &tm_b0, &c.full[s], kb * BK, brow);
                    if (Q8) tma_load_2d(sc, &tm_s0, &c.full[s], brow, kb * 2);
                }
            }
        }
        if (!ok) {
            atomicOr(p.status, kDevTimeout);
            c.abort_flag = 1;
            // let loads already issued land before the CTA exits
            for (uint32_t j = (it >= STAGES ? it - STAGES : 0); j < it; ++j) {
                volatile int no_abort = 0;
                mbar_wait(&c.full[j % STAGES], (j / STAGES) & 1u, &no_abort);
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        // fp16 operands on the Q8_0 path (grouped rows and h are fp16), else
        // bf16 -- except a bf16-weight DOWN over an fp16 h, which cannot occur
        const uint32_t idesc_rt = idesc_f16(Q8 ? 1 : 0);
        uint32_t it = 0, local_tile = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++local_tile) {
            const uint32_t acc = local_tile & 1u;
            const uint32_t acc_ph = (local_tile >> 1) & 1u;
            if (!mbar_wait(&c.tempty[acc], acc_ph ^ 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d_tmem = tmem + acc * BN;
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!mbar_wait(&c.full[s], ph, abort_flag)) { ok = false; break; }
                const int cb = it & 1;
                if (Q8 && !mbar_wait(&c.cfull[cb], (it >> 1) & 1u, abort_flag)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + s * C::STAGE);
                const uint32_t b0 = Q8 ? smem_u32(sCvt + cb * B_BYTES) : a0 + A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    umma_f16(d_tmem, sw128_desc(a0 + kk * 32), sw128_desc(b0 + kk * 32), idesc_rt,
                             (kb | kk) != 0);
                }
                umma_commit(&c.empty[s]);     // frees the stage when these MMAs finish
                if (Q8) umma_commit(&c.cempty[cb]);
            }
            if (!ok) break;
            umma_commit(&c.tfull[acc]);       // accumulator ready for the epilogue
        }
        if (!ok) {
            atomicOr(p.status, kDevTimeout);
            c.abort_flag = 1;
            umma_commit(&c.drain);            // wait for MMAs in flight before TMEM is freed
            volatile int no_abort = 0;
            mbar_wait(&c.drain, 0, &no_abort);
        }
    } else if (Q8 && warp >= 6) {
        // ------------------------------------------------ Q8_0 converters (4 warps)
        // lane -> (row in an 8-row pass, 16-byte column chunk of the int8 row);
        // warp w converts rows [64(w-6), 64(w-6)+64) of the 256-row B tile
        const int cw = warp - 6;
        const int rsub = lane >> 2, q = lane & 3;
        uint32_t it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            for (int kb = 0; kb < kblocks; ++kb, ++it) {
                const int s = it % STAGES;
                const int cb = it & 1;
                if (!mbar_wait(&c.full[s], (it / STAGES) & 1u, abort_flag)) { ok = false; break; }
                if (!mbar_wait(&c.cempty[cb], ((it >> 1) & 1u) ^ 1u, abort_flag)) { ok = false; break; }
                const uint8_t *bq = smem + s * C::STAGE + A_BYTES;
                const __half *scl = reinterpret_cast<const __half *>(bq + BQ_BYTES);
                uint8_t *bo = sCvt + cb * B_BYTES;
#pragma unroll
                for (int pass = 0; pass < 8; ++pass) {
                    const int r = cw * 64 + pass * 8 + rsub;
                    // scale of (row r, 32-column block q/2): GATEUP keeps the gate
                    // rows' [2][128] scales, then the up rows'; DOWN [2][256]
                    const int blk = q >> 1;
                    const __half sv = MODE == GATEUP
                        ? scl[(r >> 7) * 256 + blk * 128 + (r & 127)]
                        : scl[blk * 256 + r];
                    const uint4 v = *reinterpret_cast<const uint4 *>(bq + r * 64 + q * 16);
                    uint4 lo, hi;
                    dequant16(v, __half2half2(sv), lo, hi);
                    *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q) ^ (r & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4 *>(bo + r * 128 + (((2 * q + 1) ^ (r & 7)) << 4)) = hi;
                }
                fence_proxy_async_smem();
                mbar_arrive(&c.cfull[cb]);
            }
        }
        if (!ok) {
            if (lane == 0) atomicOr(p.status, kDevTimeout);
            c.abort_flag = 1;
        }
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------ epilogue (4 warps)
        const int quarter = warp & 3;         // TMEM lanes this warp may access
        const int row_in_tile = quarter * 32 + lane;
        uint32_t local_tile = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++local_tile) {
            const uint32_t acc = local_tile & 1u;
            const uint32_t acc_ph = (local_tile >> 1) & 1u;
            // warp-uniform outcome: tcgen05.ld below is warp-collective
            if (!__all_sync(0xffffffffu, mbar_wait(&c.tfull[acc], acc_ph, abort_flag))) {
                if (lane == 0) atomicOr(p.status, kDevTimeout);
                c.abort_flag = 1;
                break;
            }
            tc_fence_after();
            int e, mt, nt;
            decode_tile(c, E, p.n_tiles, tile, e, mt, nt);
            const int rows_e = c.off[e + 1] - c.off[e];
            const bool valid = mt * BM + row_in_tile < rows_e;
            const int grow = c.off[e] + mt * BM + row_in_tile;
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + acc * BN;
            if (MODE == GATEUP) {
                uint16_t *hrow = p.h + (size_t)grow * p.F + nt * (BN / 2);
#pragma unroll 1
                for (int cc = 0; cc < BN / 2; cc += 16) {
                    uint32_t g[16], u[16];
                    tmem_ld16(tbase + cc, g);
                    tmem_ld16(tbase + BN / 2 + cc, u);
                    tmem_ld_wait();
                    uint32_t packed[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float h0 = silu_f(__uint_as_float(g[2 * j])) * __uint_as_float(u[2 * j]);
                        const float h1 = silu_f(__uint_as_float(g[2 * j + 1])) * __uint_as_float(u[2 * j + 1]);
                        if (p.h_fp16) {
                            __half2 v = __floats2half2_rn(h0, h1);
                            packed[j] = *reinterpret_cast<uint32_t *>(&v);
                        } else {
                            __nv_bfloat162 v = __floats2bfloat162_rn(h0, h1);
                            packed[j] = *reinterpret_cast<uint32_t *>(&v);
                        }
                    }
                    if (valid) {
                        uint4 *dst = reinterpret_cast<uint4 *>(hrow + cc);
                        dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
                        dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
                    }
                }
            } else {
                int tok = 0;
                float wgt = 0.f;
                if (valid) { tok = p.perm_tok[grow]; wgt = p.perm_w[grow]; }
                float *orow = p.out + (size_t)tok * p.d + nt * BN;
#pragma unroll 1
                for (int cc = 0; cc < BN; cc += 16) {
                    uint32_t v[16];
                    tmem_ld16(tbase + cc, v);
                    tmem_ld_wait();
                    if (valid) {
#pragma unroll
                        for (int j = 0; j < 16; j += 4) {
                            const float a = wgt * __uint_as_float(v[j]);
                            const float b = wgt * __uint_as_float(v[j + 1]);
                            const float cq = wgt * __uint_as_float(v[j + 2]);
                            const float dq = wgt * __uint_as_float(v[j + 3]);
                            if (p.k == 1)
                                *reinterpret_cast<float4 *>(orow + cc + j) = make_float4(a, b, cq, dq);
                            else
                                red_add_v4(orow + cc + j, a, b, cq, dq);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&c.tempty[acc]);
        }
    }

    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(TMEM_COLS)
                     : "memory");
    }
}

template <bool Q8> constexpr size_t smem_bytes()
{
    return 1024 + Cfg<Q8>::CTL + sizeof(SmemCtl);
}

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
// (the converters read it row by row).
static bool make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols,
                        uint32_t box_rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
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
bool tc_gemm_supports(moe_dtype w_dt) { return w_dt == MOE_BF16 || w_dt == MOE_Q8_0; }

bool tc_gemm_prefer(int T, int d, int E, int k, int F)
{
    (void)d; (void)F;
    // grouped GEMMs pay off once experts hold whole 128-row tiles on average
    return (long long)T * k >= 64LL * E && T >= 512;
}

template <bool Q8>
static cudaError_t set_smem_attrs()
{
    using namespace tc;
    static std::atomic<int> done{0};
    if (done.load()) return cudaSuccess;
    const int smem = (int)smem_bytes<Q8>();
    cudaError_t err;
    if ((err = cudaFuncSetAttribute(grouped_gemm_kernel<GATEUP, Q8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess ||
        (err = cudaFuncSetAttribute(grouped_gemm_kernel<DOWN, Q8>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
        return err;
    done.store(1);
    return cudaSuccess;
}

cudaError_t launch_tc_experts(const TcArgs &a, cudaStream_t stream)
{
    using namespace tc;
    const bool q8 = a.w_dt == MOE_Q8_0;
    if (!q8 && a.w_dt != MOE_BF16) return cudaErrorNotSupported;
    const int rows = a.T * a.k;
    cudaError_t err = cudaSuccess;
    if (!a.xp_ready &&
        (err = launch_gather_rows(a.x, a.d, a.perm_tok, rows, a.xp, q8 ? 1 : 0, a.num_sms, stream)) !=
            cudaSuccess)
        return err;
    if (a.ev_gathered && (err = cudaEventRecord(a.ev_gathered, stream)) != cudaSuccess) return err;

    // activations: bf16, or fp16 on the Q8_0 path
    const CUtensorMapDataType act = q8 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t gu_rows = (uint64_t)a.E * a.F, d_rows = (uint64_t)a.E * a.d;
    CUtensorMap m_xp, m_wg, m_wu, m_h, m_wd;
    bool ok = make_map(&m_xp, a.xp, rows, a.d, BM, act) && make_map(&m_h, a.h, rows, a.F, BM, act);
    if (q8) {
        ok = ok && make_map_u8(&m_wg, a.w_gate, gu_rows, a.d, BN / 2) &&
             make_map_u8(&m_wu, a.w_up, gu_rows, a.d, BN / 2) &&
             make_map_u8(&m_wd, a.w_down, d_rows, a.F, BN);
    } else {
        ok = ok && make_map(&m_wg, a.w_gate, gu_rows, a.d, BN / 2, act) &&
             make_map(&m_wu, a.w_up, gu_rows, a.d, BN / 2, act) &&
             make_map(&m_wd, a.w_down, d_rows, a.F, BN, act);
    }
    if (!ok) return cudaErrorInvalidValue;
    if ((err = q8 ? set_smem_attrs<true>() : set_smem_attrs<false>()) != cudaSuccess) return err;

    // Q8_0 packed buffers: int8 plane, then the fp16 scale plane [cols/32, rows]
    // at align256(rows * cols); maps with box {tile rows, 2 blocks}
    auto scale_map = [](CUtensorMap *m, const void *packed, uint64_t r, uint64_t cols,
                        uint32_t box_rows) {
        auto enc = encode_fn();
        if (!enc) return false;
        const void *base = static_cast<const char *>(packed) + align_up((size_t)(r * cols), 256);
        cuuint64_t dims[2] = {r, cols / 32};
        cuuint64_t strides[1] = {r * 2};
        cuuint32_t box[2] = {box_rows, 2};
        cuuint32_t estr[2] = {1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    CUtensorMap m_sg, m_su, m_sd;
    if (q8 && !(scale_map(&m_sg, a.w_gate, gu_rows, a.d, BN / 2) &&
                scale_map(&m_su, a.w_up, gu_rows, a.d, BN / 2) &&
                scale_map(&m_sd, a.w_down, d_rows, a.F, BN)))
        return cudaErrorInvalidValue;
    Params p{};
    p.offsets = a.offsets; p.E = a.E; p.F = a.F; p.d = a.d; p.k = a.k;
    p.h = static_cast<uint16_t *>(a.h); p.perm_tok = a.perm_tok; p.perm_w = a.perm_w;
    p.out = a.out; p.status = a.status; p.h_fp16 = q8 ? 1 : 0;

    // upper bound on tiles: every expert could own a ragged tile
    const long long max_mtiles = rows / BM + (a.E < rows ? a.E : rows);
    auto grid_for = [&](long long tiles) { return (int)(tiles < a.num_sms ? (tiles < 1 ? 1 : tiles) : a.num_sms); };

    p.K = a.d; p.n_tiles = a.F / (BN / 2);
    if (q8) {
        launch_pdl(grouped_gemm_kernel<GATEUP, true>, dim3(grid_for(max_mtiles * p.n_tiles)),
                   dim3(Cfg<true>::THREADS), smem_bytes<true>(), stream, m_xp, m_wg, m_wu, m_sg,
                   m_su, p);
    } else {
        launch_pdl(grouped_gemm_kernel<GATEUP, false>, dim3(grid_for(max_mtiles * p.n_tiles)),
                   dim3(Cfg<false>::THREADS), smem_bytes<false>(), stream, m_xp, m_wg, m_wu, m_xp,
                   m_xp, p);
    }
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (a.ev_gateup && (err = cudaEventRecord(a.ev_gateup, stream)) != cudaSuccess) return err;

    p.K = a.F; p.n_tiles = a.d / BN;
    if (q8) {
        launch_pdl(grouped_gemm_kernel<DOWN, true>, dim3(grid_for(max_mtiles * p.n_tiles)),
                   dim3(Cfg<true>::THREADS), smem_bytes<true>(), stream, m_h, m_wd, m_wd, m_sd,
                   m_sd, p);
    } else {
        launch_pdl(grouped_gemm_kernel<DOWN, false>, dim3(grid_for(max_mtiles * p.n_tiles)),
                   dim3(Cfg<false>::THREADS), smem_bytes<false>(), stream, m_h, m_wd, m_wd, m_h,
                   m_h, p);
    }
    return cudaGetLastError();
}

}  // namespace moe
