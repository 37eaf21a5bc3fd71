// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;

// Device status word values (first word of the workspace).
constexpr uint32_t kDevOk = 0;
constexpr uint32_t kDevTimeout = 1u;       // bounded mbarrier wait gave up
constexpr uint32_t kDevCheckFailed = 2u;   // device consistency check failed

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- conversions
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Eight consecutive elements -> fp32, for each storage type.
struct Chunk8 { float v[8]; };

__device__ __forceinline__ void load8(const float *p, Chunk8 &c)
{
    float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    c.v[0] = a.x; c.v[1] = a.y; c.v[2] = a.z; c.v[3] = a.w;
    c.v[4] = b.x; c.v[5] = b.y; c.v[6] = b.z; c.v[7] = b.w;
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, Chunk8 &c)
{
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    c.v[0] = bf16lo(u.x); c.v[1] = bf16hi(u.x);
    c.v[2] = bf16lo(u.y); c.v[3] = bf16hi(u.y);
    c.v[4] = bf16lo(u.z); c.v[5] = bf16hi(u.z);
    c.v[6] = bf16lo(u.w); c.v[7] = bf16hi(u.w);
}

// Streaming (read-once) weight loads: do not keep the lines in L1.
__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ld_stream_u2(const void *p)
{
    uint2 r;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];"
                 : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

// Raw weight chunk of 8 elements as loaded from HBM (converted later).
template <typename WT> struct RawW;
template <> struct RawW<float> { uint4 a, b; };
template <> struct RawW<__nv_bfloat16> { uint4 a; };
struct Q8Tag {};   // Q8_0 planes: int8 q plane + fp16 scale per 32 values
template <> struct RawW<Q8Tag> { uint2 q; float s; };
struct Q4Tag {};   // affine 4-bit planes: codes + fp16 scale and bias per 64 values
struct F8Tag {};   // fp8 planes: E4M3 codes + fp32 scale per row
template <> struct RawW<F8Tag> { uint2 q; float s; };
template <> struct RawW<Q4Tag> { uint32_t q; float s, b, z; };

// Weight matrix view: row-major [rows, cols] in one of the storage types.
template <typename WT> struct WView {
    const WT *p;
    size_t cols;
    __device__ __forceinline__ void load(size_t row, int col, RawW<WT> &r) const;
    __device__ __forceinline__ static void cvt(const RawW<WT> &r, Chunk8 &c);
};

template <> __device__ __forceinline__ void WView<float>::load(size_t row, int col, RawW<float> &r) const
{
    const float *q = p + row * cols + col;
    r.a = ld_stream_u4(q);
    r.b = ld_stream_u4(q + 4);
}
template <> __device__ __forceinline__ void WView<float>::cvt(const RawW<float> &r, Chunk8 &c)
{
    c.v[0] = __uint_as_float(r.a.x); c.v[1] = __uint_as_float(r.a.y);
    c.v[2] = __uint_as_float(r.a.z); c.v[3] = __uint_as_float(r.a.w);
    c.v[4] = __uint_as_float(r.b.x); c.v[5] = __uint_as_float(r.b.y);
    c.v[6] = __uint_as_float(r.b.z); c.v[7] = __uint_as_float(r.b.w);
}
template <> __device__ __forceinline__ void WView<__nv_bfloat16>::load(size_t row, int col,
                                                                        RawW<__nv_bfloat16> &r) const
{
    r.a = ld_stream_u4(p + row * cols + col);
}
template <> __device__ __forceinline__ void WView<__nv_bfloat16>::cvt(const RawW<__nv_bfloat16> &r,
                                                                       Chunk8 &c)
{
    c.v[0] = bf16lo(r.a.x); c.v[1] = bf16hi(r.a.x);
    c.v[2] = bf16lo(r.a.y); c.v[3] = bf16hi(r.a.y);
    c.v[4] = bf16lo(r.a.z); c.v[5] = bf16hi(r.a.z);
    c.v[6] = bf16lo(r.a.w); c.v[7] = bf16hi(r.a.w);
}

// 8-bit planes view (Q8_0, Q6_K): p points at the q plane; the fp16 scale
// plane [cols/group, rows] follows at align256(rows*cols) bytes.  `scales`,
// `rows` and `group` (32 or 16 values per scale) are set by the host.
template <> struct WView<Q8Tag> {
    const int8_t *q;
    const __half *scales;
    size_t cols;
    size_t rows;
    int group;
    __device__ __forceinline__ void load(size_t row, int col, RawW<Q8Tag> &r) const
    {
        r.q = ld_stream_u2(q + row * cols + col);
        r.s = __half2float(scales[(size_t)(col / group) * rows + row]);
    }
    __device__ __forceinline__ static void cvt(const RawW<Q8Tag> &r, Chunk8 &c)
    {
        const uint32_t w[2] = {r.q.x, r.q.y};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            int v = (int)(int8_t)((w[i >> 2] >> (8 * (i & 3))) & 0xff);
            c.v[i] = (float)v * r.s;
        }
    }
};

// Affine 4-bit view: q points at the code plane [rows, cols/2] (value 2j in the
// low nibble of byte j); fp16 scale and bias planes [cols/64, rows].  Set by
// the host.
// Packed 4-bit weights are tiles of 128 rows x 64 columns in row-tile-major
// order: tile (rt, kb) at ((rt * groups) + kb) * tile bytes, groups = cols / 64.
// Inside: the 128 rows' 32 code bytes, then gpr x 128 fp16 scales, then gpr x
// 128 fp16 biases ([group][row]), where a row's 64 values form gpr affine
// groups (value = scale * q + bias): one for the affine 4-bit format
// (moe_pack_q4_a64, 4608-byte tiles), two of 32 for Q4_K (moe_pack_q4_k,
// 5120-byte tiles).  A k-block of one row tile is one contiguous copy.  Each
// 32-bit word of a row's codes holds 8 consecutive values, the even ones in
// nibbles 0-3 and the odd ones in nibbles 4-7 (value i in nibble
// q4_nibble(i)), so that one mask of the word yields two neighbouring values,
// one per 16-bit half.
// the 4-bit storage types (packed tiles) and their affine groups per tile row
__host__ __device__ __forceinline__ constexpr bool is_q4(int w_dt) { return w_dt == MOE_Q4_A64 || w_dt == MOE_Q4_K; }
// the 8-bit planes (int8 plane + fp16 scale plane [cols / group, rows]): Q8_0
// with a scale per 32 values, Q6_K repacked with one per 16
__host__ __device__ __forceinline__ constexpr bool is_q8p(int w_dt) { return w_dt == MOE_Q8_0 || w_dt == MOE_Q6_K; }
__host__ __device__ __forceinline__ constexpr int q8_group(int w_dt) { return w_dt == MOE_Q6_K ? 16 : 32; }
// fp8 (E4M3) planes: code plane [rows, cols], then one fp32 scale per row at
// align256(rows * cols)
__host__ __device__ __forceinline__ constexpr bool is_fp8(int w_dt) { return w_dt == MOE_FP8; }
// converted weights (fp16 operands on the tensor cores): 4-bit tiles, 8-bit planes
__host__ __device__ __forceinline__ constexpr bool is_conv(int w_dt) { return is_q4(w_dt) || is_q8p(w_dt) || is_fp8(w_dt); }

// two E4M3 codes (low byte: the first) -> fp16x2 (low half: the first), exact
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two)
{
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(two));
    return out;
}

// fp8 view: q points at the E4M3 plane [rows, cols]; `scales` (fp32 [rows])
// follow at align256(rows * cols).  Set by the host.
template <> struct WView<F8Tag> {
    const uint8_t *q;
    const float *scales;
    size_t cols;
    __device__ __forceinline__ void load(size_t row, int col, RawW<F8Tag> &r) const
    {
        r.q = ld_stream_u2(q + row * cols + col);
        r.s = scales[row];
    }
    __device__ __forceinline__ static void cvt(const RawW<F8Tag> &r, Chunk8 &c)
    {
        const uint32_t w[2] = {r.q.x, r.q.y};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)(w[i >> 1] >> (16 * (i & 1))));
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h2));
            c.v[2 * i] = f.x * r.s;
            c.v[2 * i + 1] = f.y * r.s;
        }
    }
};
__host__ __device__ __forceinline__ constexpr int q4_gpr(int w_dt) { return w_dt == MOE_Q4_K ? 2 : 1; }
constexpr int kQ4TileRows = 128, kQ4ScaleOff = 4096;
constexpr int kQ4TileBytes = 4608, kQ4BiasOff = 4352;   // one group per row (affine 4-bit)
constexpr int kQ4KTileBytes = 5120;                     // two groups per row (Q4_K)
__host__ __device__ __forceinline__ constexpr int q4_tile_bytes(int gpr) { return 4096 + 512 * gpr; }
__host__ __device__ __forceinline__ constexpr int q4_bias_off(int gpr) { return 4096 + 256 * gpr; }
__host__ __device__ __forceinline__ constexpr int q4_nibble(int i) { return (i >> 1) + 4 * (i & 1); }
// The code a tile's bias belongs to: value = scale * (q - z) + bias.  z = 0
// for the affine 4-bit tiles (the format's own zero point); z = 8 for the
// Q4_K tiles, whose bias is the value at code 8, the middle of the group's
// range: its fp16 rounding error is then small, and |q - 8| <= 8 halves the
// weight of the scale's rounding error (both roundings are systematic over a
// group).
__host__ __device__ __forceinline__ constexpr int q4_zero_code(int gpr) { return gpr == 2 ? 8 : 0; }
__host__ __device__ __forceinline__ size_t q4_tile_offset(long long row, int g, int groups, int gpr = 1)
{
    return ((size_t)(row / kQ4TileRows) * (size_t)groups + (size_t)g) * (size_t)q4_tile_bytes(gpr);
}

// One 32-bit word of packed codes (8 consecutive values, q4_nibble order) ->
// 8 fp16 values scale * (q - z) + bias in K order.  Masked under the fp16
// exponent of 1024 (ulp 1), nibbles 0 and 4 give the pair (1024 + q_0, 1024 +
// q_1) and nibbles 1 and 5, left in bits 4-7 of each half, (1024 + 16 q_2,
// 1024 + 16 q_3); the word shifted by 8 gives values 4-7 the same way.  One
// exact fma by (1, 1) or (1/16, 1/16) and the matching offset (Q4Fix) leaves
// q - z, a second one gives scale * (q - z) + bias with a single rounding.
struct Q4Fix {
    __half2 lo, hi;   // -(1024 + z) and -(64 + z), in both halves
    __device__ __forceinline__ explicit Q4Fix(int z)
        : lo(__float2half2_rn(-1024.0f - (float)z)), hi(__float2half2_rn(-64.0f - (float)z)) {}
};
__device__ __forceinline__ uint32_t q4_pair_fp16(uint32_t t, __half2 mul, __half2 add, __half2 sc2, __half2 bi2)
{
    t |= 0x64006400u;
    const __half2 v = __hfma2(__hfma2(*reinterpret_cast<const __half2 *>(&t), mul, add), sc2, bi2);
    return *reinterpret_cast<const uint32_t *>(&v);
}
__device__ __forceinline__ uint4 q4_word_fp16x8(uint32_t w, __half2 sc2, __half2 bi2, Q4Fix fx)
{
    const __half2 one2 = __float2half2_rn(1.0f), sixteenth2 = __float2half2_rn(0.0625f);
    const uint32_t w8 = w >> 8;
    return make_uint4(q4_pair_fp16(w & 0x000F000Fu, one2, fx.lo, sc2, bi2),
                      q4_pair_fp16(w & 0x00F000F0u, sixteenth2, fx.hi, sc2, bi2),
                      q4_pair_fp16(w8 & 0x000F000Fu, one2, fx.lo, sc2, bi2),
                      q4_pair_fp16(w8 & 0x00F000F0u, sixteenth2, fx.hi, sc2, bi2));
}

// int8 x 16 (one uint4) -> fp16 x 16 scaled by s: (q ^ 0x80) placed in the
// mantissa of 1024.0 gives 1024 + 128 + q exactly; subtracting 1152 leaves q,
// and the product with s is the one rounding.  Output in value order (lo:
// values 0-7, hi: 8-15, two per 32-bit word).
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

template <> struct WView<Q4Tag> {
    const uint8_t *q;     // packed tiles
    int groups;           // cols / 64
    int gpr;              // affine groups per row of a tile: 1 (affine 4-bit) or 2 (Q4_K)
    __device__ __forceinline__ void load(size_t row, int col, RawW<Q4Tag> &r) const
    {
        const uint8_t *t = q + q4_tile_offset((long long)row, col / 64, groups, gpr);
        const int rr = (int)(row % kQ4TileRows);
        const int g = gpr == 2 ? (col % 64) / 32 : 0;
        uint32_t v;
        asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];"
                     : "=r"(v) : "l"(t + rr * 32 + (col % 64) / 2));
        r.q = v;
        r.s = __half2float(reinterpret_cast<const __half *>(t + kQ4ScaleOff)[g * kQ4TileRows + rr]);
        r.b = __half2float(reinterpret_cast<const __half *>(t + q4_bias_off(gpr))[g * kQ4TileRows + rr]);
        r.z = (float)q4_zero_code(gpr);
    }
    __device__ __forceinline__ static void cvt(const RawW<Q4Tag> &r, Chunk8 &c)
    {
#pragma unroll
        for (int i = 0; i < 8; ++i) c.v[i] = fmaf(r.s, (float)((r.q >> (4 * q4_nibble(i))) & 15u) - r.z, r.b);
    }
};

// fp16 rows of the Q8_0 tensor-core path: each bf16 row is scaled by a power
// of two, 2^-e, so that its largest magnitude is at most 1 (e = 0 for an
// all-zero or non-finite row).  The scaling is exact, so fp16 keeps the
// bf16 values' digits while no row can leave fp16's range; the epilogues undo
// it exactly.  e is the exponent of the row maximum (warp-collective: every
// lane gets the same e).
__device__ __forceinline__ int fp16_row_exponent(const uint16_t *row, int d, int lane)
{
    float m = 0.f;
    constexpr int U = 8;   // loads in flight per lane
    for (int c0 = lane; c0 < d / 8; c0 += 32 * U) {
        uint4 u[U];
#pragma unroll
        for (int q = 0; q < U; ++q)
            u[q] = c0 + 32 * q < d / 8 ? __ldg(reinterpret_cast<const uint4 *>(row) + c0 + 32 * q)
                                       : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int q = 0; q < U; ++q) {
            const uint32_t w[4] = {u[q].x, u[q].y, u[q].z, u[q].w};
#pragma unroll
            for (int r = 0; r < 4; ++r) m = fmaxf(m, fmaxf(fabsf(bf16lo(w[r])), fabsf(bf16hi(w[r]))));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (!(m > 0.f) || !isfinite(m)) return 0;
    int e;
    frexpf(m, &e);   // m = f * 2^e, f in [0.5, 1): m <= 2^e
    return e;
}
// Eight bf16 values (one uint4) times 2^-e, as fp16.
__device__ __forceinline__ uint4 bf16x8_to_fp16_scaled(uint4 u, int e)
{
    const float sc = ldexpf(1.f, -e);
    uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        __half2 hh = __floats2half2_rn(bf16lo(w[q]) * sc, bf16hi(w[q]) * sc);
        w[q] = *reinterpret_cast<uint32_t *>(&hh);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Programmatic dependent launch.  Every kernel of the library is launched so
// that it may start while its predecessor in the stream finishes; it calls
// pdl_wait() before touching global memory (this waits for the predecessor to
// complete and its writes to be visible) and pdl_trigger() right after, which
// lets the next kernel of the stream start launching in turn.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter() { pdl_wait(); pdl_trigger(); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// launch_pdl for a kernel that runs in clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t stream, int cluster, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Record a device-detected error in the status word (calls without a status
// word -- moe_route, moe_route_scored -- have none to report to).
__device__ __forceinline__ void flag_status(uint32_t *status, uint32_t bits)
{
    if (status) atomicOr(status, bits);
}

// Debug builds (MOE_DEBUG=1, libmoe_gb300_debug.so) check the grouped-row
// offsets every expert kernel is given before it uses them -- offsets[0] = 0,
// non-decreasing, offsets[E] = the number of grouped rows -- and the token
// indices the row gathers read; a kernel given inconsistent offsets does no
// work and records kDevCheckFailed, and a token index out of range is recorded
// and its row skipped.  Release builds compile the checks away.
#ifndef MOE_DEBUG
#define MOE_DEBUG 0
#endif
// CTA-collective (every thread calls it): the offsets as above.
__device__ __forceinline__ bool debug_offsets_ok(const int32_t *off, int E, int rows, uint32_t *status)
{
#if MOE_DEBUG
    bool bad = false;
    for (int e = threadIdx.x; e < E; e += blockDim.x) bad |= off[e] > off[e + 1];
    if (threadIdx.x == 0) bad |= off[0] != 0 || off[E] != rows;
    bad = __syncthreads_or(bad) != 0;
    if (bad && threadIdx.x == 0) flag_status(status, kDevCheckFailed);
    return !bad;
#else
    (void)off; (void)E; (void)rows; (void)status;
    return true;
#endif
}
// A token index v in [0, n) (debug builds; release: always true).
__device__ __forceinline__ bool debug_index_ok(int v, int n, uint32_t *status)
{
#if MOE_DEBUG
    if (v >= 0 && v < n) return true;
    flag_status(status, kDevCheckFailed);
    return false;
#else
    (void)v; (void)n; (void)status;
    return true;
#endif
}

// True (uniformly across the CTA) when an earlier kernel of this call has
// already recorded an error in the status word: the caller then returns
// without touching scratch whose contents may be incomplete.
__device__ __forceinline__ bool upstream_failed(const uint32_t *status)
{
    __shared__ int failed;
    if (threadIdx.x == 0) failed = status ? (int)*(volatile const uint32_t *)status : 0;
    __syncthreads();
    return failed != 0;
}

// ------------------------------------------------------ host: per-device state
// Index of the current device (0 when the query fails; the launch that
// follows then reports the error).
inline int current_device()
{
    int dev = 0;
    return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 ? dev : 0;
}
// Streaming multiprocessors of the current device (read per call, so grids
// follow the part the process runs on; a failed query gives 1 and the launch
// reports the error).
inline int device_sm_count()
{
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, current_device()) !=
            cudaSuccess || n < 1)
        return 1;
    return n;
}
// Set-up that every device needs once (kernel attributes, occupancy
// queries), remembered per device: devices 0-63 are cached, any further
// device repeats the set-up on each call.
constexpr int kCachedDevices = 64;
struct PerDeviceFlag {
    std::atomic<uint64_t> bits{0};
    bool done(int dev) const { return dev < kCachedDevices && ((bits.load() >> dev) & 1u); }
    void mark(int dev) { if (dev < kCachedDevices) bits.fetch_or(uint64_t(1) << dev); }
};
struct PerDeviceInt {   // -1 = not cached yet
    std::atomic<int> v[kCachedDevices];
    PerDeviceInt() { for (auto &x : v) x.store(-1); }
    int get(int dev) const { return dev < kCachedDevices ? v[dev].load() : -1; }
    void put(int dev, int value) { if (dev < kCachedDevices) v[dev].store(value); }
};

// -------------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Reduce 8 per-lane values across the warp so that afterwards every lane
// holds the full sum of value index r = ((lane>>4)&1)*4 + ((lane>>3)&1)*2 + ((lane>>2)&1).
// Uses 9 shuffles instead of 8 x 5.
__device__ __forceinline__ float warp_transpose_sum8(float (&v)[8], int lane)
{
    // stage offset 16: keep half, send half
    {
        const bool hi = lane & 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float send = hi ? v[i] : v[i + 4];
            float keep = hi ? v[i + 4] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
    }
    {
        const bool hi = lane & 8;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            float send = hi ? v[i] : v[i + 2];
            float keep = hi ? v[i + 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
    }
    {
        const bool hi = lane & 4;
        float send = hi ? v[0] : v[1];
        float keep = hi ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    float s = v[0];
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    return s;
}

__device__ __forceinline__ int transpose8_row(int lane)
{
    return ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
}

}  // namespace moe
