// q8.cu -- repack Q8_0 expert weights into planes the kernels can stream.
//
// Q8_0 (ggml's 8-bit block format, used for the ZONOS2 experts:
// "zonos2.cpp internals", §Quantization): each block of 32 consecutive values
// along the contiguous axis is 34 bytes, an fp16 scale then 32 int8 values;
// value = scale * q.  34-byte blocks are not 16-byte aligned, so the library
// repacks once, at load time, into an int8 plane [rows, cols] and an fp16 scale
// plane [cols/32, rows] (same bytes, aligned for 128-bit and TMA loads; the
// scales of one 32-column block are contiguous over rows, so a weight tile's
// scales are one TMA box).
#include "common.cuh"
#include "kernels.h"

namespace moe {

__global__ void pack_q8_0_kernel(const uint8_t *__restrict__ blocks, long long nblocks,
                                 long long rows, int bpr, int8_t *__restrict__ q,
                                 __half *__restrict__ scales)
{
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
         b += (long long)gridDim.x * blockDim.x) {
        const uint8_t *src = blocks + b * 34;
        uint16_t s = (uint16_t)src[0] | ((uint16_t)src[1] << 8);
        const long long row = b / bpr, blk = b - row * bpr;   // block blk of row `row`
        scales[blk * rows + row] = __ushort_as_half(s);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = (uint32_t)src[2 + 4 * i] | ((uint32_t)src[3 + 4 * i] << 8) |
                   ((uint32_t)src[4 + 4 * i] << 16) | ((uint32_t)src[5 + 4 * i] << 24);
        uint4 *dst = reinterpret_cast<uint4 *>(q + b * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

cudaError_t launch_pack_q8_0(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream)
{
    const long long nblocks = rows * (cols / 32);
    if (nblocks == 0) return cudaSuccess;
    int8_t *q = static_cast<int8_t *>(packed);
    __half *s = reinterpret_cast<__half *>(static_cast<char *>(packed) +
                                           align_up((size_t)rows * cols, 256));
    long long grid = (nblocks + 255) / 256;
    if (grid > 65535LL * 16) grid = 65535LL * 16;
    pack_q8_0_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks),
                                                          nblocks, rows, cols / 32, q, s);
    return cudaGetLastError();
}

// Affine 4-bit, groups of 64 (the experts of the MLX build, "Zyphra-ZONOS2-4bit",
// §How this was quantized): 36-byte blocks {fp16 scale, fp16 bias, 32 bytes of
// codes, value 2j in the low nibble of byte j} -> tiles of 128 rows x one group
// (q4_tile_offset): the rows' codes (each 4 bytes regrouped so that the even
// values fill the low 16 bits and the odd ones the high 16 bits, q4_nibble),
// their scales, their biases.  One thread per (tile, row); rows past the last
// one are written as zeros.
__global__ void pack_q4_a64_kernel(const uint8_t *__restrict__ blocks, long long rows, int groups,
                                   long long n, uint8_t *__restrict__ packed)
{
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
         t += (long long)gridDim.x * blockDim.x) {
        const long long tile = t / kQ4TileRows;
        const int rr = (int)(t - tile * kQ4TileRows);
        const long long rt = tile / groups;
        const int g = (int)(tile - rt * groups);
        const long long row = rt * kQ4TileRows + rr;
        uint8_t *dst = packed + (size_t)tile * kQ4TileBytes;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint16_t sc = 0, bi = 0;
        if (row < rows) {
            const uint8_t *src = blocks + ((size_t)row * groups + g) * 36;
            sc = (uint16_t)src[0] | ((uint16_t)src[1] << 8);
            bi = (uint16_t)src[2] | ((uint16_t)src[3] << 8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                uint32_t lo = 0, hi = 0;   // even values (low nibbles), odd values (high nibbles)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    lo |= (uint32_t)(src[4 + 4 * i + b] & 15u) << (4 * b);
                    hi |= (uint32_t)(src[4 + 4 * i + b] >> 4) << (4 * b);
                }
                w[i] = lo | (hi << 16);
            }
        }
        uint4 *c = reinterpret_cast<uint4 *>(dst + rr * 32);
        c[0] = make_uint4(w[0], w[1], w[2], w[3]);
        c[1] = make_uint4(w[4], w[5], w[6], w[7]);
        reinterpret_cast<uint16_t *>(dst + kQ4ScaleOff)[rr] = sc;
        reinterpret_cast<uint16_t *>(dst + kQ4BiasOff)[rr] = bi;
    }
}

// Q4_K super-blocks ("zonos2.cpp internals", §Recommended: F16 spine + K-quant
// experts; the GGUF layout: fp16 d, fp16 dmin, 12 bytes of six-bit sub-block
// scales and mins, 128 bytes of codes, sub-block j = values 32j .. 32j+31
// decoding as d * sc[j] * q - dmin * m[j]) -> tiles of 128 rows x 64 columns
// with two affine groups per row: group g of tile column block kb is
// sub-block j = 2 (kb % 4) + g of super-block kb / 4, scale = d * sc[j] and
// bias = 8 d sc[j] - dmin m[j] (the value at code 8: value = scale * (q - 8)
// + bias), each rounded to fp16.  One thread per (tile, row).
__global__ void pack_q4_k_kernel(const uint8_t *__restrict__ blocks, long long rows, int groups,
                                 long long n, uint8_t *__restrict__ packed)
{
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
         t += (long long)gridDim.x * blockDim.x) {
        const long long tile = t / kQ4TileRows;
        const int rr = (int)(t - tile * kQ4TileRows);
        const long long rt = tile / groups;
        const int kb = (int)(tile - rt * groups);
        const long long row = rt * kQ4TileRows + rr;
        uint8_t *dst = packed + (size_t)tile * kQ4KTileBytes;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        uint16_t sc16[2] = {0, 0}, bi16[2] = {0, 0};
        if (row < rows) {
            const uint8_t *blk = blocks + ((size_t)row * (groups / 4) + kb / 4) * 144;
            const float d = __half2float(__ushort_as_half((uint16_t)(blk[0] | (blk[1] << 8))));
            const float dmin = __half2float(__ushort_as_half((uint16_t)(blk[2] | (blk[3] << 8))));
            const uint8_t *s = blk + 4;
            const uint8_t *run = blk + 16 + 32 * (kb % 4);   // sub-block 2c low, 2c+1 high nibbles
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                const int j = 2 * (kb % 4) + g;
                int sc, m;
                if (j < 4) {
                    sc = s[j] & 63;
                    m = s[j + 4] & 63;
                } else {
                    sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
                    m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
                }
                // both products exact in fp32 (11-bit d or dmin times a 6-bit integer)
                const float s32 = d * (float)sc, mb = dmin * (float)m;
                sc16[g] = __half_as_ushort(__float2half_rn(s32));
                bi16[g] = __half_as_ushort(__float2half_rn(8.0f * s32 - mb));   // the value at code 8

            }
            // value v of the 64: v < 32 the low nibble of run[v], else the high nibble of run[v - 32]
#pragma unroll
            for (int i = 0; i < 8; ++i) {   // word i: values 8i .. 8i+7
                uint32_t word = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int v = 8 * i + e;
                    const uint32_t q = v < 32 ? (run[v] & 15u) : (run[v - 32] >> 4);
                    word |= q << (4 * q4_nibble(e));
                }
                w[i] = word;
            }
        }
        uint4 *c = reinterpret_cast<uint4 *>(dst + rr * 32);
        c[0] = make_uint4(w[0], w[1], w[2], w[3]);
        c[1] = make_uint4(w[4], w[5], w[6], w[7]);
        uint16_t *scp = reinterpret_cast<uint16_t *>(dst + kQ4ScaleOff);
        uint16_t *bip = reinterpret_cast<uint16_t *>(dst + q4_bias_off(2));
        scp[rr] = sc16[0]; scp[kQ4TileRows + rr] = sc16[1];
        bip[rr] = bi16[0]; bip[kQ4TileRows + rr] = bi16[1];
    }
}

size_t q4_k_packed_bytes(long long rows, int cols)
{
    const long long tiles_r = (rows + kQ4TileRows - 1) / kQ4TileRows;
    return (size_t)tiles_r * (size_t)(cols / 64) * kQ4KTileBytes;
}

cudaError_t launch_pack_q4_k(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream)
{
    const int groups = cols / 64;
    const long long n = (rows + kQ4TileRows - 1) / kQ4TileRows * groups * kQ4TileRows;
    if (n == 0) return cudaSuccess;
    long long grid = (n + 255) / 256;
    if (grid > 65535LL * 16) grid = 65535LL * 16;
    pack_q4_k_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), rows,
                                                         groups, n, static_cast<uint8_t *>(packed));
    return cudaGetLastError();
}

// Q6_K super-blocks ("zonos2.cpp internals", §Recommended: F16 spine + K-quant
// experts; the GGUF layout: ql[128] low 4 bits, qh[64] top 2 bits, int8
// scales[16], fp16 d; value v = d * scales[v / 16] * (q - 32)) -> the 8-bit
// planes with one scale per 16 values: int8 q - 32 and fp16(d * scales[j]).
// One thread per (row, 16-value group).
__global__ void pack_q6_k_kernel(const uint8_t *__restrict__ blocks, long long n, int groups_per_row,
                                 long long rows, int8_t *__restrict__ q, __half *__restrict__ scales)
{
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
         t += (long long)gridDim.x * blockDim.x) {
        const long long row = t / groups_per_row;
        const int j = (int)(t - row * groups_per_row);   // 16-value group of the row
        const uint8_t *blk = blocks + ((size_t)row * (groups_per_row / 16) + j / 16) * 210;
        const float d = __half2float(__ushort_as_half((uint16_t)(blk[208] | (blk[209] << 8))));
        const int jb = j % 16;                          // group within the super-block
        scales[(size_t)j * rows + row] = __float2half_rn(d * (float)(int8_t)blk[192 + jb]);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int v = 16 * jb + i, h = v / 128, g = (v % 128) / 32, l = v % 32;
            const uint8_t lo_byte = blk[64 * h + l + 32 * (g % 2)];
            const int lo = g < 2 ? (lo_byte & 15) : (lo_byte >> 4);
            const int hi = (blk[128 + 32 * h + l] >> (2 * g)) & 3;
            const uint32_t code = (uint32_t)(uint8_t)(int8_t)((lo | (hi << 4)) - 32);
            w[i / 4] |= code << (8 * (i % 4));
        }
        *reinterpret_cast<uint4 *>(q + (size_t)t * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_pack_q6_k(const void *blocks, long long rows, int cols, void *packed,
                             cudaStream_t stream)
{
    const long long n = rows * (cols / 16);
    if (n == 0) return cudaSuccess;
    int8_t *q = static_cast<int8_t *>(packed);
    __half *s = reinterpret_cast<__half *>(static_cast<char *>(packed) + align_up((size_t)rows * cols, 256));
    long long grid = (n + 255) / 256;
    if (grid > 65535LL * 16) grid = 65535LL * 16;
    pack_q6_k_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), n,
                                                         cols / 16, rows, q, s);
    return cudaGetLastError();
}

// fp8 rows {fp32 scale, E4M3 codes[cols]} (4 + cols bytes each, any
// alignment) -> the E4M3 plane [rows, cols] and the fp32 row scales at
// align256(rows * cols).  One thread per byte of the plane; the first byte's
// thread of each row also moves its scale.
__global__ void pack_fp8_kernel(const uint8_t *__restrict__ src, long long n, int cols,
                                uint8_t *__restrict__ q, float *__restrict__ scales)
{
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < n;
         t += (long long)gridDim.x * blockDim.x) {
        const long long row = t / cols;
        const int c = (int)(t - row * cols);
        const uint8_t *r = src + (size_t)row * (size_t)(cols + 4);
        q[t] = r[4 + c];
        if (c == 0)
            scales[row] = __uint_as_float((uint32_t)r[0] | ((uint32_t)r[1] << 8) | ((uint32_t)r[2] << 16) |
                                          ((uint32_t)r[3] << 24));
    }
}

cudaError_t launch_pack_fp8(const void *rows_in, long long rows, int cols, void *packed, cudaStream_t stream)
{
    const long long n = rows * cols;
    if (n == 0) return cudaSuccess;
    uint8_t *q = static_cast<uint8_t *>(packed);
    float *s = reinterpret_cast<float *>(static_cast<char *>(packed) + align_up((size_t)rows * cols, 256));
    long long grid = (n + 255) / 256;
    if (grid > 65535LL * 16) grid = 65535LL * 16;
    pack_fp8_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint8_t *>(rows_in), n, cols, q, s);
    return cudaGetLastError();
}

size_t q4_a64_packed_bytes(long long rows, int cols)
{
    const long long tiles_r = (rows + kQ4TileRows - 1) / kQ4TileRows;
    return (size_t)tiles_r * (size_t)(cols / 64) * kQ4TileBytes;
}

cudaError_t launch_pack_q4_a64(const void *blocks, long long rows, int cols, void *packed,
                               cudaStream_t stream)
{
    const int groups = cols / 64;
    const long long n = (rows + kQ4TileRows - 1) / kQ4TileRows * groups * kQ4TileRows;
    if (n == 0) return cudaSuccess;
    long long grid = (n + 255) / 256;
    if (grid > 65535LL * 16) grid = 65535LL * 16;
    pack_q4_a64_kernel<<<(unsigned)grid, 256, 0, stream>>>(static_cast<const uint8_t *>(blocks), rows,
                                                           groups, n, static_cast<uint8_t *>(packed));
    return cudaGetLastError();
}

}  // namespace moe
