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
// §How this was quantized):
// 36-byte blocks {fp16 scale, fp16 bias, 32 bytes of codes, value 2j in the low
// nibble of byte j} -> a code plane [rows, cols/2] (the blocks' code bytes in
// order) and fp16 scale and bias planes [cols/64, rows].
__global__ void pack_q4_a64_kernel(const uint8_t *__restrict__ blocks, long long nblocks,
                                   long long rows, int bpr, uint8_t *__restrict__ codes,
                                   __half *__restrict__ scales, __half *__restrict__ biases)
{
    for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < nblocks;
         b += (long long)gridDim.x * blockDim.x) {
        const uint8_t *src = blocks + b * 36;
        const long long row = b / bpr, blk = b - row * bpr;   // block blk of row `row`
        scales[blk * rows + row] = __ushort_as_half((uint16_t)src[0] | ((uint16_t)src[1] << 8));
        biases[blk * rows + row] = __ushort_as_half((uint16_t)src[2] | ((uint16_t)src[3] << 8));
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = (uint32_t)src[4 + 4 * i] | ((uint32_t)src[5 + 4 * i] << 8) |
                   ((uint32_t)src[6 + 4 * i] << 16) | ((uint32_t)src[7 + 4 * i] << 24);
        uint4 *dst = reinterpret_cast<uint4 *>(codes + b * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
}

size_t q4_a64_scale_offset(long long rows, int cols) { return align_up((size_t)rows * cols / 2, 256); }
size_t q4_a64_bias_offset(long long rows, int cols)
{
    return align_up(q4_a64_scale_offset(rows, cols) + (size_t)rows * (cols / 64) * 2, 256);
}

cudaError_t launch_pack_q4_a64(const void *blocks, long long rows, int cols, void *packed,
                               cudaStream_t stream)
{
    const long long nblocks = rows * (cols / 64);
    if (nblocks == 0) return cudaSuccess;
    char *base = static_cast<char *>(packed);
    long long grid = (nblocks + 255) / 256;
    if (grid > 65535LL * 16) grid = 65535LL * 16;
    pack_q4_a64_kernel<<<(unsigned)grid, 256, 0, stream>>>(
        static_cast<const uint8_t *>(blocks), nblocks, rows, cols / 64,
        reinterpret_cast<uint8_t *>(base),
        reinterpret_cast<__half *>(base + q4_a64_scale_offset(rows, cols)),
        reinterpret_cast<__half *>(base + q4_a64_bias_offset(rows, cols)));
    return cudaGetLastError();
}

}  // namespace moe
