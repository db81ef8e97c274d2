// Load-time layout kernels of libpi (not on the timed path).
//
// The offline hot/cold placement of the PowerInfer pages (blog.csdn.net
// QbitAI/IPADS article, "CPU/GPU混合推理设计": neurons are profiled offline and
// placed by how often they fire) becomes, on one device, a permutation of the
// neurons: physical neuron i is original neuron perm[i], hot neurons first.
// These kernels apply it while converting to the layouts the step kernel
// streams: one contiguous row per neuron for W_up / W_gate / W_down^T, and for
// Q4_0 rows a 16-byte-aligned run of fp16 scales followed by the nibbles.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pi_kernels.h"

namespace pi {

// dst row i = src row perm[i]; rowBytes is a multiple of 16.
__global__ void permute_rows_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                    const int32_t *__restrict__ perm, int rows, size_t row16, size_t dst16)
{
    for (int i = blockIdx.x; i < rows; i += gridDim.x) {
        const int o = perm ? perm[i] : i;
        const uint4 *s = src + (size_t)o * row16;
        uint4 *d = dst + (size_t)i * dst16;
        for (size_t k = threadIdx.x; k < row16; k += blockDim.x) d[k] = s[k];
    }
}

// dst [n][d] (row i = physical neuron i) from src [d][nsrc] (column o =
// original neuron o): dst[i][j] = src[j][perm[i]] (n = nsrc, or fewer rows
// for a shard of the neurons).  32x32 tiles through shared memory.
__global__ void transpose_permute16_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                           const int32_t *__restrict__ perm, int d, int n, int nsrc)
{
    __shared__ uint16_t tile[32][33];
    const int i0 = blockIdx.x * 32, j0 = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y; // 32 x 8
    for (int yy = ty; yy < 32; yy += 8) {
        const int i = i0 + tx, j = j0 + yy;
        if (i < n && j < d) {
            const int o = perm ? perm[i] : i;
            tile[yy][tx] = src[(size_t)j * nsrc + o];
        }
    }
    __syncthreads();
    for (int yy = ty; yy < 32; yy += 8) {
        const int i = i0 + yy, j = j0 + tx;
        if (i < n && j < d) dst[(size_t)i * d + j] = tile[tx][yy];
    }
}

// Q4_0 rows of 18-byte blocks -> [scales (d/32 fp16, padded to scB bytes)]
// [nibbles (d/32 x 16 bytes)], rows permuted.  One thread per block.
__global__ void q4_split_kernel(const uint8_t *__restrict__ src, uint8_t *__restrict__ dst,
                                const int32_t *__restrict__ perm, int n, int nb, int scB, size_t rowB)
{
    const size_t total = (size_t)n * nb;
    for (size_t k = (size_t)blockIdx.x * blockDim.x + threadIdx.x; k < total; k += (size_t)gridDim.x * blockDim.x) {
        const int i = (int)(k / nb), b = (int)(k % nb);
        const int o = perm ? perm[i] : i;
        const uint8_t *s = src + ((size_t)o * nb + b) * 18;
        uint8_t *row = dst + (size_t)i * rowB;
        row[2 * b] = s[0];
        row[2 * b + 1] = s[1];
        uint8_t *q = row + scB + (size_t)b * 16;
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = s[2 + j];
        if (b == nb - 1) // zero the padding after the last scale
            for (int z = 2 * nb; z < scB; ++z) row[z] = 0;
    }
}

__global__ void permute16_kernel(const uint16_t *__restrict__ src, uint16_t *__restrict__ dst,
                                 const int32_t *__restrict__ perm, int n)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        dst[i] = src[perm ? perm[i] : i];
}

cudaError_t launch_permute_rows(const void *src, void *dst, const int32_t *perm, int rows, size_t rowBytes,
                                cudaStream_t s, size_t dstStride)
{
    if (rows <= 0) return cudaSuccess;
    const int grid = rows < 65535 ? rows : 65535;
    permute_rows_kernel<<<grid, 256, 0, s>>>((const uint4 *)src, (uint4 *)dst, perm, rows, rowBytes / 16,
                                             (dstStride ? dstStride : rowBytes) / 16);
    return cudaGetLastError();
}

// Bias tails: up row i (stride upB) gets b[i] at byte rowB, zeros after it,
// so a predicted neuron's bias travels with its W_up row.
__global__ void bias_tail_kernel(const uint16_t *__restrict__ b, uint8_t *__restrict__ up, int n, size_t rowB,
                                 size_t upB)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        uint4 *t = reinterpret_cast<uint4 *>(up + (size_t)i * upB + rowB);
        *t = make_uint4((uint32_t)b[i], 0u, 0u, 0u);
    }
}

cudaError_t launch_bias_tail(const uint16_t *b, uint8_t *up, int n, size_t rowB, size_t upB, cudaStream_t s)
{
    const int grid = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    bias_tail_kernel<<<grid, 256, 0, s>>>(b, up, n, rowB, upB);
    return cudaGetLastError();
}

cudaError_t launch_transpose_permute16(const uint16_t *src, uint16_t *dst, const int32_t *perm, int d, int n,
                                       int nsrc, cudaStream_t s)
{
    dim3 grid((n + 31) / 32, (d + 31) / 32), block(32, 8);
    transpose_permute16_kernel<<<grid, block, 0, s>>>(src, dst, perm, d, n, nsrc);
    return cudaGetLastError();
}

cudaError_t launch_q4_split(const uint8_t *src, uint8_t *dst, const int32_t *perm, int n, int d, int scB,
                            cudaStream_t s, size_t dstStride)
{
    const int nb = d / 32;
    const size_t total = (size_t)n * nb;
    const int grid = (int)((total + 255) / 256 < 65535 ? (total + 255) / 256 : 65535);
    const size_t rowB = (size_t)scB + (size_t)nb * 16;
    q4_split_kernel<<<grid, 256, 0, s>>>(src, dst, perm, n, nb, scB, dstStride ? dstStride : rowB);
    return cudaGetLastError();
}

// x[i] += u[i], i < n (fp32): a layer's update, reduced over the shards of a
// neuron-sharded layer, added into the residual stream
__global__ void residual_add_kernel(float *__restrict__ x, const float *__restrict__ u, size_t n)
{
    const size_t n4 = n / 4;
    float4 *x4 = reinterpret_cast<float4 *>(x);
    const float4 *u4 = reinterpret_cast<const float4 *>(u);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (size_t)gridDim.x * blockDim.x) {
        float4 a = x4[i];
        const float4 b = u4[i];
        a.x += b.x, a.y += b.y, a.z += b.z, a.w += b.w;
        x4[i] = a;
    }
    for (size_t i = 4 * n4 + (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
        x[i] += u[i];
}

cudaError_t launch_residual_add(float *x, const float *u, size_t n, cudaStream_t s)
{
    const size_t blocks = (n / 4 + 255) / 256;
    residual_add_kernel<<<(unsigned)(blocks < 1 ? 1 : (blocks > 1024 ? 1024 : blocks)), 256, 0, s>>>(x, u, n);
    return cudaGetLastError();
}

cudaError_t launch_permute16(const uint16_t *src, uint16_t *dst, const int32_t *perm, int n, cudaStream_t s)
{
    const int grid = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    permute16_kernel<<<grid, 256, 0, s>>>(src, dst, perm, n);
    return cudaGetLastError();
}

} // namespace pi
