// kernels_transpose.cu -- the image transpose behind the column-order directional
// scans: a scan that visits a rows x cols image (stored in raster order) column by
// column (Mamba SSM complete guide (youngju.dev), section 9, VMamba's four
// directions) is the raster scan of the transposed image. The directional entry
// point with a workspace transposes u, delta, z, B and C into it, runs the
// prefill's own scan, and transposes y back.
//
// One CTA moves a square tile of one image through shared memory (rows read and
// written along the contiguous dimension, the padded tile column avoiding bank
// conflicts); images are the leading index (batch x channels, or batch x states).
#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace ssm {
namespace {

constexpr int kRowsPerPass = 8;   // blockDim.y (blockDim.x = 32)

// A kTile x kTile tile per CTA and image: 64 for 2-byte elements (a warp's row is
// then 128 bytes; a 56 x 56 image is one tile), 32 for 4-byte ones.
template <typename T, int kTile>
__global__ void __launch_bounds__(32 * kRowsPerPass)
    transpose_images_kernel(const T* __restrict__ src, T* __restrict__ dst, int64_t images, int rows, int cols) {
    constexpr int kPerLane = kTile / 32;   // columns (then rows) per lane
    __shared__ T tile[kTile][kTile + 1];
    const int c0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile;
    for (int64_t img = blockIdx.z; img < images; img += gridDim.z) {
        const T* s = src + img * (int64_t)rows * cols;
        T* d = dst + img * (int64_t)rows * cols;
        // read rows r0 .. r0+kTile-1 of columns c0 .. c0+kTile-1, a warp along a row
        for (int i = threadIdx.y; i < kTile; i += kRowsPerPass) {
            const int r = r0 + i;
#pragma unroll
            for (int e = 0; e < kPerLane; e++) {
                const int cl = threadIdx.x + 32 * e, c = c0 + cl;
                if (r < rows && c < cols) tile[i][cl] = s[(int64_t)r * cols + c];
            }
        }
        __syncthreads();
        // write them as rows c0 .. of the transposed image (length rows), a warp along a row
        for (int i = threadIdx.y; i < kTile; i += kRowsPerPass) {
            const int c = c0 + i;
#pragma unroll
            for (int e = 0; e < kPerLane; e++) {
                const int rl = threadIdx.x + 32 * e, r = r0 + rl;
                if (c < cols && r < rows) d[(int64_t)c * rows + r] = tile[rl][i];
            }
        }
        __syncthreads();
    }
}

template <typename T, int kTile>
cudaError_t launch_tiles(const void* src, void* dst, int64_t images, int64_t rows, int64_t cols, cudaStream_t s) {
    const int64_t gx = (cols + kTile - 1) / kTile, gy = (rows + kTile - 1) / kTile;
    if (gx > INT32_MAX || gy > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)(images < 65535 ? images : 65535));
    transpose_images_kernel<T, kTile><<<grid, dim3(32, kRowsPerPass), 0, s>>>(
        static_cast<const T*>(src), static_cast<T*>(dst), images, (int)rows, (int)cols);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_transpose_images(const void* src, void* dst, int64_t images, int64_t rows, int64_t cols,
                                    int esize, cudaStream_t s) {
    if (images <= 0 || rows <= 0 || cols <= 0) return cudaSuccess;
    if (rows > INT32_MAX || cols > INT32_MAX) return cudaErrorInvalidValue;
    if (esize == 2) return launch_tiles<uint16_t, 64>(src, dst, images, rows, cols, s);
    if (esize == 4) return launch_tiles<uint32_t, 32>(src, dst, images, rows, cols, s);
    return cudaErrorInvalidValue;
}

}  // namespace ssm
