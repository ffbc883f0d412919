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

// Up to three tensors of the same image shape, transposed together: a CTA moves
// the same kTile x kTile tile of one image of every tensor, so each CTA has
// kNT tiles of loads in flight before its barrier. kTile = 64 for 2-byte
// elements (a warp's row is then 128 bytes; a 56 x 56 image is one tile), 32 for
// 4-byte ones.
template <typename T>
struct TransposeSet {
    const T* src[3];
    T* dst[3];
};

template <typename T, int kTile, int kNT>
__global__ void __launch_bounds__(32 * kRowsPerPass)
    transpose_images_kernel(const TransposeSet<T> set, int64_t images, int rows, int cols) {
    constexpr int kPerLane = kTile / 32;   // columns (then rows) per lane
    __shared__ T tile[kNT][kTile][kTile + 1];
    const int c0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile;
    for (int64_t img = blockIdx.z; img < images; img += gridDim.z) {
        const int64_t base = img * (int64_t)rows * cols;
        // read rows r0 .. r0+kTile-1 of columns c0 .. c0+kTile-1, a warp along a row
#pragma unroll
        for (int t = 0; t < kNT; t++) {
            const T* s = set.src[t] + base;
            for (int i = threadIdx.y; i < kTile; i += kRowsPerPass) {
                const int r = r0 + i;
#pragma unroll
                for (int e = 0; e < kPerLane; e++) {
                    const int cl = threadIdx.x + 32 * e, c = c0 + cl;
                    if (r < rows && c < cols) tile[t][i][cl] = s[(int64_t)r * cols + c];
                }
            }
        }
        __syncthreads();
        // write them as rows c0 .. of the transposed image (length rows), a warp along a row
#pragma unroll
        for (int t = 0; t < kNT; t++) {
            T* d = set.dst[t] + base;
            for (int i = threadIdx.y; i < kTile; i += kRowsPerPass) {
                const int c = c0 + i;
#pragma unroll
                for (int e = 0; e < kPerLane; e++) {
                    const int rl = threadIdx.x + 32 * e, r = r0 + rl;
                    if (c < cols && r < rows) d[(int64_t)c * rows + r] = tile[t][rl][i];
                }
            }
        }
        __syncthreads();
    }
}

template <typename T, int kTile, int kNT>
cudaError_t launch_tiles(const TransposeSet<T>& set, int64_t images, int64_t rows, int64_t cols, cudaStream_t s) {
    const int64_t gx = (cols + kTile - 1) / kTile, gy = (rows + kTile - 1) / kTile;
    if (gx > INT32_MAX || gy > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)gx, (unsigned)gy, (unsigned)(images < 65535 ? images : 65535));
    transpose_images_kernel<T, kTile, kNT><<<grid, dim3(32, kRowsPerPass), 0, s>>>(set, images, (int)rows,
                                                                                   (int)cols);
    return cudaGetLastError();
}

template <typename T, int kTile>
cudaError_t launch_set(const void* const* src, void* const* dst, int n, int64_t images, int64_t rows, int64_t cols,
                       cudaStream_t s) {
    TransposeSet<T> set;
    for (int t = 0; t < 3; t++) {
        set.src[t] = t < n ? static_cast<const T*>(src[t]) : nullptr;
        set.dst[t] = t < n ? static_cast<T*>(dst[t]) : nullptr;
    }
    if (n == 1) return launch_tiles<T, kTile, 1>(set, images, rows, cols, s);
    if (n == 2) return launch_tiles<T, kTile, 2>(set, images, rows, cols, s);
    return launch_tiles<T, kTile, 3>(set, images, rows, cols, s);
}

}  // namespace

cudaError_t launch_transpose_images(const void* const* src, void* const* dst, int n, int64_t images, int64_t rows,
                                    int64_t cols, int esize, cudaStream_t s) {
    if (n < 1 || n > 3) return cudaErrorInvalidValue;
    if (images <= 0 || rows <= 0 || cols <= 0) return cudaSuccess;
    if (rows > INT32_MAX || cols > INT32_MAX) return cudaErrorInvalidValue;
    if (esize == 2) return launch_set<uint16_t, 64>(src, dst, n, images, rows, cols, s);
    if (esize == 4) return launch_set<uint32_t, 32>(src, dst, n, images, rows, cols, s);
    return cudaErrorInvalidValue;
}

}  // namespace ssm
