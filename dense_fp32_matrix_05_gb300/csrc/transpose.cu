// Out-of-place transpose of a row-major fp32 matrix, the staging step of
// transposed operands (BLAS transa / transb): dst[c][r] = src[r][c].
//
// 32 x 32 tiles through shared memory padded to 33 columns, so that the
// column reads of a tile hit 32 different banks.  A warp reads 32
// consecutive floats of a source row and writes 32 consecutive floats of a
// destination row, so both sides of the copy are coalesced; the kernel is
// bound by HBM.  Grid-stride over tiles in both directions, any size, and
// over the matrices of a strided batch.
#include "launch.h"

namespace sg {
namespace {

constexpr int kTile = 32;
constexpr int kRowsPerPass = 8;  // block: 32 x 8 threads

__global__ void __launch_bounds__(kTile * kRowsPerPass) transpose_kernel(const float *__restrict__ src0, long long lds,
                                                                         int rows, int cols, float *__restrict__ dst0,
                                                                         long long ldd, int count, long long ss,
                                                                         long long ds) {
    __shared__ float tile[kTile][kTile + 1];
    const int tx = threadIdx.x, ty = threadIdx.y;
    for (int z = blockIdx.z; z < count; z += gridDim.z) {
        const float *src = src0 + static_cast<long long>(z) * ss;
        float *dst = dst0 + static_cast<long long>(z) * ds;
        for (int r0 = blockIdx.y * kTile; r0 < rows; r0 += gridDim.y * kTile) {
            for (int c0 = blockIdx.x * kTile; c0 < cols; c0 += gridDim.x * kTile) {
#pragma unroll
                for (int i = 0; i < kTile; i += kRowsPerPass) {
                    const int r = r0 + ty + i, c = c0 + tx;
                    if (r < rows && c < cols) tile[ty + i][tx] = src[static_cast<long long>(r) * lds + c];
                }
                __syncthreads();
#pragma unroll
                for (int i = 0; i < kTile; i += kRowsPerPass) {
                    const int c = c0 + ty + i, r = r0 + tx;  // destination row c, column r
                    if (c < cols && r < rows) dst[static_cast<long long>(c) * ldd + r] = tile[tx][ty + i];
                }
                __syncthreads();
            }
        }
    }
}

}  // namespace

cudaError_t transpose_launch(const float *src, long long lds, int rows, int cols, float *dst, long long ldd,
                             cudaStream_t stream, int count, long long src_stride, long long dst_stride) {
    if (rows <= 0 || cols <= 0 || count <= 0) return cudaSuccess;
    const long long gx = (cols + kTile - 1) / kTile, gy = (rows + kTile - 1) / kTile;
    const dim3 grid(static_cast<unsigned>(gx < 4096 ? gx : 4096), static_cast<unsigned>(gy < 4096 ? gy : 4096),
                    static_cast<unsigned>(count < 1024 ? count : 1024));
    transpose_kernel<<<grid, dim3(kTile, kRowsPerPass), 0, stream>>>(src, lds, rows, cols, dst, ldd, count,
                                                                     src_stride, dst_stride);
    return cudaGetLastError();
}

}  // namespace sg
