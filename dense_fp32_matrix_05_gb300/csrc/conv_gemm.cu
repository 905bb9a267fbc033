// Instantiations and launcher of the implicit-GEMM convolution form of the
// 3xTF32 kernel: the producers gather B, the im2col matrix of each image,
// straight from the NCHW input (ConvGeom), so it never exists in memory.
// The filter (A) is staged by the host into 16-byte aligned rows in the
// kernel's k order and always goes through its tensor map; the output (C)
// keeps its tensor-map copies when aligned; the images of a batch are the
// kernel's strided batch.
#include <cuda.h>

#include <cstring>

#include "launch.h"
#include "tf32x3_gemm.cuh"
#include "tmap.h"

namespace sg {
namespace {

template <int TM, int ORDER>
cudaError_t launch_conv_tm(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int tma_c, int grid,
                           const CUtensorMap &map_a, const CUtensorMap &map_c, cudaStream_t stream) {
    using C = tf32x3::Cfg<TM, false>;
    auto kern = tf32x3::tf32x3_gemm_kernel<TM, true, false, ORDER>;
    const int smem = C::kSmemBytes + (ORDER == kConvTapsDense ? C::kConvTabBytes : 0);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // no B maps: the kernel does not read them when TMA_B is false
    return launch_pdl(kern, grid, tf32x3::Roles<TM, true, false>::kThreads, smem, stream, g, s, ctl, 1, tma_c, 0u,
                      map_a, map_a, map_c, map_a, map_a, map_a);
}

template <int TM>
cudaError_t launch_conv_rows(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int order, int vec_c,
                             int grid, int batch, cudaStream_t stream) {
    CUtensorMap ma, mc;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(&mc, 0, sizeof(mc));
    if (!make_tmap_a(g, TM, batch, &ma)) return cudaErrorNotSupported;
    const int tc = (vec_c && make_tmap_c(g, batch, &mc)) ? 1 : 0;
    if (map_range_error()) return cudaErrorInvalidValue;  // SGEMM_DEBUG only
    if (order == kConvChannels) return launch_conv_tm<TM, kConvChannels>(g, s, ctl, tc, grid, ma, mc, stream);
    if (order == kConvTapsDense) {
        if (g.K > kConvTabMax) return cudaErrorInvalidValue;
        return launch_conv_tm<TM, kConvTapsDense>(g, s, ctl, tc, grid, ma, mc, stream);
    }
    return launch_conv_tm<TM, kConvTaps>(g, s, ctl, tc, grid, ma, mc, stream);
}

// dst[f][(kh * KW + kw) * C + c] = w[f][c][kh][kw]: OIHW rows to OHWI rows of
// leading dimension ld.  Grid-stride over the destination, which is written
// in order; the filter is small, so its strided reads stay in cache.
__global__ void filter_ohwi_kernel(const float *__restrict__ w, int F, int C, int KHW, float *__restrict__ dst,
                                   long long ld) {
    const long long row = static_cast<long long>(C) * KHW;
    const long long total = static_cast<long long>(F) * row;
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long f = i / row;
        const int r = static_cast<int>(i - f * row);
        const int tap = r / C, c = r - tap * C;
        dst[f * ld + r] = w[(f * C + c) * KHW + tap];
    }
}

// xp = x with zero borders: planes of H x W become (H + 2 ph) x (W + 2 pw),
// the image at (ph, pw).  A warp copies one destination row (lanes along it,
// both sides coalesced), 8 rows per block; a grid-stride loop covers the rest.
// Four independent loads per lane are in flight before the stores.
__global__ void __launch_bounds__(256) pad_planes_kernel(const float *__restrict__ x, long long rows, int H, int W,
                                                         int ph, int pw, float *__restrict__ xp) {
    const int Hp = H + 2 * ph, Wp = W + 2 * pw;
    const int lane = threadIdx.x & 31;
    for (long long row = blockIdx.x * 8LL + (threadIdx.x >> 5); row < rows; row += gridDim.x * 8LL) {
        const long long plane = row / Hp;
        const int y = static_cast<int>(row - plane * Hp) - ph;
        const bool y_in = static_cast<unsigned>(y) < static_cast<unsigned>(H);
        const float *src = x + (plane * H + (y_in ? y : 0)) * W;
        float *dst = xp + row * Wp;
        for (int c0 = lane; c0 < Wp; c0 += 128) {
            float v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int sx = c0 + 32 * u - pw;
                v[u] = (y_in && static_cast<unsigned>(sx) < static_cast<unsigned>(W)) ? __ldg(src + sx) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (c0 + 32 * u < Wp) dst[c0 + 32 * u] = v[u];
        }
    }
}

}  // namespace

cudaError_t pad_planes_launch(const float *x, long long planes, int H, int W, int ph, int pw, float *xp,
                              cudaStream_t stream) {
    const long long rows = planes * (H + 2LL * ph);
    if (rows <= 0) return cudaSuccess;
    const long long blocks = (rows + 7) / 8;
    pad_planes_kernel<<<static_cast<unsigned>(blocks < 8192 ? blocks : 8192), 256, 0, stream>>>(x, rows, H, W, ph,
                                                                                                pw, xp);
    return cudaGetLastError();
}

cudaError_t filter_ohwi_launch(const float *w, int F, int C, int KH, int KW, float *dst, long long ld,
                               cudaStream_t stream) {
    const long long total = static_cast<long long>(F) * C * KH * KW;
    if (total <= 0) return cudaSuccess;
    const long long blocks = (total + 255) / 256;
    filter_ohwi_kernel<<<static_cast<unsigned>(blocks < 4096 ? blocks : 4096), 256, 0, stream>>>(w, F, C, KH * KW,
                                                                                                 dst, ld);
    return cudaGetLastError();
}

cudaError_t tf32x3_conv_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int order,
                               int vec_c, int grid, cudaStream_t stream, int batch) {
    switch (tm) {
        case 16: return launch_conv_rows<16>(g, s, ctl, order, vec_c, grid, batch, stream);
        case 32: return launch_conv_rows<32>(g, s, ctl, order, vec_c, grid, batch, stream);
        case 64: return launch_conv_rows<64>(g, s, ctl, order, vec_c, grid, batch, stream);
        case 128: return launch_conv_rows<128>(g, s, ctl, order, vec_c, grid, batch, stream);
        case 192: return launch_conv_rows<192>(g, s, ctl, order, vec_c, grid, batch, stream);
        case 256: return launch_conv_rows<256>(g, s, ctl, order, vec_c, grid, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
