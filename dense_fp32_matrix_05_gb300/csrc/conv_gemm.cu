// Instantiations and launcher of the implicit-GEMM convolution form of the
// 3xTF32 kernel: the producers gather B, the im2col matrix of each image,
// straight from the NCHW input (ConvGeom), so it never exists in memory.
// The filter (A) and the output (C) keep their tensor-map copies when
// aligned; the images of a batch are the kernel's strided batch.
#include <cuda.h>

#include <cstring>

#include "launch.h"
#include "tf32x3_gemm.cuh"
#include "tmap.h"

namespace sg {
namespace {

template <int TM, bool TA>
cudaError_t launch_conv_tm(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int tma_c,
                           int grid, const CUtensorMap &map_a, const CUtensorMap &map_c, cudaStream_t stream) {
    using C = tf32x3::Cfg<TM, false>;
    auto kern = tf32x3::tf32x3_gemm_kernel<TM, TA, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    // no B map: the kernel does not read it when TMA_B is false
    kern<<<grid, tf32x3::Roles<TM, TA, false>::kThreads, C::kSmemBytes, stream>>>(g, s, ctl, vec_a, tma_c, map_a,
                                                                                    map_a, map_c);
    return cudaGetLastError();
}

template <int TM>
cudaError_t launch_conv_rows(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int vec_c,
                             int grid, int batch, cudaStream_t stream) {
    CUtensorMap ma, mc;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(&mc, 0, sizeof(mc));
    const bool ta = vec_a && make_tmap_a(g, TM, batch, &ma);
    const int tc = (vec_c && make_tmap_c(g, batch, &mc)) ? 1 : 0;
    if (ta) return launch_conv_tm<TM, true>(g, s, ctl, vec_a, tc, grid, ma, mc, stream);
    return launch_conv_tm<TM, false>(g, s, ctl, vec_a, tc, grid, ma, mc, stream);
}

}  // namespace

cudaError_t tf32x3_conv_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a,
                               int vec_c, int grid, cudaStream_t stream, int batch) {
    switch (tm) {
        case 16: return launch_conv_rows<16>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 32: return launch_conv_rows<32>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 64: return launch_conv_rows<64>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 128: return launch_conv_rows<128>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 192: return launch_conv_rows<192>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 256: return launch_conv_rows<256>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
