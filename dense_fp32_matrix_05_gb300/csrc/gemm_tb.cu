// Instantiations and launcher of the 3xTF32 kernel for a transposed B
// (BLAS transb: B stored N x K, k innermost).  TMA copies each 16 k x 128 n
// slab of B^T with the 64-byte swizzle; the producers read a column's 16 k
// values as four 16-byte chunks instead of a strided walk, and the rest of
// the kernel is the row-major one.  A must be 16-byte aligned too (its tile
// also comes by TMA; the element-load form spills at this register budget).
// A transposed A still goes through the transpose pass of the API.
#include <cuda.h>

#include <cstring>

#include "launch.h"
#include "tf32x3_gemm.cuh"
#include "tmap.h"

namespace sg {
namespace {

template <int TM>
cudaError_t launch_tb_tm(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int tma_c, int grid,
                         const CUtensorMap &map_a, const CUtensorMap &map_b, const CUtensorMap &map_c,
                         cudaStream_t stream) {
    using C = tf32x3::Cfg<TM, true>;
    auto kern = tf32x3::tf32x3_gemm_kernel<TM, true, true, kConvNone, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    // the residue-class maps are unused by the transposed-B form
    return launch_pdl(kern, grid, tf32x3::Roles<TM, true, true>::kThreads, C::kSmemBytes, stream, g, s, ctl, 1, tma_c,
                      0u, map_a, map_b, map_c, map_b, map_b, map_b);
}

template <int TM>
cudaError_t launch_tb_rows(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int vec_c,
                           int grid, int batch, cudaStream_t stream) {
    CUtensorMap ma, mb, mc;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(&mb, 0, sizeof(mb));
    std::memset(&mc, 0, sizeof(mc));
    if (!vec_a || !make_tmap_a(g, TM, batch, &ma) || !make_tmap_bt(g, batch, &mb)) return cudaErrorNotSupported;
    const int tc = (vec_c && make_tmap_c(g, batch, &mc)) ? 1 : 0;
    if (map_range_error()) return cudaErrorInvalidValue;  // SGEMM_DEBUG only
    return launch_tb_tm<TM>(g, s, ctl, tc, grid, ma, mb, mc, stream);
}

}  // namespace

cudaError_t tf32x3_launch_tb(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a,
                             int vec_c, int grid, cudaStream_t stream, int batch) {
    switch (tm) {
        case 16: return launch_tb_rows<16>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 32: return launch_tb_rows<32>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 64: return launch_tb_rows<64>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 128: return launch_tb_rows<128>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 192: return launch_tb_rows<192>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        case 256: return launch_tb_rows<256>(g, s, ctl, vec_a, vec_c, grid, batch, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
