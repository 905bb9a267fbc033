// Instantiations and launcher of the 3xTF32 tensor-core kernel.
#include "launch.h"
#include "tf32x3_gemm.cuh"

namespace sg {

static_assert(kTf32x3TileN == tf32x3::kTileN && kTf32x3BK == tf32x3::kBK, "planner constants");

namespace {
template <int TM>
cudaError_t launch_tm(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int grid,
                      cudaStream_t stream) {
    using C = tf32x3::Cfg<TM>;
    auto kern = tf32x3::tf32x3_gemm_kernel<TM>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, tf32x3::kThreads, C::kSmemBytes, stream>>>(g, s, ctl, vec_a);
    return cudaGetLastError();
}
}  // namespace

bool tf32x3_supported_tm(int tm) {
    return tm == 16 || tm == 32 || tm == 64 || tm == 128 || tm == 192 || tm == 256;
}

int tf32x3_stages(int tm) { return tf32x3::stages_for(tm); }

int tf32x3_smem_bytes(int tm) {
    switch (tm) {
        case 16: return tf32x3::Cfg<16>::kSmemBytes;
        case 32: return tf32x3::Cfg<32>::kSmemBytes;
        case 64: return tf32x3::Cfg<64>::kSmemBytes;
        case 128: return tf32x3::Cfg<128>::kSmemBytes;
        case 192: return tf32x3::Cfg<192>::kSmemBytes;
        case 256: return tf32x3::Cfg<256>::kSmemBytes;
        default: return -1;
    }
}

cudaError_t tf32x3_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a,
                          int grid, cudaStream_t stream) {
    switch (tm) {
        case 16: return launch_tm<16>(g, s, ctl, vec_a, grid, stream);
        case 32: return launch_tm<32>(g, s, ctl, vec_a, grid, stream);
        case 64: return launch_tm<64>(g, s, ctl, vec_a, grid, stream);
        case 128: return launch_tm<128>(g, s, ctl, vec_a, grid, stream);
        case 192: return launch_tm<192>(g, s, ctl, vec_a, grid, stream);
        case 256: return launch_tm<256>(g, s, ctl, vec_a, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
