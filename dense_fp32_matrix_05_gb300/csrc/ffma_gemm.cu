// Instantiations and launcher of the FFMA kernel and the C = beta*C kernel.
#include "ffma_gemm.cuh"
#include "launch.h"

namespace sg {

static_assert(kFfmaBK == ffma::kBK, "planner constants");

namespace {
constexpr int kFfmaStages = 4;

template <int BM, int BN>
cudaError_t launch_tile(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int vec_b,
                        int vec_c, cudaStream_t stream) {
    using C = ffma::Cfg<BM, BN, kFfmaStages>;
    auto kern = ffma::ffma_gemm_kernel<BM, BN, kFfmaStages>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<s.units, ffma::kThreads, C::kSmemBytes, stream>>>(g, s, ctl, vec_a, vec_b, vec_c);
    return cudaGetLastError();
}
}  // namespace

bool ffma_supported_tile(int bm, int bn) {
    return (bm == 128 && bn == 128) || (bm == 64 && bn == 256) || (bm == 32 && bn == 512) ||
           (bm == ffma::kBigBM && bn == ffma::kBigBN);
}

int ffma_stages(int bm, int bn) { return (bm == ffma::kBigBM && bn == ffma::kBigBN) ? ffma::kBigStages : kFfmaStages; }

int ffma_smem_bytes(int bm, int bn) {
    if (!ffma_supported_tile(bm, bn)) return -1;
    if (bm == ffma::kBigBM && bn == ffma::kBigBN) return ffma::BigCfg::kSmemBytes;
    return (bm + bn) * ffma::kBK * 4 * kFfmaStages + 16;
}

cudaError_t ffma_launch(int bm, int bn, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a,
                        int vec_b, int vec_c, cudaStream_t stream) {
    if (bm == ffma::kBigBM && bn == ffma::kBigBN) {
        // one CTA per SM; A goes through 4-byte copies whatever its alignment
        (void)vec_a;
        cudaError_t e = cudaFuncSetAttribute(ffma::ffma_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             ffma::BigCfg::kSmemBytes);
        if (e != cudaSuccess) return e;
        ffma::ffma_big_kernel<<<s.units, ffma::kThreads, ffma::BigCfg::kSmemBytes, stream>>>(g, s, ctl, vec_b, vec_c);
        return cudaGetLastError();
    }
    if (bm == 128 && bn == 128) return launch_tile<128, 128>(g, s, ctl, vec_a, vec_b, vec_c, stream);
    if (bm == 64 && bn == 256) return launch_tile<64, 256>(g, s, ctl, vec_a, vec_b, vec_c, stream);
    if (bm == 32 && bn == 512) return launch_tile<32, 512>(g, s, ctl, vec_a, vec_b, vec_c, stream);
    return cudaErrorInvalidValue;
}

cudaError_t scale_c_preload() {
    cudaFuncAttributes attr;
    return cudaFuncGetAttributes(&attr, ffma::scale_c_kernel);
}

cudaError_t scale_c_launch(float *C, long long ldc, int M, int N, float beta, int num_sms,
                           cudaStream_t stream) {
    const long long total = static_cast<long long>(M) * N;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(num_sms > 0 ? num_sms : 1) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    ffma::scale_c_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(C, ldc, M, N, beta);
    return cudaGetLastError();
}

}  // namespace sg
