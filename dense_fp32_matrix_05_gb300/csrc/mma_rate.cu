// Peak-rate probes, the roofline denominators of the two paths.
//
// sgemm_tf32_mma_rate: throughput of the tensor cores on the MMA form the
// 3xTF32 kernel issues (tcgen05.mma, kind::tf32, M = 128, A from tensor
// memory, B from shared memory, one fp32 accumulator), measured on this
// GPU.  It is the roofline denominator of the 3xTF32 path: the nominal
// tf32 rate is quoted for another clock and part, so the peak is measured
// the way the kernel uses it.
//
// One CTA per SM.  One thread issues `iters` MMAs of size 128 x n x 8 back
// to back into one accumulator (zero operands: the tensor pipe's speed does
// not depend on the values).  A tcgen05.commit then signals an mbarrier,
// and the thread waits for it with a bounded wait.  The launch is timed with
// CUDA events.
//
// sgemm_ffma_rate: throughput of the CUDA cores' fp32 FMA, the peak of the
// FFMA path.  Every thread of 4 x 512 threads per SM runs 16 independent
// chains of FMAs (as scalar fma.rn.f32, or as 8 chains of packed
// fma.rn.f32x2, the form the FFMA kernels issue), enough independent work
// to cover the FMA latency on every scheduler.  The launch is timed with
// CUDA events; the chains' sum is kept live by a store that never happens.
#include <cuda_runtime.h>

#include "common.cuh"
#include "sgemm_gb300.h"

namespace {

constexpr int kProbeThreads = 128;
constexpr int kProbeMaxN = 256;
constexpr int kProbeBBytes = kProbeMaxN * 64;  // B tile: n rows of 16 fp32 (K-major, 64-byte swizzle)
constexpr int kProbeSmem = 1024 + kProbeBBytes + 64;
constexpr uint32_t kProbeTmemCols = 512;
constexpr uint32_t kProbeACol = 256;           // A operand: tensor-memory columns [256, 272)
constexpr long long kProbeWaitBudget = 20000000000LL;

__device__ int g_probe_status;

__global__ void __launch_bounds__(kProbeThreads, 1) tf32_mma_rate_kernel(int n, int iters) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = sg::smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_base);
    const uint32_t bar = base + kProbeBBytes;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + kProbeBBytes + 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5;

    for (int i = threadIdx.x; i < kProbeBBytes / 4; i += kProbeThreads)
        reinterpret_cast<float *>(base_ptr)[i] = 0.f;
    if (threadIdx.x == 0) {
        sg::mbar_init(bar, 1);
        *abort_flag = 0;
        sg::fence_mbar_init();
    }
    if (warp == 0) {
        sg::tmem_alloc(sg::smem_u32(tmem_slot), kProbeTmemCols);
        sg::tmem_relinquish();
    }
    sg::tc_fence_before();
    __syncthreads();
    sg::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // zero A operand: each warp its 32 lanes of columns [256, 272)
    {
        uint32_t z[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) z[j] = 0u;
        sg::tmem_st32x16(tmem_base + (static_cast<uint32_t>(warp * 32) << 16) + kProbeACol, z);
        sg::tmem_st_wait();
    }
    sg::fence_proxy_async_smem();
    sg::tc_fence_before();
    __syncthreads();
    sg::tc_fence_after();

    if (threadIdx.x == 0) {
        const uint32_t idesc = sg::umma_idesc_tf32(128, n);
        const uint64_t b0 = sg::umma_desc_kmajor_sw64(base);
        const uint64_t b1 = sg::umma_desc_kmajor_sw64(base + 32);
#pragma unroll 1
        for (int i = 0; i < iters; ++i) {
            const uint32_t a = tmem_base + kProbeACol + static_cast<uint32_t>((i & 1) * 8);
            sg::mma_tf32_ts(tmem_base, a, (i & 1) ? b1 : b0, idesc, i > 0 ? 1u : 0u);
        }
        sg::mma_commit(bar);
        sg::DeviceCtl ctl{};
        ctl.status = &g_probe_status;
        ctl.wait_budget = kProbeWaitBudget;
        sg::mbar_wait_bounded(bar, 0u, abort_flag, ctl, sg::kStatusTimeoutMma);
    }
    sg::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        sg::tc_fence_after();
        sg::tmem_dealloc(tmem_base, kProbeTmemCols);
    }
}

constexpr int kFfmaProbeThreads = 512;
constexpr int kFfmaProbeBlocksPerSm = 4;
constexpr int kFfmaProbeChains = 16;  // fp32 FMAs in flight per thread per step

template <bool PACKED>
__global__ void __launch_bounds__(kFfmaProbeThreads) ffma_rate_kernel(float a, float b, int iters, float *sink) {
    float sum = 0.f;
    if constexpr (PACKED) {
        uint64_t x[kFfmaProbeChains / 2];
        const uint64_t a2 = sg::pair_bcast(a), b2 = sg::pair_bcast(b);
#pragma unroll
        for (int j = 0; j < kFfmaProbeChains / 2; ++j) x[j] = sg::pair_bcast(static_cast<float>(threadIdx.x + j));
#pragma unroll 1
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int j = 0; j < kFfmaProbeChains / 2; ++j)  // x = x * a + b, both lanes
                asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[j]) : "l"(a2), "l"(b2));
        }
#pragma unroll
        for (int j = 0; j < kFfmaProbeChains / 2; ++j) {
            float lo, hi;
            sg::pair_split(x[j], lo, hi);
            sum += lo + hi;
        }
    } else {
        float x[kFfmaProbeChains];
#pragma unroll
        for (int j = 0; j < kFfmaProbeChains; ++j) x[j] = static_cast<float>(threadIdx.x + j);
#pragma unroll 1
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int j = 0; j < kFfmaProbeChains; ++j) x[j] = fmaf(x[j], a, b);
        }
#pragma unroll
        for (int j = 0; j < kFfmaProbeChains; ++j) sum += x[j];
    }
    if (sum == -1.0f) *sink = sum;  // never true for the inputs used: keeps the chains live
}

__device__ float g_ffma_probe_sink;

int from_cuda(cudaError_t e) { return e == cudaSuccess ? 0 : static_cast<int>(e); }

}  // namespace

extern "C" int sgemm_tf32_mma_rate(int n, int iters, sgemm_stream_t stream, double *tflops) {
    if (n < 16 || n > kProbeMaxN || n % 16 != 0) return -1;
    if (iters < 1) return -2;
    if (tflops == nullptr) return -4;
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return SGEMM_ERR_NO_DEVICE;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return from_cuda(e);
    if (!(major == 10 && minor == 3)) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const int zero = 0;
    if ((e = cudaMemcpyToSymbol(g_probe_status, &zero, sizeof(int))) != cudaSuccess) return from_cuda(e);
    if ((e = cudaFuncSetAttribute(tf32_mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kProbeSmem)) != cudaSuccess)
        return from_cuda(e);
    cudaEvent_t e0, e1;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess) return from_cuda(e);
    if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
        cudaEventDestroy(e0);
        return from_cuda(e);
    }
    float ms = 0.f;
    tf32_mma_rate_kernel<<<sms, kProbeThreads, kProbeSmem, st>>>(n, iters);  // warm-up
    cudaEventRecord(e0, st);
    tf32_mma_rate_kernel<<<sms, kProbeThreads, kProbeSmem, st>>>(n, iters);
    cudaEventRecord(e1, st);
    e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return from_cuda(e);
    int status = 0;
    if ((e = cudaMemcpyFromSymbol(&status, g_probe_status, sizeof(int))) != cudaSuccess) return from_cuda(e);
    if (status != 0) return SGEMM_ERR_DEVICE_TIMEOUT;
    const double flop = static_cast<double>(sms) * iters * 2.0 * 128.0 * n * 8.0;
    *tflops = ms > 0.f ? flop / (ms * 1e-3) / 1e12 : 0.0;
    return 0;
}

extern "C" int sgemm_ffma_rate(int packed, int iters, sgemm_stream_t stream, double *tflops) {
    if (packed != 0 && packed != 1) return -1;
    if (iters < 1) return -2;
    if (tflops == nullptr) return -4;
    int dev = 0, major = 0, minor = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return SGEMM_ERR_NO_DEVICE;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return from_cuda(e);
    if (!(major == 10 && minor == 3)) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    float *sink = nullptr;
    if ((e = cudaGetSymbolAddress(reinterpret_cast<void **>(&sink), g_ffma_probe_sink)) != cudaSuccess)
        return from_cuda(e);
    auto kern = packed ? ffma_rate_kernel<true> : ffma_rate_kernel<false>;
    const int grid = sms * kFfmaProbeBlocksPerSm;
    cudaEvent_t e0, e1;
    if ((e = cudaEventCreate(&e0)) != cudaSuccess) return from_cuda(e);
    if ((e = cudaEventCreate(&e1)) != cudaSuccess) {
        cudaEventDestroy(e0);
        return from_cuda(e);
    }
    float ms = 0.f;
    // x -> 0.9999 x + 0.5 stays finite and normal (it tends to 5000)
    kern<<<grid, kFfmaProbeThreads, 0, st>>>(0.9999f, 0.5f, iters, sink);  // warm-up
    cudaEventRecord(e0, st);
    kern<<<grid, kFfmaProbeThreads, 0, st>>>(0.9999f, 0.5f, iters, sink);
    cudaEventRecord(e1, st);
    e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (e != cudaSuccess) return from_cuda(e);
    const double flop = static_cast<double>(grid) * kFfmaProbeThreads * iters * kFfmaProbeChains * 2.0;
    *tflops = ms > 0.f ? flop / (ms * 1e-3) / 1e12 : 0.0;
    return 0;
}
