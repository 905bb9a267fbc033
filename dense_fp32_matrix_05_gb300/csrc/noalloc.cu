// sgemm_noalloc: the split-K 3xTF32 GEMM with its scratch memory inside the
// library image instead of in cudaMalloc'd memory.
//
// Some callers must not have a library allocate device memory behind their
// back: programs that reserve the whole GPU for their own memory pool or
// arena up front (an extra cudaMalloc then fails, or silently breaks their
// accounting of free memory), and latency-sensitive loops in which the
// implicit device-wide synchronisation of cudaMalloc/cudaFree would stall
// every other stream.  This entry point serves them: the split-K partial
// tiles, the arrival counters and the device status word live in file-scope
// __device__ arrays of fixed size, so a call only launches work.
//
// The arrays exist once per GPU that loads this library and stay resident
// until the process exits (about 16 MiB + 16 KiB per GPU).  In host code
// their names are only host-side stand-ins; the device addresses are fetched
// once per device with cudaGetSymbolAddress, with that device current, on
// the first call made on it.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "launch.h"
#include "sgemm_gb300.h"

namespace {

constexpr size_t kScratchFloats = size_t(4) << 20;  // 16 MiB of split-K partial tiles
constexpr int kScratchCounters = 4096;              // one arrival counter per output tile
constexpr int kMaxDevices = 64;
constexpr long long kWaitBudget = 20000000000LL;    // same bounded-wait budget as sgemm_ex

__device__ __align__(256) float g_scratch[kScratchFloats];
__device__ __align__(256) int g_scratch_counters[kScratchCounters];
__device__ __align__(256) int g_scratch_status;

struct DeviceScratch {
    bool ready = false;
    float *partials = nullptr;
    int *counters = nullptr;
    int *status = nullptr;
    int sms = 0;
};

std::mutex g_setup_mu;
DeviceScratch g_scratch_ptrs[kMaxDevices];

// Resolve the device addresses of the arrays on the current device (once).
int device_scratch(DeviceScratch **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e == cudaErrorNoDevice ? SGEMM_ERR_NO_DEVICE : static_cast<int>(e);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceScratch &d = g_scratch_ptrs[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return static_cast<int>(e);
        if (!(major == 10 && minor == 3)) return SGEMM_ERR_UNSUPPORTED_DEVICE;
        void *p = nullptr;
        if ((e = cudaGetSymbolAddress(&p, g_scratch)) != cudaSuccess) return static_cast<int>(e);
        d.partials = static_cast<float *>(p);
        if ((e = cudaGetSymbolAddress(&p, g_scratch_counters)) != cudaSuccess) return static_cast<int>(e);
        d.counters = static_cast<int *>(p);
        if ((e = cudaGetSymbolAddress(&p, g_scratch_status)) != cudaSuccess) return static_cast<int>(e);
        d.status = static_cast<int *>(p);
        d.sms = sms;
        d.ready = true;
    }
    *out = &d;
    return 0;
}

}  // namespace

extern "C" int sgemm_noalloc(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                             float beta, float *C, int ldc, sgemm_stream_t stream, int splits) {
    sg::TensorPlan plan;
    // argument checks first: they make no CUDA call
    int rc = sg::check_tensor_call(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, splits);
    if (rc != 0) return rc;
    if (M == 0 || N == 0) return 0;
    DeviceScratch *d = nullptr;
    if ((rc = device_scratch(&d)) != 0) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (alpha == 0.f || K == 0) {
        if (beta == 1.f) return 0;
        return static_cast<int>(sg::scale_c_launch(C, ldc, M, N, beta, d->sms, st));
    }
    if ((rc = sg::plan_tensor_call(M, N, K, A, lda, B, ldb, beta, C, ldc, splits, d->sms, kScratchFloats, &plan)) != 0)
        return rc;
    sg::DeviceCtl ctl{};
    ctl.status = d->status;
    ctl.wait_budget = kWaitBudget;
    ctl.debug_flags = 0;
    if (plan.ws_floats > 0) {  // split-K or split tail: tiles shared by several units
        if (plan.ws_floats > kScratchFloats || plan.tiles > kScratchCounters) return SGEMM_ERR_SCRATCH_LIMIT;
        // the array keeps the previous call's contents; the counters must
        // start at zero (a call that gave up a bounded wait can leave some set)
        cudaError_t e = cudaMemsetAsync(d->counters, 0, sizeof(int) * static_cast<size_t>(plan.tiles), st);
        if (e != cudaSuccess) return static_cast<int>(e);
        ctl.ws = d->partials;
        ctl.counters = d->counters;
    }
    sg::GemmArgs g{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
    return static_cast<int>(
        sg::tf32x3_launch(plan.tile_m, g, plan.sch, ctl, plan.vec_a, plan.vec_b, plan.vec_c, plan.grid, st));
}
