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
// the first call made on it.  With lazy module loading (the CUDA default)
// that first call is also when the arrays and the kernels' code are loaded
// onto the device, so the set-up loads every kernel this entry point can
// launch there and then: after it, later calls leave the device's free
// memory unchanged.
#include <cuda_runtime.h>

#include <atomic>
#include <cstddef>
#include <mutex>

#include "launch.h"
#include "sgemm_gb300.h"

namespace {

constexpr size_t kScratchFloats = size_t(4) << 20;  // 16 MiB of split-K partial tiles
constexpr int kScratchCounters = 4096;              // one arrival counter per output tile
constexpr int kMaxDevices = 64;
constexpr long long kWaitBudget = 20000000000LL;    // same bounded-wait budget as sgemm_ex
constexpr long long kDebugWaitBudget = 2000000LL;   // ~1 ms, test-only withheld-arrive mode

__device__ __align__(256) float g_scratch[kScratchFloats];
__device__ __align__(256) int g_scratch_counters[kScratchCounters];
__device__ __align__(256) int g_scratch_status;

struct DeviceScratch {
    bool ready = false;
    float *partials = nullptr;
    int *counters = nullptr;
    int *status = nullptr;
    int sms = 0;
    int pair_slots = 0;  // CTA pairs of the 3xTF32 kernel resident at once
};

std::mutex g_setup_mu;
DeviceScratch g_scratch_ptrs[kMaxDevices];
// test hook: debug flags for the next call (sgemm_noalloc_debug_flags)
std::atomic<int> g_next_debug_flags{0};

// Resolve the device addresses of the arrays on the current device and load
// the kernels (once per device).
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
        if ((e = sg::tf32x3_preload()) != cudaSuccess || (e = sg::scale_c_preload()) != cudaSuccess)
            return static_cast<int>(e);
        d.sms = sms;
        d.pair_slots = sg::tf32x3_pair_slots();
        d.ready = true;
    }
    *out = &d;
    return 0;
}

}  // namespace

namespace sg {

int noalloc_take_status() {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return -static_cast<int>(e);
    if (dev < 0 || dev >= kMaxDevices) return 0;
    std::lock_guard<std::mutex> lk(g_setup_mu);
    DeviceScratch &d = g_scratch_ptrs[dev];
    if (!d.ready) return 0;  // no call has run on this device
    int word = 0;
    if ((e = cudaMemcpy(&word, d.status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess)
        return -static_cast<int>(e);
    if (word == 0) return 0;
    // a kernel that gave up may have left arrival counters non-zero: wait for
    // every stream of the device, then clear them and the word
    if ((e = cudaDeviceSynchronize()) != cudaSuccess ||
        (e = cudaMemset(d.counters, 0, sizeof(int) * kScratchCounters)) != cudaSuccess ||
        (e = cudaMemset(d.status, 0, sizeof(int))) != cudaSuccess)
        return -static_cast<int>(e);
    return 1;
}

}  // namespace sg

extern "C" int sgemm_noalloc_debug_flags(int flags) {
    if (flags & ~SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE) return -1;
    g_next_debug_flags.store(flags);
    return 0;
}

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
    if ((rc = sg::plan_tensor_call(M, N, K, A, lda, B, ldb, beta, C, ldc, splits, d->sms, d->pair_slots,
                                   kScratchFloats, &plan)) != 0)
        return rc;
    const int debug = g_next_debug_flags.exchange(0);
    sg::DeviceCtl ctl{};
    ctl.status = d->status;
    ctl.wait_budget = (debug & SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE) ? kDebugWaitBudget : kWaitBudget;
    ctl.debug_flags = (debug & SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE) ? sg::kDebugWithholdArrive : 0;
    if (plan.ws_floats > 0) {  // split-K or split tail: tiles shared by several units
        if (plan.ws_floats > kScratchFloats || plan.tiles > kScratchCounters) return SGEMM_ERR_SCRATCH_LIMIT;
        // The counters are zero here: they start at zero when the library's
        // device code is loaded, the kernel puts each one back to zero when
        // its tile is finished, and a call that gave up a bounded wait sets
        // the status word, whose check (sgemm_check_status) clears them.
        ctl.ws = d->partials;
        ctl.counters = d->counters;
        ctl.ws_end = d->partials + kScratchFloats;
        ctl.n_counters = kScratchCounters;
    }
    sg::GemmArgs g{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
    sg::set_extents(g, 1, false, ctl.status);
    return static_cast<int>(
        sg::tf32x3_launch(plan.tile_m, g, plan.sch, ctl, plan.vec_a, plan.vec_b, plan.vec_c, plan.grid, st));
}
