// Shared definitions of the GEMM kernels: problem arguments, split-K
// bookkeeping, the device status word and the bounded mbarrier wait.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace sg {

// Bits of the device status word (any non-zero value is reported as
// SGEMM_ERR_DEVICE_TIMEOUT by sgemm_check_status).
enum : int {
    kStatusTimeoutProducer = 1,
    kStatusTimeoutMma = 2,
    kStatusTimeoutEpilogue = 4,
    kStatusTimeoutDrain = 8,
};

// Test-only flag: withhold the first producer arrive (see the header).
enum : int { kDebugWithholdArrive = 1 };

// One GEMM call: C = alpha * A * B + beta * C, row-major, leading dimensions
// in elements.  Offsets are formed in 64-bit arithmetic.
struct GemmArgs {
    int M, N, K;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
};

// Work decomposition shared by both paths.  A work unit is one (tile, K
// slice) pair; the K tiles of slice s are [s*KT/S, (s+1)*KT/S).
struct Schedule {
    int m_tiles, n_tiles;
    int k_tiles;   // ceil(K / BK)
    int splits;    // S >= 1
    int units;     // m_tiles * n_tiles * S
    int group_m;   // tile raster: groups of group_m tile rows, row index fastest
};

struct DeviceCtl {
    float *ws;           // split-K partial tiles: [tile][split][tile elements]
    int *counters;       // split-K arrival counters, one per tile, kept at 0
    int *status;         // device status word
    long long wait_budget;  // clock64 cycles a bounded wait may spin
    int debug_flags;
};

struct UnitCoord {
    int mt, nt, tile, split, kb, ke;
};

__device__ __forceinline__ UnitCoord decode_unit(const Schedule &s, int u) {
    UnitCoord c;
    c.split = u % s.splits;
    c.tile = u / s.splits;
    const int per_group = s.group_m * s.n_tiles;
    const int g = c.tile / per_group;
    const int r = c.tile - g * per_group;
    const int rows_here = min(s.group_m, s.m_tiles - g * s.group_m);
    c.mt = g * s.group_m + r % rows_here;
    c.nt = r / rows_here;
    c.kb = static_cast<int>((static_cast<long long>(c.split) * s.k_tiles) / s.splits);
    c.ke = static_cast<int>((static_cast<long long>(c.split + 1) * s.k_tiles) / s.splits);
    return c;
}

// Spin on an mbarrier phase with a cycle budget.  Returns false when the
// budget runs out (the status word and the CTA's abort flag are then set) or
// when another role of the CTA has already aborted.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag,
                                                  const DeviceCtl &ctl, int status_bit) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > ctl.wait_budget) {
            *abort_flag = 1;
            atomicOr(ctl.status, status_bit);
            return false;
        }
    }
}

}  // namespace sg
