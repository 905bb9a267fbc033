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
    kStatusNoWorkspace = 16,  // a shared tile met a missing workspace (a planner bug)
    kStatusDeferOverflow = 32,  // a CTA got more shared tiles than it can defer (a planner bug)
    kStatusOutOfBounds = 64,    // SGEMM_DEBUG builds: an access outside its matrix was skipped
};

// SGEMM_DEBUG builds check every computed global-memory address of the
// kernels against the byte range of the matrix it belongs to (GemmArgs'
// extents, DeviceCtl's workspace); an address outside is not accessed, and
// the status bit kStatusOutOfBounds is set (never a trap).  The release
// build compiles the checks away.
#ifdef SGEMM_DEBUG
constexpr bool kDebugBounds = true;
#else
constexpr bool kDebugBounds = false;
#endif

// Test-only flag: withhold the first producer arrive (see the header).
enum : int { kDebugWithholdArrive = 1 };

// Implicit-GEMM convolution: B is not stored but read from an NCHW input X
// (B = X, matrix b of the batch = image b, sB = channels * H * W) as its
// im2col lowering, B[k][n] = X[c][oh * sh + kh * dh - ph][ow * sw + kw * dw - pw]
// with n = oh * OW + ow, zero outside the image, and k a numbering of the
// taps (c, kh, kw) (kConvTaps / kConvChannels below).  A is the filter,
// M filters x K in the same k order, C the image's NCHW output (ldc = N =
// OH * OW).
// Order of the K index of an implicit-GEMM convolution.
enum : int {
    kConvNone = 0,      // a plain GEMM
    kConvTaps = 1,      // k = (c * KH + kh) * KW + kw (OIHW filter rows)
    kConvChannels = 2,  // k = (kh * KW + kw) * C + c (OHWI filter rows, C % 16 == 0)
    kConvTapsDense = 3, // kConvTaps with every tap inside the image (no padding, or an input
                        // copied with zero borders): no bounds checks, tap offsets from a table
};
constexpr int kConvTabMax = 2048;  // taps of a kConvTapsDense table (ints in shared memory)

struct ConvGeom {
    int C;       // input channels
    int H, W;    // input plane
    int OW;      // output width
    int KH, KW;  // filter
    int sh, sw, ph, pw, dh, dw;
};

// One GEMM call: C = alpha * A * B + beta * C, row-major, leading dimensions
// in elements.  Offsets are formed in 64-bit arithmetic.  A strided batch
// (3xTF32 path) adds matrix b's offset b * sA, b * sB, b * sC (elements; a
// zero stride shares one matrix).
struct GemmArgs {
    int M, N, K;
    float alpha, beta;
    const float *A;
    long long lda;
    const float *B;
    long long ldb;
    float *C;
    long long ldc;
    long long sA = 0, sB = 0, sC = 0;
    ConvGeom cv{};  // implicit-GEMM convolution kernels only
    // One past the last float any access to A, B, C may touch (every matrix
    // of a batch, a convolution's whole input); checked in SGEMM_DEBUG
    // builds, which report into dbg_status.
    const float *a_end = nullptr, *b_end = nullptr;
    const float *c_end = nullptr;
    int *dbg_status = nullptr;
};

// SGEMM_DEBUG: is [p, p + n) inside [lo, hi)?  Reports when it is not.
template <typename T>
__device__ __forceinline__ bool in_bounds(const T *p, int n, const void *lo, const void *hi, int *status) {
    if constexpr (!kDebugBounds) {
        return true;
    } else {
        const char *b = reinterpret_cast<const char *>(p);
        const bool ok = lo != nullptr && b >= static_cast<const char *>(lo) &&
                        b + static_cast<long long>(n) * sizeof(T) <= static_cast<const char *>(hi);
        if (!ok && status) atomicOr(status, kStatusOutOfBounds);
        return ok;
    }
}
#define SG_IN_A(g, p, n) ::sg::in_bounds((p), (n), (g).A, (g).a_end, (g).dbg_status)
#define SG_IN_B(g, p, n) ::sg::in_bounds((p), (n), (g).B, (g).b_end, (g).dbg_status)
#define SG_IN_C(g, p, n) ::sg::in_bounds((p), (n), (g).C, (g).c_end, (g).dbg_status)

// Work decomposition.  A work unit is one (tile, K range) pair; a tile whose
// K range is spread over nseg > 1 units is finished by the last of its units
// to arrive, which adds the partial tiles in segment order.
//   Split-K (tail_tiles == 0): unit u = (tile u / S, slice u % S); slice s
//     covers K tiles [s*KT/S, (s+1)*KT/S); units are strided over the grid.
//   Whole waves + split tail (tail_tiles > 0): the first dp_tiles tiles (a
//     whole number of waves over the grid) are whole units, strided over the
//     grid, so every wave walks K in step and shares A/B slices in L2; the
//     remaining tail_tiles (< one wave) are cut into tail_splits K slices, one
//     slice per CTA, so the last wave is not left mostly idle.
struct Schedule {
    int m_tiles, n_tiles;
    int k_tiles;      // ceil(K / BK)
    int splits;       // S >= 1 (split-K)
    int units;        // split-K: m_tiles * n_tiles * S
    int group_m;      // tile raster: groups of group_m tile rows, row index fastest
    int dp_tiles;     // whole-wave tiles
    int tail_tiles;   // tiles after them, split along K (0 = split-K schedule)
    int tail_splits;  // K slices per tail tile
    int tpb;          // tiles per matrix of a batch (0: one matrix); tile t is tile t % tpb of matrix t / tpb
    int pair_shift;   // 1: the units are walked by CTA pairs (clusters of two CTAs, one walker each;
                      //    a tile is then 256 columns, 128 per CTA); 0: by single CTAs
};

struct DeviceCtl {
    float *ws;           // partial tiles, one slot of tile elements per unit of a shared tile
    int *counters;       // arrival counters, one per tile, kept at 0
    int *status;         // device status word
    long long wait_budget;  // clock64 cycles a bounded wait may spin
    int debug_flags;
    const float *ws_end = nullptr;  // one past the workspace (SGEMM_DEBUG checks)
    long long n_counters = 0;       // arrival counters available (SGEMM_DEBUG checks)
};
#define SG_IN_WS(ctl, p, n) ::sg::in_bounds((p), (n), (ctl).ws, (ctl).ws_end, (ctl).status)

struct UnitCoord {
    int b;            // matrix of the batch
    int mt, nt, tile;
    int kb, ke;       // K tiles [kb, ke)
    int seg, nseg;    // this unit's index among the tile's units, and their count
    long long slot0;  // workspace slot of segment 0 of this tile
};

__device__ __forceinline__ void tile_coords(const Schedule &s, int tile, UnitCoord &c) {
    int t = tile;
    c.b = 0;
    if (s.tpb > 0) {
        c.b = tile / s.tpb;
        t = tile - c.b * s.tpb;
    }
    const int per_group = s.group_m * s.n_tiles;
    const int g = t / per_group;
    const int r = t - g * per_group;
    const int rows_here = min(s.group_m, s.m_tiles - g * s.group_m);
    c.tile = tile;
    c.mt = g * s.group_m + r % rows_here;
    c.nt = r / rows_here;
}

// Unit u of a tile split into `splits` K slices: slice u % splits of tile
// first_tile + u / splits; its slots start at slot_base + (u / splits) * splits.
__device__ __forceinline__ UnitCoord slice_unit(const Schedule &s, int first_tile, int u, int splits,
                                                long long slot_base) {
    UnitCoord c;
    const int split = u % splits;
    const int t = u / splits;
    tile_coords(s, first_tile + t, c);
    c.seg = split;
    c.nseg = splits;
    c.slot0 = slot_base + static_cast<long long>(t) * splits;
    c.kb = static_cast<int>((static_cast<long long>(split) * s.k_tiles) / splits);
    c.ke = static_cast<int>((static_cast<long long>(split + 1) * s.k_tiles) / splits);
    return c;
}

// Split-K unit u.
__device__ __forceinline__ UnitCoord decode_unit(const Schedule &s, int u) {
    return slice_unit(s, 0, u, s.splits, 0);
}

// The work units of one walker (a CTA, or a CTA pair: cta = its index), in
// order: next_unit() advances the position (i: index of the next strided
// unit; tail: the tail slice was handed out) and returns the unit there.
// Every role of the CTA (of both CTAs of a pair) walks the same sequence.
__device__ __forceinline__ bool next_unit(const Schedule &s, int cta, int &i, bool &tail, UnitCoord &c) {
    const int walkers = static_cast<int>(gridDim.x) >> s.pair_shift;
    if (s.tail_tiles == 0) {
        const int u = cta + i * walkers;
        ++i;
        if (u >= s.units) return false;
        c = decode_unit(s, u);
        return true;
    }
    const int t = cta + i * walkers;
    if (t < s.dp_tiles) {
        ++i;
        tile_coords(s, t, c);
        c.kb = 0;
        c.ke = s.k_tiles;
        c.seg = 0;
        c.nseg = 1;
        c.slot0 = 0;
        return true;
    }
    if (tail || cta >= s.tail_tiles * s.tail_splits) return false;
    tail = true;
    c = slice_unit(s, s.dp_tiles, cta, s.tail_splits, 0);
    return true;
}

// Full unit coordinates (epilogue, MMA issuer).
struct UnitIter {
    int cta;
    int i;
    bool tail;
    UnitCoord c;  // the current unit (valid while ok)
    bool ok;
    __device__ __forceinline__ void start(const Schedule &s, int cta_) {
        cta = cta_;
        i = 0;
        tail = false;
        next(s);
    }
    __device__ __forceinline__ void next(const Schedule &s) { ok = next_unit(s, cta, i, tail, c); }
};

// Spin on an mbarrier phase with a cycle budget.  Returns false when the
// budget runs out (the status word and the CTA's abort flag are then set) or
// when another role of the CTA has already aborted.  CLUSTER: the phase is
// completed by threads of the other CTA of a pair (acquire at cluster scope).
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    if constexpr (CLUSTER) return mbar_try_wait_cluster(bar, parity);
    else return mbar_try_wait(bar, parity);
}

template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort_flag,
                                                  const DeviceCtl &ctl, int status_bit) {
    if (mbar_try<CLUSTER>(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try<CLUSTER>(bar, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > ctl.wait_budget) {
            *abort_flag = 1;
            atomicOr(ctl.status, status_bit);
            return false;
        }
    }
}

}  // namespace sg
