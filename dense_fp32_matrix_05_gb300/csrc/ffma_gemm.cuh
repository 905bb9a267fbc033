// SGEMM on the CUDA cores (fp32 FFMA): exact fp32 products and sums.
//
// Structure (re-done for sm_103a from the ideas of "NVIDIA_SGEMM_PRACTICE",
// sections "kernel 2" shared-memory tiles, "kernel 4" 2-D thread tiles,
// "kernel 5" fragment registers, "kernel 6" 128-bit loads, "kernel 7"
// prefetching, and the zero-filled edge tiles of "matmul_opt.cu"):
//   - CTA tile BM x BN x 16, 256 threads, each thread an 8 x 8 block of C
//     (two 4-row x two 4-column sub-blocks, so fragment reads are 128-bit);
//     warp tile 32 x 64;
//   - an STAGES-deep cp.async ring: 16-byte copies when a matrix's rows are
//     16-byte aligned, 4-byte copies otherwise; edges are zero-filled by the
//     copy itself (src-size < copy size);
//   - A is kept K-major in shared memory (as stored in global memory) with
//     its 16-byte chunks XOR-swizzled by (row / 4) % 4, so the four distinct
//     rows a warp reads per instruction fall in four different bank groups;
//     B is kept N-major, read as 8 consecutive 16-byte chunks per warp;
//   - per 2-k step a thread loads its 8 rows x 2 k of A (8-byte loads: with
//     4 k at a time the A fragment pushed the 128 x 128 tile past the 128
//     registers two CTAs per SM allow, and it spilled) and, per k, 8 values
//     of B, and updates 64 accumulators, held as 32 column pairs so that
//     each k takes 32 packed fma.rn.f32x2 (same per-element rounding and
//     order as fmaf, half the issue slots);
//   - epilogue alpha*acc + beta*C (C not read when beta == 0), 128-bit
//     accesses when C rows are aligned, predicated edges; split-K partials
//     go to a workspace and the last slice to arrive sums them in order.
#pragma once
#include <cstdint>

#include "common.cuh"

namespace sg {
namespace ffma {

constexpr int kThreads = 256;
constexpr int kBK = 16;

template <int BM, int BN, int STAGES>
struct Cfg {
    static constexpr int kWarpsN = BN / 64;
    static constexpr int kWarpsM = BM / 32;
    static_assert(kWarpsM * kWarpsN == 8, "8 warps of 32 x 64");
    static constexpr int kAFloats = BM * kBK;
    static constexpr int kBFloats = kBK * BN;
    static constexpr int kStageFloats = kAFloats + kBFloats;
    static constexpr int kSmemBytes = STAGES * kStageFloats * 4 + 16;
};

template <int BM, int BN>
__device__ __forceinline__ void load_stage(const GemmArgs &g, bool vec_a, bool vec_b, int m0, int n0,
                                           int k0, uint32_t sA, uint32_t sB, int tid) {
    // A tile: BM rows x 16 k, K-major, chunk c of row r stored at c ^ ((r >> 2) & 3)
    if (vec_a) {
#pragma unroll
        for (int j = tid; j < BM * 4; j += kThreads) {
            const int r = j >> 2, kc = j & 3;
            const int m = m0 + r, k = k0 + kc * 4;
            const float *src = g.A;
            uint32_t bytes = 0;
            if (m < g.M && k < g.K) {
                src = g.A + static_cast<long long>(m) * g.lda + k;
                bytes = static_cast<uint32_t>(min(4, g.K - k) * 4);
                if (!SG_IN_A(g, src, static_cast<int>(bytes / 4))) {
                    src = g.A;
                    bytes = 0;
                }
            }
            cp_async16(sA + static_cast<uint32_t>((r * kBK + ((kc ^ ((r >> 2) & 3)) << 2)) * 4), src, bytes);
        }
    } else {
#pragma unroll 4
        for (int j = tid; j < BM * kBK; j += kThreads) {
            const int r = j >> 4, kk = j & 15;
            const int m = m0 + r, k = k0 + kk;
            const bool ok = m < g.M && k < g.K && SG_IN_A(g, g.A + static_cast<long long>(m) * g.lda + k, 1);
            const float *src = ok ? g.A + static_cast<long long>(m) * g.lda + k : g.A;
            const int col = (((kk >> 2) ^ ((r >> 2) & 3)) << 2) | (kk & 3);
            cp_async4(sA + static_cast<uint32_t>((r * kBK + col) * 4), src, ok ? 4u : 0u);
        }
    }
    // B tile: 16 k x BN, N-major
    if (vec_b) {
#pragma unroll
        for (int j = tid; j < kBK * BN / 4; j += kThreads) {
            const int r = j / (BN / 4), nc = j % (BN / 4);
            const int k = k0 + r, n = n0 + nc * 4;
            const float *src = g.B;
            uint32_t bytes = 0;
            if (k < g.K && n < g.N) {
                src = g.B + static_cast<long long>(k) * g.ldb + n;
                bytes = static_cast<uint32_t>(min(4, g.N - n) * 4);
                if (!SG_IN_B(g, src, static_cast<int>(bytes / 4))) {
                    src = g.B;
                    bytes = 0;
                }
            }
            cp_async16(sB + static_cast<uint32_t>((r * BN + nc * 4) * 4), src, bytes);
        }
    } else {
#pragma unroll 4
        for (int j = tid; j < kBK * BN; j += kThreads) {
            const int r = j / BN, c = j % BN;
            const int k = k0 + r, n = n0 + c;
            const bool ok = k < g.K && n < g.N && SG_IN_B(g, g.B + static_cast<long long>(k) * g.ldb + n, 1);
            const float *src = ok ? g.B + static_cast<long long>(k) * g.ldb + n : g.B;
            cp_async4(sB + static_cast<uint32_t>((r * BN + c) * 4), src, ok ? 4u : 0u);
        }
    }
}

template <int BM, int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 2)
    ffma_gemm_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ Schedule sch,
                     const __grid_constant__ DeviceCtl ctl, int vec_a, int vec_b, int vec_c) {
    using Cf = Cfg<BM, BN, STAGES>;
    extern __shared__ __align__(16) float smem_f[];
    __shared__ int s_last;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp / Cf::kWarpsN, wn = warp % Cf::kWarpsN;
    const int lm = lane >> 3, ln = lane & 7;
    const int row_base = wm * 32 + lm * 4;  // rows row_base+i and row_base+16+i, i < 4
    const int col_base = wn * 64 + ln * 4;  // cols col_base+j and col_base+32+j, j < 4

    const UnitCoord c = decode_unit(sch, blockIdx.x);
    const int m0 = c.mt * BM, n0 = c.nt * BN;
    const int KT = c.ke - c.kb;
    const uint32_t s0 = smem_u32(smem_f);

    // accumulators in column pairs: acc2[i][q] = (C[i][2q], C[i][2q + 1])
    uint64_t acc2[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc2[i][q] = 0ull;

#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) {
        if (s < KT) {
            const uint32_t st = s0 + static_cast<uint32_t>(s * Cf::kStageFloats * 4);
            load_stage<BM, BN>(g, vec_a, vec_b, m0, n0, (c.kb + s) * kBK, st, st + Cf::kAFloats * 4, tid);
        }
        cp_async_commit();
    }

#pragma unroll 1
    for (int t = 0; t < KT; ++t) {
        cp_async_wait<STAGES - 2>();
        __syncthreads();
        {
            const int nt = t + STAGES - 1;
            if (nt < KT) {
                const uint32_t st = s0 + static_cast<uint32_t>((nt % STAGES) * Cf::kStageFloats * 4);
                load_stage<BM, BN>(g, vec_a, vec_b, m0, n0, (c.kb + nt) * kBK, st, st + Cf::kAFloats * 4, tid);
            }
            cp_async_commit();
        }
        const uint32_t sA = s0 + static_cast<uint32_t>((t % STAGES) * Cf::kStageFloats * 4);
        const uint32_t sB = sA + Cf::kAFloats * 4;
#pragma unroll
        for (int kh = 0; kh < 8; ++kh) {
            const int kq = kh >> 1;
            float a[8][2];
            const uint32_t chunk = static_cast<uint32_t>(((kq ^ lm) << 2) + 2 * (kh & 1));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                lds2f(sA + ((row_base + i) * kBK + chunk) * 4, a[i][0], a[i][1]);
                lds2f(sA + ((row_base + 16 + i) * kBK + chunk) * 4, a[4 + i][0], a[4 + i][1]);
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                const int k = kh * 2 + kk;
                uint64_t b[4];
                lds_pairs(sB + (k * BN + col_base) * 4, b[0], b[1]);
                lds_pairs(sB + (k * BN + col_base + 32) * 4, b[2], b[3]);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint64_t ai = pair_bcast(a[i][kk]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) ffma2(acc2[i][q], ai, b[q]);
                }
            }
        }
    }
    cp_async_wait<0>();

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) pair_split(acc2[i][q], acc[i][2 * q], acc[i][2 * q + 1]);

    if (c.nseg > 1 && (ctl.ws == nullptr || ctl.counters == nullptr)) {
        // a shared tile without a workspace: report, never dereference
        if (tid == 0) atomicOr(ctl.status, kStatusNoWorkspace);
        return;
    }
    if (c.nseg > 1) {
        constexpr int kTileElems = BM * BN;
        float *wt = ctl.ws + (c.slot0 + c.seg) * kTileElems + tid * 64;
        if (SG_IN_WS(ctl, wt, 64)) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                __stcg(reinterpret_cast<float4 *>(wt + i * 8), make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]));
                __stcg(reinterpret_cast<float4 *>(wt + i * 8 + 4),
                       make_float4(acc[i][4], acc[i][5], acc[i][6], acc[i][7]));
            }
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const bool cnt_ok = !kDebugBounds || (c.tile >= 0 && c.tile < ctl.n_counters);
            if (!cnt_ok) atomicOr(ctl.status, kStatusOutOfBounds);
            const int prev = cnt_ok ? atomicAdd(ctl.counters + c.tile, 1) : -1;
            s_last = (prev == c.nseg - 1) ? 1 : 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const float *wb = ctl.ws + c.slot0 * kTileElems + tid * 64;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
#pragma unroll 1
        for (int sp = 0; sp < c.nseg; ++sp) {
            const float *p = wb + static_cast<long long>(sp) * kTileElems;
            if (!SG_IN_WS(ctl, p, 64)) continue;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(p + i * 8));
                const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(p + i * 8 + 4));
                acc[i][0] += x0.x; acc[i][1] += x0.y; acc[i][2] += x0.z; acc[i][3] += x0.w;
                acc[i][4] += x1.x; acc[i][5] += x1.y; acc[i][6] += x1.z; acc[i][7] += x1.w;
            }
        }
        if (tid == 0) ctl.counters[c.tile] = 0;
    }

    // epilogue: C = alpha * acc + beta * C
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + row_base + (i < 4 ? i : 12 + i);
        if (m >= g.M) continue;
        float *crow = g.C + static_cast<long long>(m) * g.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + col_base + h * 32;
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) r[e] = g.alpha * acc[i][h * 4 + e];
            if (vec_c && n + 3 < g.N) {
                if (!SG_IN_C(g, crow + n, 4)) continue;
                float4 *p = reinterpret_cast<float4 *>(crow + n);
                if (g.beta != 0.f) {
                    const float4 o = *p;
                    r[0] = fmaf(g.beta, o.x, r[0]);
                    r[1] = fmaf(g.beta, o.y, r[1]);
                    r[2] = fmaf(g.beta, o.z, r[2]);
                    r[3] = fmaf(g.beta, o.w, r[3]);
                }
                *p = make_float4(r[0], r[1], r[2], r[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (n + e < g.N && SG_IN_C(g, crow + n + e, 1)) {
                        float *p = crow + n + e;
                        *p = (g.beta == 0.f) ? r[e] : fmaf(g.beta, *p, r[e]);
                    }
                }
            }
        }
    }
}

// Large-tile form: CTA tile 128 x 256 x 32, one CTA of 256 threads per SM,
// warps 2 (M) x 4 (N) of 64 x 64, each thread 8 rows x 16 columns (64 packed
// column pairs).  A is stored transposed in shared memory (k rows of the
// tile's 128 m, pitch 132 floats, filled by 4-byte cp.async copies that
// transpose on the way), so per k a thread reads its 8 A values with two
// 128-bit loads and its 16 B values with four, broadcasts the 8 A values
// into pairs and issues 64 fma.rn.f32x2: 82 % of its instructions are FMAs
// (70 % in the 128 x 128 form), and one CTA per SM leaves room for the 128
// accumulators and the next k's operands in registers.  A thread's rows are
// two groups of 4 (lm * 4 and 32 + lm * 4 in its warp's 64) and its columns
// four groups of 4 (ln * 4 + 16 q), so each 128-bit shared load of a warp
// touches every bank once.  Same per-element arithmetic and order as the
// other FFMA kernels (an in-order fma.rn chain over k).  Stages of 32 k
// (two of the schedule's 16-k tiles; one barrier per 32 k) measured 2 %
// faster than 16 k on GB300 at 2048-8192 cubed.
constexpr int kBigBM = 128;
constexpr int kBigBN = 256;
constexpr int kBigBK = 32;              // k per stage (a whole number of the schedule's 16-k tiles)
constexpr int kBigPitchA = kBigBM + 4;  // A^T row pitch: stores of a warp hit 2 banks at most
constexpr int kBigStages = 4;
static_assert(kBigBK % kBK == 0, "stages hold whole schedule k tiles");

struct BigCfg {
    static constexpr int kAFloats = kBigBK * kBigPitchA;
    static constexpr int kBFloats = kBigBK * kBigBN;
    static constexpr int kStageFloats = kAFloats + kBFloats;
    static constexpr int kSmemBytes = kBigStages * kStageFloats * 4 + 16;
};

// One stage: A^T (kBigBK k x 128 m) and B (kBigBK k x 256 n); elements at
// or beyond kend (the end of K, or of this unit's K slice) or outside M, N
// are zero-filled by the copies.
__device__ __forceinline__ void big_load_stage(const GemmArgs &g, bool vec_b, int m0, int n0, int k0, int kend,
                                               uint32_t sA, uint32_t sB, int tid) {
    // element e = tid + 256 i: row m = e / kBigBK, k = e % kBigBK (a warp
    // reads pieces of A's rows kBigBK floats long)
#pragma unroll
    for (int i = 0; i < kBigBM * kBigBK / kThreads; ++i) {
        const int e = tid + i * kThreads;
        const int r = e / kBigBK, kk = e % kBigBK;
        const int m = m0 + r, k = k0 + kk;
        const bool ok = m < g.M && k < kend && SG_IN_A(g, g.A + static_cast<long long>(m) * g.lda + k, 1);
        const float *src = ok ? g.A + static_cast<long long>(m) * g.lda + k : g.A;
        cp_async4(sA + static_cast<uint32_t>((kk * kBigPitchA + r) * 4), src, ok ? 4u : 0u);
    }
    if (vec_b) {
#pragma unroll
        for (int i = 0; i < kBigBK * kBigBN / 4 / kThreads; ++i) {
            const int j = tid + i * kThreads;
            const int r = j / (kBigBN / 4), nc = j % (kBigBN / 4);
            const int k = k0 + r, n = n0 + nc * 4;
            const float *src = g.B;
            uint32_t bytes = 0;
            if (k < kend && n < g.N) {
                src = g.B + static_cast<long long>(k) * g.ldb + n;
                bytes = static_cast<uint32_t>(min(4, g.N - n) * 4);
                if (!SG_IN_B(g, src, static_cast<int>(bytes / 4))) {
                    src = g.B;
                    bytes = 0;
                }
            }
            cp_async16(sB + static_cast<uint32_t>((r * kBigBN + nc * 4) * 4), src, bytes);
        }
    } else {
#pragma unroll 4
        for (int j = tid; j < kBigBK * kBigBN; j += kThreads) {
            const int r = j / kBigBN, c = j % kBigBN;
            const int k = k0 + r, n = n0 + c;
            const bool ok = k < kend && n < g.N && SG_IN_B(g, g.B + static_cast<long long>(k) * g.ldb + n, 1);
            const float *src = ok ? g.B + static_cast<long long>(k) * g.ldb + n : g.B;
            cp_async4(sB + static_cast<uint32_t>((r * kBigBN + c) * 4), src, ok ? 4u : 0u);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 1)
    ffma_big_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ Schedule sch,
                    const __grid_constant__ DeviceCtl ctl, int vec_b, int vec_c) {
    extern __shared__ __align__(16) float smem_f[];
    __shared__ int s_last;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int wm = warp >> 2, wn = warp & 3;
    const int lm = lane >> 2, ln = lane & 3;
    const int rowa = wm * 64 + lm * 4;  // rows rowa + i and rowa + 32 + i, i < 4
    const int colb = wn * 64 + ln * 4;  // columns colb + 16 q + j, q < 4, j < 4

    // one unit per CTA: split-K units, or whole tiles followed by the K
    // slices of a split tail (the leftover tiles of a partly empty last wave)
    const int u = static_cast<int>(blockIdx.x);
    UnitCoord c;
    if (sch.tail_tiles > 0 && u >= sch.dp_tiles) {
        c = slice_unit(sch, sch.dp_tiles, u - sch.dp_tiles, sch.tail_splits, 0);
    } else if (sch.tail_tiles > 0) {
        tile_coords(sch, u, c);
        c.kb = 0;
        c.ke = sch.k_tiles;
        c.seg = 0;
        c.nseg = 1;
        c.slot0 = 0;
    } else {
        c = decode_unit(sch, u);
    }
    const int m0 = c.mt * kBigBM, n0 = c.nt * kBigBN;
    const int kend = min(g.K, c.ke * kBK);             // end of this unit's K range
    constexpr int kTilesPerStage = kBigBK / kBK;
    const int KT = (c.ke - c.kb + kTilesPerStage - 1) / kTilesPerStage;  // stages of this unit
    const uint32_t s0 = smem_u32(smem_f);

    // acc[i][p]: row i of the thread (rowa + i, then rowa + 32 + i - 4),
    // column pair p (columns colb + 16 (p / 2) + 2 (p % 2) and + 1)
    uint64_t acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int p = 0; p < 8; ++p) acc[i][p] = 0ull;

#pragma unroll
    for (int s = 0; s < kBigStages - 1; ++s) {
        if (s < KT) {
            const uint32_t st = s0 + static_cast<uint32_t>(s * BigCfg::kStageFloats * 4);
            big_load_stage(g, vec_b != 0, m0, n0, c.kb * kBK + s * kBigBK, kend, st, st + BigCfg::kAFloats * 4, tid);
        }
        cp_async_commit();
    }

#pragma unroll 1
    for (int t = 0; t < KT; ++t) {
        cp_async_wait<kBigStages - 2>();
        __syncthreads();
        {
            const int nt = t + kBigStages - 1;
            if (nt < KT) {
                const uint32_t st = s0 + static_cast<uint32_t>((nt % kBigStages) * BigCfg::kStageFloats * 4);
                big_load_stage(g, vec_b != 0, m0, n0, c.kb * kBK + nt * kBigBK, kend, st, st + BigCfg::kAFloats * 4,
                               tid);
            }
            cp_async_commit();
        }
        const float *sA = smem_f + (t % kBigStages) * BigCfg::kStageFloats;
        const float *sB = sA + BigCfg::kAFloats;
#pragma unroll
        for (int k = 0; k < kBigBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4 *>(sA + k * kBigPitchA + rowa);
            const float4 a1 = *reinterpret_cast<const float4 *>(sA + k * kBigPitchA + rowa + 32);
            uint64_t b[8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const ulonglong2 v = *reinterpret_cast<const ulonglong2 *>(sB + k * kBigBN + colb + 16 * q);
                b[2 * q] = v.x;
                b[2 * q + 1] = v.y;
            }
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint64_t ai = pair_bcast(a[i]);
#pragma unroll
                for (int p = 0; p < 8; ++p) ffma2(acc[i][p], ai, b[p]);
            }
        }
    }
    cp_async_wait<0>();

    if (c.nseg > 1 && (ctl.ws == nullptr || ctl.counters == nullptr)) {
        if (tid == 0) atomicOr(ctl.status, kStatusNoWorkspace);
        return;
    }
    float out[8][16];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int p = 0; p < 8; ++p) pair_split(acc[i][p], out[i][2 * p], out[i][2 * p + 1]);

    if (c.nseg > 1) {
        // shared tile: partials in the workspace, the last unit sums them in order
        constexpr int kTileElems = kBigBM * kBigBN;
        float *wt = ctl.ws + (c.slot0 + c.seg) * kTileElems + tid * 128;
        if (SG_IN_WS(ctl, wt, 128)) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    __stcg(reinterpret_cast<float4 *>(wt + i * 16 + 4 * q),
                           make_float4(out[i][4 * q], out[i][4 * q + 1], out[i][4 * q + 2], out[i][4 * q + 3]));
        }
        __threadfence();
        __syncthreads();
        if (tid == 0) {
            const bool cnt_ok = !kDebugBounds || (c.tile >= 0 && c.tile < ctl.n_counters);
            if (!cnt_ok) atomicOr(ctl.status, kStatusOutOfBounds);
            const int prev = cnt_ok ? atomicAdd(ctl.counters + c.tile, 1) : -1;
            s_last = (prev == c.nseg - 1) ? 1 : 0;
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        const float *wb = ctl.ws + c.slot0 * kTileElems + tid * 128;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 16; ++j) out[i][j] = 0.f;
#pragma unroll 1
        for (int sp = 0; sp < c.nseg; ++sp) {
            const float *pw = wb + static_cast<long long>(sp) * kTileElems;
            if (!SG_IN_WS(ctl, pw, 128)) continue;
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(pw + i * 16 + 4 * q));
                    out[i][4 * q] += x.x;
                    out[i][4 * q + 1] += x.y;
                    out[i][4 * q + 2] += x.z;
                    out[i][4 * q + 3] += x.w;
                }
        }
        if (tid == 0) ctl.counters[c.tile] = 0;
    }

    // epilogue: C = alpha * acc + beta * C
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int m = m0 + rowa + (i < 4 ? i : 28 + i);
        if (m >= g.M) continue;
        float *crow = g.C + static_cast<long long>(m) * g.ldc;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int n = n0 + colb + 16 * q;
            float r[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) r[e] = g.alpha * out[i][4 * q + e];
            if (vec_c && n + 3 < g.N) {
                if (!SG_IN_C(g, crow + n, 4)) continue;
                float4 *p = reinterpret_cast<float4 *>(crow + n);
                if (g.beta != 0.f) {
                    const float4 o = *p;
                    r[0] = fmaf(g.beta, o.x, r[0]);
                    r[1] = fmaf(g.beta, o.y, r[1]);
                    r[2] = fmaf(g.beta, o.z, r[2]);
                    r[3] = fmaf(g.beta, o.w, r[3]);
                }
                *p = make_float4(r[0], r[1], r[2], r[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (n + e < g.N && SG_IN_C(g, crow + n + e, 1)) {
                        float *p = crow + n + e;
                        *p = (g.beta == 0.f) ? r[e] : fmaf(g.beta, *p, r[e]);
                    }
                }
            }
        }
    }
}

// C = beta * C (C := 0 when beta == 0, without reading C): the alpha == 0 /
// K == 0 case of the problem statement.
__global__ void scale_c_kernel(float *C, long long ldc, int M, int N, float beta) {
    const long long total = static_cast<long long>(M) * N;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long m = idx / N, n = idx - m * N;
        float *p = C + m * ldc + n;
        *p = (beta == 0.f) ? 0.f : beta * *p;
    }
}

}  // namespace ffma
}  // namespace sg
