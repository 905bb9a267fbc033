// Wide-N SGEMM on the CUDA cores for short, shallow A (M <= 32, K <= 64),
// the im2col shapes whose time is the stream of B and C through HBM.
//
// The tiled kernels re-stage a sliver of A for every C tile and pay a
// pipeline fill per tile that K = 27 never amortises.  Here A stays resident
// in shared memory for the whole launch, transposed and zero-padded to
// 64 k x 32 rows, and persistent CTAs stream B through a cp.async ring in
// slabs of 16 k rows x 512 columns (16-byte copies when B's rows are
// 16-byte aligned, 4-byte copies otherwise; edges zero-filled by the copy).
// Thread t owns columns 2t and 2t + 1 of the current 512-column block and all
// 32 rows, held as packed row pairs: per k it reads 16 A row pairs (the same
// address for the whole warp, a broadcast) and its two B values, and issues
// 32 fma.rn.f32x2.  Each element is an in-order fp32 FMA chain over k, as
// in the tiled FFMA kernel.  When a block's last slab is done, C is written
// with 8-byte stores, 256 consecutive bytes per warp and row, then the next
// block's slabs are already in flight.
//
// Work decomposition follows the 2-D thread tiles of "NVIDIA_SGEMM_PRACTICE"
// (sections "kernel 4" and "kernel 5", here 32 x 2 per thread) and the
// prefetching of its "kernel 7", reorganised around a resident A.
//
// Convolution form (CONV): the implicit GEMM of a layer with at most 32
// filters and 64 taps (ConvGeom, k = (c * KH + kh) * KW + kw, the OIHW filter
// rows as A).  The columns run over the output pixels of all images
// (n = image * ldc + pixel, ldc = OH * OW); the slab copies gather B from the
// input image, 4 bytes each, zero-filled outside it, and C goes to the
// image's NCHW output (sC floats per image).  kConvTapsDense: every tap lies
// in the image (no padding, or an input copied with zero borders), so a copy
// is the column's window origin plus the tap's offset from a table in shared
// memory, without bounds checks.
#include <cstdint>

#include "common.cuh"
#include "launch.h"

namespace sg {
namespace wide {

constexpr int kThreads = 256;
constexpr int kCols = 2 * kThreads;  // C columns per block
constexpr int kMaxM = 32;
constexpr int kMaxK = 64;
constexpr int kKc = 16;              // k rows per slab
constexpr int kStages = 3;
constexpr int kStageFloats = kKc * kCols;
constexpr int kAFloats = kMaxK * kMaxM;  // A^T: row k holds A[0..31][k]
constexpr int kSmemBytes = (kStages * kStageFloats + kAFloats + kMaxK) * 4;  // + tap table (kMaxK ints)

// Slab q of this CTA: k rows [kc * 16, +16) of column block cb.
template <int CONV>
__device__ __forceinline__ void load_slab(const GemmArgs &g, bool vec_b, int cb, int kc, uint32_t dst, int tid,
                                          const int *tab) {
    const int n0 = cb * kCols;
    if constexpr (CONV == kConvTapsDense) {
        const ConvGeom &cv = g.cv;
        const float *col[2];
        bool n_ok[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + tid + h * kThreads;
            n_ok[h] = n < g.N;
            const int img = n_ok[h] ? n / static_cast<int>(g.ldc) : 0;
            const int pix = n_ok[h] ? n - img * static_cast<int>(g.ldc) : 0;
            const int oh = pix / cv.OW;
            col[h] = g.B + img * g.sB + (oh * cv.sh * cv.W + (pix - oh * cv.OW) * cv.sw);
        }
        const int kb = kc * kKc;
#pragma unroll 4
        for (int r = 0; r < kKc; ++r) {
            const bool k_ok = kb + r < g.K;
            const int off = tab[kb + r];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const bool ok = k_ok && n_ok[h] && SG_IN_B(g, col[h] + off, 1);
                cp_async4(dst + static_cast<uint32_t>((r * kCols + tid + h * kThreads) * 4), ok ? col[h] + off : g.B,
                          ok ? 4u : 0u);
            }
        }
    } else if constexpr (CONV == kConvTaps) {
        // this thread copies columns tid and tid + 256 of every slab row
        const ConvGeom &cv = g.cv;
        const float *col[2];
        int ih0[2], iw0[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + tid + h * kThreads;
            const bool n_ok = n < g.N;
            const int img = n_ok ? n / static_cast<int>(g.ldc) : 0;
            const int pix = n_ok ? n - img * static_cast<int>(g.ldc) : 0;
            const int oh = pix / cv.OW;
            ih0[h] = n_ok ? oh * cv.sh - cv.ph : -(1 << 20);  // a column past N reads nothing
            iw0[h] = (pix - oh * cv.OW) * cv.sw - cv.pw;
            col[h] = g.B + img * g.sB;
        }
        const int khw = cv.KH * cv.KW;
        const int kb = kc * kKc;
        int c = kb / khw;
        int kh = (kb - c * khw) / cv.KW;
        int kw = kb - c * khw - kh * cv.KW;
#pragma unroll 4
        for (int r = 0; r < kKc; ++r) {
            const bool k_ok = kb + r < g.K;
            const int dy = kh * cv.dh, dx = kw * cv.dw;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ih = ih0[h] + dy, iw = iw0[h] + dx;
                const bool ok = k_ok && static_cast<unsigned>(ih) < static_cast<unsigned>(cv.H) &&
                                static_cast<unsigned>(iw) < static_cast<unsigned>(cv.W);
                const float *src = ok ? col[h] + (static_cast<long long>(c) * cv.H + ih) * cv.W + iw : g.B;
                const bool in = ok && SG_IN_B(g, src, 1);
                cp_async4(dst + static_cast<uint32_t>((r * kCols + tid + h * kThreads) * 4), in ? src : g.B,
                          in ? 4u : 0u);
            }
            if (++kw == cv.KW) {
                kw = 0;
                if (++kh == cv.KH) {
                    kh = 0;
                    ++c;
                }
            }
        }
    } else if (vec_b) {
#pragma unroll
        for (int i = 0; i < kKc * kCols / 4 / kThreads; ++i) {
            const int c = tid + i * kThreads;
            const int r = c / (kCols / 4), cc = c % (kCols / 4);
            const int k = kc * kKc + r, n = n0 + cc * 4;
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
            cp_async16(dst + static_cast<uint32_t>((r * kCols + cc * 4) * 4), src, bytes);
        }
    } else {
#pragma unroll 4
        for (int i = 0; i < kKc * kCols / kThreads; ++i) {
            const int c = tid + i * kThreads;
            const int r = c / kCols, cc = c % kCols;
            const int k = kc * kKc + r, n = n0 + cc;
            const bool ok = k < g.K && n < g.N && SG_IN_B(g, g.B + static_cast<long long>(k) * g.ldb + n, 1);
            const float *src = ok ? g.B + static_cast<long long>(k) * g.ldb + n : g.B;
            cp_async4(dst + static_cast<uint32_t>((r * kCols + cc) * 4), src, ok ? 4u : 0u);
        }
    }
}

// C[m][n], C[m][n + 1] for the rows m < M of this thread's two columns.
// CONV: column n is pixel n % ldc of image n / ldc, whose output starts
// sC floats after the previous image's.
template <int CONV>
__device__ __forceinline__ void store_block(const GemmArgs &g, int n, const uint64_t (&acc0)[16],
                                            const uint64_t (&acc1)[16]) {
    if (n >= g.N) return;
    if constexpr (CONV != kConvNone) {
        const int ld = static_cast<int>(g.ldc);
        float *cp[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int nn = min(n + h, g.N - 1);
            const int img = nn / ld;
            cp[h] = g.C + img * g.sC + (nn - img * ld);
        }
        const bool two = n + 1 < g.N;
        const bool read_c = g.beta != 0.f;
#pragma unroll
        for (int mp = 0; mp < kMaxM / 2; ++mp) {
            float c0[2], c1[2];
            pair_split(acc0[mp], c0[0], c0[1]);
            pair_split(acc1[mp], c1[0], c1[1]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int m = 2 * mp + h;
                if (m >= g.M) break;
                float *p0 = cp[0] + static_cast<long long>(m) * ld;
                float *p1 = cp[1] + static_cast<long long>(m) * ld;
                if (SG_IN_C(g, p0, 1)) p0[0] = read_c ? fmaf(g.beta, p0[0], g.alpha * c0[h]) : g.alpha * c0[h];
                if (two && SG_IN_C(g, p1, 1)) p1[0] = read_c ? fmaf(g.beta, p1[0], g.alpha * c1[h]) : g.alpha * c1[h];
            }
        }
        return;
    }
    const bool pair = ((reinterpret_cast<uintptr_t>(g.C) & 7u) == 0) && ((g.ldc & 1) == 0) && n + 1 < g.N;
    const bool read_c = g.beta != 0.f;
#pragma unroll
    for (int mp = 0; mp < kMaxM / 2; ++mp) {
        float c0[2], c1[2];  // (row 2mp, row 2mp + 1) of column n and of column n + 1
        pair_split(acc0[mp], c0[0], c0[1]);
        pair_split(acc1[mp], c1[0], c1[1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int m = 2 * mp + h;
            if (m >= g.M) break;
            float *p = g.C + static_cast<long long>(m) * g.ldc + n;
            float r0 = g.alpha * c0[h], r1 = g.alpha * c1[h];
            if (!SG_IN_C(g, p, (pair || n + 1 < g.N) ? 2 : 1)) continue;
            if (pair) {
                if (read_c) {
                    const float2 o = *reinterpret_cast<const float2 *>(p);
                    r0 = fmaf(g.beta, o.x, r0);
                    r1 = fmaf(g.beta, o.y, r1);
                }
                *reinterpret_cast<float2 *>(p) = make_float2(r0, r1);
            } else {
                p[0] = read_c ? fmaf(g.beta, p[0], r0) : r0;
                if (n + 1 < g.N) p[1] = read_c ? fmaf(g.beta, p[1], r1) : r1;
            }
        }
    }
}

template <int CONV>
__global__ void __launch_bounds__(kThreads, 2) ffma_wide_kernel(const __grid_constant__ GemmArgs g, int vec_b) {
    extern __shared__ __align__(16) float smem_w[];
    const int tid = threadIdx.x;
    const uint32_t s0 = smem_u32(smem_w);
    const uint32_t sA = s0 + static_cast<uint32_t>(kStages * kStageFloats * 4);
    float *a_t = smem_w + kStages * kStageFloats;
    int *tab = reinterpret_cast<int *>(a_t + kAFloats);  // tap offsets (kConvTapsDense)

    const int KC = (g.K + kKc - 1) / kKc;
    const int nblk = (g.N + kCols - 1) / kCols;
    const int mine = nblk > static_cast<int>(blockIdx.x)
                         ? (nblk - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                               static_cast<int>(gridDim.x)
                         : 0;
    const int jobs = mine * KC;  // slabs of this CTA, block-major
    auto issue = [&](int q) {
        if (q < jobs)
            load_slab<CONV>(g, vec_b != 0, static_cast<int>(blockIdx.x) + (q / KC) * static_cast<int>(gridDim.x), q % KC,
                      s0 + static_cast<uint32_t>((q % kStages) * kStageFloats * 4), tid, tab);
        cp_async_commit();
    };
    if constexpr (CONV == kConvTapsDense) {  // tap offsets, needed by the first slab copies
        const ConvGeom &cv = g.cv;
        const int khw = cv.KH * cv.KW;
        for (int k = tid; k < kMaxK; k += kThreads) {
            const int c = k / khw, r = k - c * khw, kh = r / cv.KW, kw = r - kh * cv.KW;
            tab[k] = k < g.K ? (c * cv.H + kh * cv.dh) * cv.W + kw * cv.dw : 0;
        }
        __syncthreads();
    }
#pragma unroll
    for (int q = 0; q < kStages - 1; ++q) issue(q);

    // A^T, zero outside M x K (its loads overlap the first slab copies)
    for (int i = tid; i < kAFloats; i += kThreads) {
        const int k = i / kMaxM, m = i % kMaxM;
        const float *pa = g.A + static_cast<long long>(m) * g.lda + k;
        a_t[i] = (m < g.M && k < g.K && SG_IN_A(g, pa, 1)) ? *pa : 0.f;
    }

    uint64_t acc0[kMaxM / 2], acc1[kMaxM / 2];  // row pairs of columns 2t and 2t + 1
#pragma unroll
    for (int mp = 0; mp < kMaxM / 2; ++mp) acc0[mp] = acc1[mp] = 0ull;

    int q = 0;
#pragma unroll 1
    for (int bi = 0; bi < mine; ++bi) {
#pragma unroll 1
        for (int kc = 0; kc < KC; ++kc, ++q) {
            cp_async_wait<kStages - 2>();
            __syncthreads();  // slab q landed for all threads; slab q - 1's stage is free (and A^T is staged)
            issue(q + kStages - 1);
            const uint32_t st = s0 + static_cast<uint32_t>((q % kStages) * kStageFloats * 4);
            const int kn = min(kKc, g.K - kc * kKc);  // rows of this slab inside K
#pragma unroll 2
            for (int kk = 0; kk < kn; ++kk) {
                float bx, by;
                lds2f(st + static_cast<uint32_t>((kk * kCols + 2 * tid) * 4), bx, by);
                const uint32_t arow = sA + static_cast<uint32_t>((kc * kKc + kk) * kMaxM * 4);
                const uint64_t b0 = pair_bcast(bx), b1 = pair_bcast(by);
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // rows 16h .. 16h + 15: 8 A pairs live at a time
                    uint64_t a[kMaxM / 4];
#pragma unroll
                    for (int p = 0; p < kMaxM / 8; ++p) lds_pairs(arow + h * 64 + p * 16, a[2 * p], a[2 * p + 1]);
#pragma unroll
                    for (int i = 0; i < kMaxM / 4; ++i) {
                        ffma2(acc0[h * 8 + i], a[i], b0);
                        ffma2(acc1[h * 8 + i], a[i], b1);
                    }
                }
            }
        }
        const int cb = static_cast<int>(blockIdx.x) + bi * static_cast<int>(gridDim.x);
        store_block<CONV>(g, cb * kCols + 2 * tid, acc0, acc1);
#pragma unroll
        for (int mp = 0; mp < kMaxM / 2; ++mp) acc0[mp] = acc1[mp] = 0ull;
    }
    cp_async_wait<0>();
}

// Bulk-copy form (B's rows and N 16-byte aligned, no convolution): one CTA
// per SM with 8 compute warps and one loader warp.  The loader copies each
// slab row (up to 2 KB of one B row) with a 1-D cp.async.bulk into a ring
// of kBulkStages slabs with full/empty mbarriers, up to three blocks ahead
// of the compute warps, which only wait, multiply and store C.  In the
// cp.async form every thread issues its own copies between its FMAs and
// the CTA's loads, FMAs and C stores took turns (measured on GB300 at
// 32 x 1605632 x 27: loads and stores alone 74 us, with the FMAs 103 us).
// The arithmetic is the cp.async form's, in the same order.
constexpr int kBulkStages = 6;
constexpr int kBulkThreads = kThreads + 32;  // + the loader warp
constexpr int kBulkBarBytes = 16 * kBulkStages + 16;
constexpr int kBulkSmemBytes = (kBulkStages * kStageFloats + kAFloats) * 4 + kBulkBarBytes;

__global__ void __launch_bounds__(kBulkThreads, 1)
    ffma_wide_bulk_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ DeviceCtl ctl) {
    extern __shared__ __align__(16) float smem_w[];
    const int tid = threadIdx.x;
    const uint32_t s0 = smem_u32(smem_w);
    float *a_t = smem_w + kBulkStages * kStageFloats;
    const uint32_t sA = smem_u32(a_t);
    const uint32_t bars = sA + kAFloats * 4;  // full[s] at bars + 8 s, empty[s] at bars + 8 (S + s)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(a_t + kAFloats + 4 * kBulkStages);
    constexpr int S = kBulkStages;

    const int KC = (g.K + kKc - 1) / kKc;
    const int nblk = (g.N + kCols - 1) / kCols;
    const int mine = nblk > static_cast<int>(blockIdx.x)
                         ? (nblk - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                               static_cast<int>(gridDim.x)
                         : 0;
    const int jobs = mine * KC;  // slabs of this CTA, block-major
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bars + 8u * s, 1);                      // full: the loader's expect_tx arrive
            mbar_init(bars + 8u * (S + s), kThreads / 32);    // empty: one arrive per compute warp
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    // A^T, zero outside M x K
    for (int i = tid; i < kAFloats; i += kBulkThreads) {
        const int k = i / kMaxM, m = i % kMaxM;
        const float *pa = g.A + static_cast<long long>(m) * g.lda + k;
        a_t[i] = (m < g.M && k < g.K && SG_IN_A(g, pa, 1)) ? *pa : 0.f;
    }
    __syncthreads();

    if (tid >= kThreads) {
        // ---------------------------------------------------- loader
        if (tid == kThreads) {
            int s = 0;
            uint32_t ph = 0, used = 0, last_ph = 0;
#pragma unroll 1
            for (int q = 0; q < jobs; ++q) {
                if (!mbar_wait_bounded(bars + 8u * (S + s), ph ^ 1u, abort_flag, ctl, kStatusTimeoutProducer)) break;
                const int cb = static_cast<int>(blockIdx.x) + (q / KC) * static_cast<int>(gridDim.x);
                const int kc = q % KC;
                const int n0 = cb * kCols;
                const uint32_t bytes = static_cast<uint32_t>(min(kCols, g.N - n0) * 4);
                const int rows = min(kKc, g.K - kc * kKc);
                mbar_arrive_expect_tx(bars + 8u * s, bytes * static_cast<uint32_t>(rows));
                const uint32_t dst = s0 + static_cast<uint32_t>(s * kStageFloats * 4);
#pragma unroll 1
                for (int r = 0; r < rows; ++r) {
                    const float *src = g.B + static_cast<long long>(kc * kKc + r) * g.ldb + n0;
                    // SGEMM_DEBUG: a row outside B is not copied (the wait then runs out)
                    if (SG_IN_B(g, src, static_cast<int>(bytes / 4)))
                        bulk_load_1d(dst + static_cast<uint32_t>(r * kCols * 4), src, bytes, bars + 8u * s);
                }
                used |= 1u << s;
                last_ph = (last_ph & ~(1u << s)) | (ph << s);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // every copy issued has landed before the CTA can exit
            volatile int no_abort = 0;
            for (int t = 0; t < S; ++t)
                if (used & (1u << t))
                    mbar_wait_bounded(bars + 8u * t, (last_ph >> t) & 1u, &no_abort, ctl, kStatusTimeoutDrain);
        }
        return;
    }

    // -------------------------------------------------------- compute
    uint64_t acc0[kMaxM / 2], acc1[kMaxM / 2];  // row pairs of columns 2t and 2t + 1
#pragma unroll
    for (int mp = 0; mp < kMaxM / 2; ++mp) acc0[mp] = acc1[mp] = 0ull;
    int s = 0;
    uint32_t ph = 0;
    const int lane = tid & 31;
#pragma unroll 1
    for (int bi = 0; bi < mine; ++bi) {
        bool ok = true;
#pragma unroll 1
        for (int kc = 0; kc < KC; ++kc) {
            if (!mbar_wait_bounded(bars + 8u * s, ph, abort_flag, ctl, kStatusTimeoutMma)) {
                ok = false;
                break;
            }
            const uint32_t st = s0 + static_cast<uint32_t>(s * kStageFloats * 4);
            const int kn = min(kKc, g.K - kc * kKc);  // rows of this slab inside K
#pragma unroll 2
            for (int kk = 0; kk < kn; ++kk) {
                float bx, by;
                lds2f(st + static_cast<uint32_t>((kk * kCols + 2 * tid) * 4), bx, by);
                const uint32_t arow = sA + static_cast<uint32_t>((kc * kKc + kk) * kMaxM * 4);
                const uint64_t b0 = pair_bcast(bx), b1 = pair_bcast(by);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint64_t a[kMaxM / 4];
#pragma unroll
                    for (int p = 0; p < kMaxM / 8; ++p) lds_pairs(arow + h * 64 + p * 16, a[2 * p], a[2 * p + 1]);
#pragma unroll
                    for (int i = 0; i < kMaxM / 4; ++i) {
                        ffma2(acc0[h * 8 + i], a[i], b0);
                        ffma2(acc1[h * 8 + i], a[i], b1);
                    }
                }
            }
            // this warp is done with the slab: the loader may refill it
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8u * (S + s));
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (!ok) break;
        const int cb = static_cast<int>(blockIdx.x) + bi * static_cast<int>(gridDim.x);
        store_block<kConvNone>(g, cb * kCols + 2 * tid, acc0, acc1);
#pragma unroll
        for (int mp = 0; mp < kMaxM / 2; ++mp) acc0[mp] = acc1[mp] = 0ull;
    }
}

}  // namespace wide

bool ffma_wide_bulk(const GemmArgs &g, int vec_b) { return vec_b && g.N % 4 == 0; }

bool ffma_wide_fits(int M, int K) { return M >= 1 && M <= wide::kMaxM && K >= 1 && K <= wide::kMaxK; }

int ffma_wide_blocks(int N) { return (N + wide::kCols - 1) / wide::kCols; }

int ffma_wide_smem_bytes() { return wide::kSmemBytes; }

cudaError_t ffma_wide_launch(const GemmArgs &g, int vec_b, int grid, cudaStream_t stream, int conv,
                             const DeviceCtl *ctl) {
    if (conv == kConvNone && ctl != nullptr && ffma_wide_bulk(g, vec_b)) {
        // one CTA per SM (the caller's grid counts two per SM for the cp.async form)
        cudaError_t e = cudaFuncSetAttribute(wide::ffma_wide_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             wide::kBulkSmemBytes);
        if (e != cudaSuccess) return e;
        wide::ffma_wide_bulk_kernel<<<grid, wide::kBulkThreads, wide::kBulkSmemBytes, stream>>>(g, *ctl);
        return cudaGetLastError();
    }
    auto kern = conv == kConvTapsDense ? wide::ffma_wide_kernel<kConvTapsDense>
                : conv == kConvTaps    ? wide::ffma_wide_kernel<kConvTaps>
                                       : wide::ffma_wide_kernel<kConvNone>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, wide::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<grid, wide::kThreads, wide::kSmemBytes, stream>>>(g, vec_b);
    return cudaGetLastError();
}

}  // namespace sg
