// Instantiations and launcher of the 3xTF32 tensor-core kernel, including
// the TMA tensor map for A (built on the host with the driver's
// cuTensorMapEncodeTiled, reached through the runtime's entry-point query so
// that the library needs no link-time dependency on the driver).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "launch.h"
#include "tf32x3_gemm.cuh"
#include "tmap.h"

namespace sg {

static_assert(kTf32x3TileN == tf32x3::kTileN && kTf32x3BK == tf32x3::kBK &&
                  kTf32x3MaxDefer == tf32x3::kMaxDefer,
              "planner constants");

namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode;
}

}  // namespace

// SGEMM_DEBUG: a tensor map that could address bytes outside its operand
// ([lo, hi)) is not made, and the launch fails with cudaErrorInvalidValue
// (map_range_error tells the launchers).
thread_local bool t_map_range_error = false;

bool map_in(const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides, const void *lo,
            const void *hi) {
    if (!kDebugBounds) return true;
    unsigned long long last = (dims[0] - 1) * sizeof(float);
    for (int i = 1; i < rank; ++i) last += (dims[i] - 1) * strides[i - 1];
    const char *b = static_cast<const char *>(base);
    const bool ok = lo != nullptr && hi != nullptr && b >= static_cast<const char *>(lo) &&
                    b + last + sizeof(float) <= static_cast<const char *>(hi);
    if (!ok) t_map_range_error = true;
    return ok;
}

bool map_range_error() {
    const bool e = t_map_range_error;
    t_map_range_error = false;
    return e;
}

// Third (batch) dimension of a tensor map: `batch` matrices `stride`
// elements apart, or one matrix when the stride is 0 (an operand shared by
// the batch, or no batch).  The stride must be a multiple of 16 bytes.
static bool batch_dim(long long stride, int batch, long long one_matrix_elems, cuuint64_t &dim, cuuint64_t &bytes) {
    if (stride == 0 || batch <= 1) {
        dim = 1;
        bytes = (static_cast<cuuint64_t>(one_matrix_elems) * sizeof(float) + 15) & ~cuuint64_t(15);
        return true;
    }
    if ((stride * sizeof(float)) % 16 != 0) return false;
    dim = static_cast<cuuint64_t>(batch);
    bytes = static_cast<cuuint64_t>(stride) * sizeof(float);
    return true;
}

// Tensor map of A for the TMA path: a K x M fp32 tensor (K innermost) with
// row stride lda * 4 bytes, copied in boxes of 16 (k) x tm (rows) with the
// 64-byte swizzle, out-of-range elements filled with zeros.  Requires A and
// lda * 4 to be multiples of 16 bytes.  Returns false when no map can be made.
bool make_tmap_a(const GemmArgs &g, int tm, int batch, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t nb, sb;
    if (!batch_dim(g.sA, batch, g.lda * g.M, nb, sb)) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.K), static_cast<cuuint64_t>(g.M), nb};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.lda) * sizeof(float), sb};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(tf32x3::kBK), static_cast<cuuint32_t>(tm), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (!map_in(g.A, 3, dims, strides, g.A, g.a_end)) return false;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(g.A), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map of B for the TMA path of narrow tiles: a N x K fp32 tensor (N
// innermost) with row stride ldb * 4 bytes, copied in boxes of 128 (n) x 16
// (k) without swizzle, out-of-range elements filled with zeros.
bool make_tmap_b(const GemmArgs &g, int batch, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t nb, sb;
    if (!batch_dim(g.sB, batch, g.ldb * g.K, nb, sb)) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.N), static_cast<cuuint64_t>(g.K), nb};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.ldb) * sizeof(float), sb};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(tf32x3::kTileN), static_cast<cuuint32_t>(tf32x3::kBK), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (!map_in(g.B, 3, dims, strides, g.B, g.b_end)) return false;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(g.B), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map of C for the TMA epilogue: a N x M fp32 tensor (N innermost)
// with row stride ldc * 4 bytes, copied in and out in boxes of 128 (n) x 16
// (rows) without swizzle; loads fill out-of-range elements with zeros and
// stores skip them.
// Tensor map of a transposed B (stored N x K, k innermost, row stride ldb):
// a K x N tensor copied in boxes of 16 (k) x 128 (n) with the 64-byte
// swizzle, so that each n row of the slab is one swizzled 64-byte row.
bool make_tmap_bt(const GemmArgs &g, int batch, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    cuuint64_t nb, sb;
    if (!batch_dim(g.sB, batch, g.ldb * g.N, nb, sb)) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.K), static_cast<cuuint64_t>(g.N), nb};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.ldb) * sizeof(float), sb};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(tf32x3::kBK), static_cast<cuuint32_t>(tf32x3::kTileN), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (!map_in(g.B, 3, dims, strides, g.B, g.b_end)) return false;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(g.B), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor maps of a B whose rows are not 16-byte aligned (ldb % 4 != 0),
// one per residue class r = k % 4: rows r, r + 4, r + 8, ... are 4 * ldb
// floats apart (a multiple of 16 bytes).  Class r starts at B + r * ldb -
// o_r, rounded down to a 16-byte boundary (o_r = (r * ldb) % 4), and is
// N + o_r floats wide, so its rows' columns 0..N-1 sit o_r floats into the
// box of 132 x 4 (columns x rows of the class) copied without swizzle;
// out-of-range elements read as zero.  Needs a 16-byte aligned B (so the
// leading floats of a row are the tail of the row before it, inside B),
// K >= 4 (every class has a row) and a batch stride that is a multiple of 4
// floats.  *offs packs o_r in bits 2r..2r+1.
bool make_tmap_b4(const GemmArgs &g, int batch, CUtensorMap maps[4], uint32_t *offs) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    if ((reinterpret_cast<uintptr_t>(g.B) & 15u) != 0 || g.K < 4 || (g.sB & 3) != 0) return false;
    cuuint64_t nb, sb;
    if (!batch_dim(g.sB, batch, g.ldb * g.K, nb, sb)) return false;
    *offs = 0;
    for (int r = 0; r < 4; ++r) {
        const long long o = (static_cast<long long>(r) * g.ldb) & 3;
        const float *base = g.B + static_cast<long long>(r) * g.ldb - o;
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.N + o), static_cast<cuuint64_t>((g.K - r + 3) / 4), nb};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(4 * g.ldb) * sizeof(float), sb};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(tf32x3::kB4Row), 4, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (!map_in(base, 3, dims, strides, g.B, g.b_end)) return false;
        const CUresult res = enc(&maps[r], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), dims,
                                 strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (res != CUDA_SUCCESS) return false;
        *offs |= static_cast<uint32_t>(o) << (2 * r);
    }
    return true;
}

bool make_tmap_c(const GemmArgs &g, int batch, CUtensorMap *map) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    // A TMA store writes whole 16-byte units at the end of a row: with N not
    // a multiple of 4 it would write the first floats of the ld padding
    // (measured on GB300: N = 15, ldc = 20).  Such a C takes the epilogue's
    // own stores.
    if (g.N % 4 != 0) return false;
    cuuint64_t nb, sb;
    if (!batch_dim(g.sC, batch, g.ldc * g.M, nb, sb)) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.N), static_cast<cuuint64_t>(g.M), nb};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.ldc) * sizeof(float), sb};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(tf32x3::kTileN), static_cast<cuuint32_t>(tf32x3::kEpiRows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (!map_in(g.C, 3, dims, strides, g.C, g.c_end)) return false;
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, g.C, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

namespace {

template <int TM, bool TA, bool TB, bool B4 = false, bool PAIR = false>
cudaError_t launch_tm(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int tma_c, int grid,
                      const CUtensorMap &map_a, const CUtensorMap (&map_b)[4], uint32_t b_offs,
                      const CUtensorMap &map_c, cudaStream_t stream) {
    using C = tf32x3::Cfg<TM, TB, B4, PAIR>;
    auto kern = tf32x3::tf32x3_gemm_kernel<TM, TA, TB, kConvNone, false, B4, PAIR>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if constexpr (PAIR)
        return launch_pdl_pairs(kern, grid, tf32x3::Roles<TM, TA, TB>::kThreads, C::kSmemBytes, stream, g, s, ctl,
                                vec_a, tma_c, b_offs, map_a, map_b[0], map_c, map_b[1], map_b[2], map_b[3]);
    else
        return launch_pdl(kern, grid, tf32x3::Roles<TM, TA, TB>::kThreads, C::kSmemBytes, stream, g, s, ctl, vec_a,
                          tma_c, b_offs, map_a, map_b[0], map_c, map_b[1], map_b[2], map_b[3]);
}

// The CTA-pair form (s.pair_shift = 1): A and B copied by TMA (B's rows
// aligned, or as residue classes), A in boxes of TM / 2 rows, one per CTA.
template <int TM>
cudaError_t launch_pairs(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int vec_b,
                         int vec_c, int grid, int batch, bool b_rows, cudaStream_t stream) {
    if constexpr (TM != 192 && TM != 256) {
        return cudaErrorInvalidValue;
    } else {
        CUtensorMap ma, mb[4], mc;
        std::memset(&ma, 0, sizeof(ma));
        std::memset(mb, 0, sizeof(mb));
        std::memset(&mc, 0, sizeof(mc));
        uint32_t offs = 0;
        if (grid % 2 != 0 || !vec_a || !make_tmap_a(g, TM / 2, batch, &ma)) return cudaErrorInvalidValue;
        const bool tb = vec_b && make_tmap_b(g, batch, &mb[0]);
        const bool tb4 = !tb && !vec_b && !b_rows && make_tmap_b4(g, batch, mb, &offs);
        const int tc = (vec_c && make_tmap_c(g, batch, &mc)) ? 1 : 0;
        if (map_range_error()) return cudaErrorInvalidValue;  // SGEMM_DEBUG only
        if (tb) return launch_tm<TM, true, true, false, true>(g, s, ctl, vec_a, tc, grid, ma, mb, 0, mc, stream);
        if (tb4) return launch_tm<TM, true, true, true, true>(g, s, ctl, vec_a, tc, grid, ma, mb, offs, mc, stream);
        return cudaErrorInvalidValue;
    }
}

// Operands go through TMA whenever their rows are 16-byte aligned: the deep
// asynchronous ring hides memory latency and the producers then hold almost
// nothing in registers (the extra shared-memory pass for B^T is cheaper than
// the register spills and load stalls it removes).  A B whose rows are not
// aligned (but whose start is) comes by TMA too, as four residue classes of
// rows.  SGEMM_FLAG_B_ROWS_LOADED (b_rows) keeps such a B on the producers'
// own loads.
template <int TM>
cudaError_t launch_rows(const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a, int vec_b,
                        int vec_c, int grid, int batch, bool b_rows, cudaStream_t stream) {
    if (s.pair_shift) return launch_pairs<TM>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
    CUtensorMap ma, mb[4], mc;
    std::memset(&ma, 0, sizeof(ma));
    std::memset(mb, 0, sizeof(mb));
    std::memset(&mc, 0, sizeof(mc));
    uint32_t offs = 0;
    const bool ta = vec_a && make_tmap_a(g, TM, batch, &ma);
    const bool tb = vec_b && make_tmap_b(g, batch, &mb[0]);
    const bool tb4 = !vec_b && !b_rows && make_tmap_b4(g, batch, mb, &offs);
    const int tc = (vec_c && make_tmap_c(g, batch, &mc)) ? 1 : 0;
    if (map_range_error()) return cudaErrorInvalidValue;  // SGEMM_DEBUG only
    if (tb) {
        if (ta) return launch_tm<TM, true, true>(g, s, ctl, vec_a, tc, grid, ma, mb, 0, mc, stream);
        return launch_tm<TM, false, true>(g, s, ctl, vec_a, tc, grid, ma, mb, 0, mc, stream);
    }
    if (tb4) {
        if (ta) return launch_tm<TM, true, true, true>(g, s, ctl, vec_a, tc, grid, ma, mb, offs, mc, stream);
        return launch_tm<TM, false, true, true>(g, s, ctl, vec_a, tc, grid, ma, mb, offs, mc, stream);
    }
    if (ta) return launch_tm<TM, true, false>(g, s, ctl, vec_a, tc, grid, ma, mb, 0, mc, stream);
    return launch_tm<TM, false, false>(g, s, ctl, vec_a, tc, grid, ma, mb, 0, mc, stream);
}

}  // namespace

namespace {

template <int TM, bool TA, bool TB, bool B4 = false, bool PAIR = false>
cudaError_t preload_one() {
    cudaFuncAttributes attr;
    return cudaFuncGetAttributes(&attr, tf32x3::tf32x3_gemm_kernel<TM, TA, TB, kConvNone, false, B4, PAIR>);
}

template <int TM>
cudaError_t preload_tm() {
    cudaError_t e;
    if ((e = preload_one<TM, false, false>()) != cudaSuccess) return e;
    if ((e = preload_one<TM, false, true>()) != cudaSuccess) return e;
    if ((e = preload_one<TM, true, false>()) != cudaSuccess) return e;
    if ((e = preload_one<TM, false, true, true>()) != cudaSuccess) return e;
    if ((e = preload_one<TM, true, true, true>()) != cudaSuccess) return e;
    return preload_one<TM, true, true>();
}

}  // namespace

cudaError_t tf32x3_preload() {
    cudaError_t e;
    if ((e = preload_tm<16>()) != cudaSuccess) return e;
    if ((e = preload_tm<32>()) != cudaSuccess) return e;
    if ((e = preload_tm<64>()) != cudaSuccess) return e;
    if ((e = preload_tm<128>()) != cudaSuccess) return e;
    if ((e = preload_tm<192>()) != cudaSuccess) return e;
    if ((e = preload_one<192, true, true, false, true>()) != cudaSuccess) return e;
    if ((e = preload_one<192, true, true, true, true>()) != cudaSuccess) return e;
    if ((e = preload_one<256, true, true, false, true>()) != cudaSuccess) return e;
    if ((e = preload_one<256, true, true, true, true>()) != cudaSuccess) return e;
    return preload_tm<256>();
}

bool tf32x3_pair_tm(int tm) { return tm == 192 || tm == 256; }

int tf32x3_pair_slots() {
    // both pair kernels hold one CTA per SM; the larger shared-memory
    // footprint bounds how many clusters of two can be resident
    using C = tf32x3::Cfg<256, true, false, true>;
    auto kern = tf32x3::tf32x3_gemm_kernel<256, true, true, kConvNone, false, false, true>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(tf32x3::Roles<256, true, true>::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

bool tf32x3_supported_tm(int tm) {
    return tm == 16 || tm == 32 || tm == 64 || tm == 128 || tm == 192 || tm == 256;
}

int tf32x3_stages(int tm, bool pair) {
    if (pair) {
        switch (tm) {
            case 192: return tf32x3::Cfg<192, true, false, true>::kStages;
            case 256: return tf32x3::Cfg<256, true, false, true>::kStages;
            default: return 0;
        }
    }
    switch (tm) {  // with B copied by TMA (the usual case)
        case 16: return tf32x3::Cfg<16, true>::kStages;
        case 32: return tf32x3::Cfg<32, true>::kStages;
        case 64: return tf32x3::Cfg<64, true>::kStages;
        case 128: return tf32x3::Cfg<128, true>::kStages;
        case 192: return tf32x3::Cfg<192, true>::kStages;
        case 256: return tf32x3::Cfg<256, true>::kStages;
        default: return 0;
    }
}

int tf32x3_smem_bytes(int tm) {
    switch (tm) {
        case 16: return tf32x3::Cfg<16, true>::kSmemBytes;
        case 32: return tf32x3::Cfg<32, true>::kSmemBytes;
        case 64: return tf32x3::Cfg<64, true>::kSmemBytes;
        case 128: return tf32x3::Cfg<128, true>::kSmemBytes;
        case 192: return tf32x3::Cfg<192, true>::kSmemBytes;
        case 256: return tf32x3::Cfg<256, true>::kSmemBytes;
        default: return -1;
    }
}

cudaError_t tf32x3_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a,
                          int vec_b, int vec_c, int grid, cudaStream_t stream, int batch, bool b_rows) {
    switch (tm) {
        case 16: return launch_rows<16>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
        case 32: return launch_rows<32>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
        case 64: return launch_rows<64>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
        case 128: return launch_rows<128>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
        case 192: return launch_rows<192>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
        case 256: return launch_rows<256>(g, s, ctl, vec_a, vec_b, vec_c, grid, batch, b_rows, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace sg
