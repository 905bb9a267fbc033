// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace sg {

// Launch with programmatic stream serialization: the kernel may begin while
// the kernel ahead of it in the stream is finishing, so its on-chip set-up
// overlaps that kernel's tail.  Only for kernels that call grid_dep_wait()
// before their first global-memory access (the 3xTF32 kernel).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Same, in clusters of two CTAs along x (grid even): the CTA pairs of the
// 3xTF32 kernel's cta_group::2 form.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_pairs(void (*kern)(KArgs...), int grid, int threads, int smem, cudaStream_t stream,
                             Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Extents of a GEMM's operands for the SGEMM_DEBUG bounds checks: one past
// the last float of A (M x K), B (K x N, or N x K when transposed) and C
// (M x N) over `batch` matrices with the strides in g; dbg_status is where
// violations are reported.
inline void set_extents(GemmArgs &g, int batch, bool trans_b, int *status) {
    const long long nb = batch > 1 ? batch - 1 : 0;
    g.a_end = (g.A && g.M > 0 && g.K > 0) ? g.A + nb * g.sA + (g.M - 1) * g.lda + g.K : nullptr;
    g.b_end = (g.B && g.N > 0 && g.K > 0)
                  ? g.B + nb * g.sB + (trans_b ? (g.N - 1) * g.ldb + g.K : (g.K - 1) * g.ldb + g.N)
                  : nullptr;
    g.c_end = (g.C && g.M > 0 && g.N > 0) ? g.C + nb * g.sC + (g.M - 1) * g.ldc + g.N : nullptr;
    g.dbg_status = status;
}

// Tile constants the planner needs (checked against the kernels' own).
constexpr int kTf32x3TileN = 128;  // C columns per 3xTF32 tile
constexpr int kTf32x3BK = 16;      // K per 3xTF32 pipeline stage
constexpr int kTf32x3MaxDefer = 8;  // shared (split-K) tiles one 3xTF32 CTA may finish
constexpr int kFfmaBK = 16;        // K per FFMA pipeline stage

// 3xTF32 tensor-core path.  tm = C rows per tile: 16, 32, 64, 128, 192, 256.
bool tf32x3_supported_tm(int tm);
int tf32x3_stages(int tm, bool pair = false);
int tf32x3_smem_bytes(int tm);
// CTA pairs (clusters of two sharing a cta_group::2 MMA; tiles of 192 or 256
// rows x 256 columns, s.pair_shift = 1, grid = 2 x pairs): whether tm has the
// form, and how many pairs the device holds at once (0 if none, or on error).
bool tf32x3_pair_tm(int tm);
int tf32x3_pair_slots();
// B stored transposed (N x K, row stride g.ldb; BLAS transb): the 3xTF32
// kernel copies B^T slabs by TMA and reads them column by column, with no
// transpose pass.  A's and B's rows (and batch strides) must be 16-byte
// aligned; cudaErrorNotSupported if a tensor map cannot be made.
cudaError_t tf32x3_launch_tb(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int vec_a,
                             int vec_c, int grid, cudaStream_t stream, int batch);

// Implicit-GEMM convolution (g.cv; B = the NCHW input, batch = images;
// order: kConvTaps or kConvChannels; g.A: the filter in that k order with
// 16-byte aligned rows).
cudaError_t tf32x3_conv_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl, int order,
                               int vec_c, int grid, cudaStream_t stream, int batch);
// planes H x W of x copied into (H + 2 ph) x (W + 2 pw) planes with zero borders.
cudaError_t pad_planes_launch(const float *x, long long planes, int H, int W, int ph, int pw, float *xp,
                              cudaStream_t stream);
// OIHW filter w (F x C x KH x KW) to OHWI rows of leading dimension ld.
cudaError_t filter_ohwi_launch(const float *w, int F, int C, int KH, int KW, float *dst, long long ld,
                               cudaStream_t stream);

// batch: matrices of a strided batch (g.sA / sB / sC; s.tpb tiles each).
// b_rows: a B whose rows are not 16-byte aligned is loaded by the producers
// instead of being copied by TMA as four residue classes of rows.
cudaError_t tf32x3_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl,
                          int vec_a, int vec_b, int vec_c, int grid, cudaStream_t stream, int batch = 1,
                          bool b_rows = false);

// FFMA path.  (bm, bn) in {(128,128), (64,256), (32,512)}.
bool ffma_supported_tile(int bm, int bn);
int ffma_stages(int bm, int bn);
int ffma_smem_bytes(int bm, int bn);
cudaError_t ffma_launch(int bm, int bn, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl,
                        int vec_a, int vec_b, int vec_c, cudaStream_t stream);

// Planner and argument checks of the 3xTF32 path, for entry points defined
// outside api.cu (noalloc.cu).  check_tensor_call makes no CUDA call.
struct TensorPlan {
    int tile_m = 0;
    Schedule sch{};
    int grid = 0;
    int vec_a = 0;
    int vec_b = 0;
    int vec_c = 0;
    size_t ws_floats = 0;  // split-K partial-tile floats needed (0 without split-K)
    int tiles = 0;         // arrival counters needed (one per tile; two per tile of a CTA pair)
};
int check_tensor_call(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                      float beta, const float *C, int ldc, int splits);
// pair_slots: CTA pairs the device holds at once (tf32x3_pair_slots; 0: none).
int plan_tensor_call(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float beta,
                     const float *C, int ldc, int splits, int sms, int pair_slots, size_t max_ws_floats,
                     TensorPlan *out);
// Read and clear sgemm_noalloc's status word on the current device (after
// the caller has waited for its stream).  Returns 0 when the word is clear
// or sgemm_noalloc has not been set up on this device, 1 when it was set
// (the word and sgemm_noalloc's arrival counters are then cleared, after a
// device-wide wait), or -e for a failed CUDA call returning e.
int noalloc_take_status();
// Load the device code of every kernel sgemm_noalloc can launch (with lazy
// module loading, a kernel's code is otherwise loaded, and device memory
// taken for it, at its first launch).
cudaError_t tf32x3_preload();
cudaError_t scale_c_preload();

// Wide-N FFMA kernel for M <= 32, K <= 64 (A resident, B streamed):
// persistent CTAs over blocks of 512 columns.
bool ffma_wide_fits(int M, int K);
int ffma_wide_blocks(int N);
int ffma_wide_smem_bytes();
// conv: kConvNone, or the implicit-GEMM convolution form kConvTaps /
// kConvTapsDense (g.cv; N = images * ldc pixels).
// With ctl given, a plain GEMM whose B rows and N are 16-byte aligned runs
// the bulk-copy form (ffma_wide_bulk; one CTA per SM: grid <= SMs).
cudaError_t ffma_wide_launch(const GemmArgs &g, int vec_b, int grid, cudaStream_t stream, int conv = kConvNone,
                             const DeviceCtl *ctl = nullptr);
bool ffma_wide_bulk(const GemmArgs &g, int vec_b);

// dst (cols x rows, leading dimension ldd) = transpose of src (rows x cols,
// leading dimension lds); row-major fp32.  count matrices, src_stride /
// dst_stride elements apart.
cudaError_t transpose_launch(const float *src, long long lds, int rows, int cols, float *dst, long long ldd,
                             cudaStream_t stream, int count = 1, long long src_stride = 0,
                             long long dst_stride = 0);

// C = beta * C (alpha == 0 or K == 0).
cudaError_t scale_c_launch(float *C, long long ldc, int M, int N, float beta, int num_sms,
                           cudaStream_t stream);

}  // namespace sg
