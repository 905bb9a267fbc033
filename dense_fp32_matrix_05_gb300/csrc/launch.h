// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cuda_runtime.h>

#include "common.cuh"

namespace sg {

// Tile constants the planner needs (checked against the kernels' own).
constexpr int kTf32x3TileN = 128;  // C columns per 3xTF32 tile
constexpr int kTf32x3BK = 16;      // K per 3xTF32 pipeline stage
constexpr int kFfmaBK = 16;        // K per FFMA pipeline stage

// 3xTF32 tensor-core path.  tm = C rows per tile: 16, 32, 64, 128, 192, 256.
bool tf32x3_supported_tm(int tm);
int tf32x3_stages(int tm);
int tf32x3_smem_bytes(int tm);
cudaError_t tf32x3_launch(int tm, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl,
                          int vec_a, int grid, cudaStream_t stream);

// FFMA path.  (bm, bn) in {(128,128), (64,256), (32,512)}.
bool ffma_supported_tile(int bm, int bn);
int ffma_stages(int bm, int bn);
int ffma_smem_bytes(int bm, int bn);
cudaError_t ffma_launch(int bm, int bn, const GemmArgs &g, const Schedule &s, const DeviceCtl &ctl,
                        int vec_a, int vec_b, int vec_c, cudaStream_t stream);

// C = beta * C (alpha == 0 or K == 0).
cudaError_t scale_c_launch(float *C, long long ldc, int M, int N, float beta, int num_sms,
                           cudaStream_t stream);

}  // namespace sg
