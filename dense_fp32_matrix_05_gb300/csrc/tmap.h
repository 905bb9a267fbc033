// Host-side TMA tensor maps of the 3xTF32 kernel's operands (built in
// tf32x3_gemm.cu with the driver's cuTensorMapEncodeTiled).  Each map has a
// third, batch dimension: the matrices of a strided batch, or extent 1.
// A map is made only when the rows and the batch stride are 16-byte
// aligned; false means the operand goes through element loads instead.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace sg {

// A: K x M fp32 (K innermost), box 16 x tm.
bool make_tmap_a(const GemmArgs &g, int tm, int batch, CUtensorMap *map);
// B: N x K fp32 (N innermost), box 128 x 16.
bool make_tmap_b(const GemmArgs &g, int batch, CUtensorMap *map);
// A transposed B (stored N x K, K innermost) as K x N, box 16 x 128,
// 64-byte swizzle.
bool make_tmap_bt(const GemmArgs &g, int batch, CUtensorMap *map);
// B with rows that are not 16-byte aligned: one map per residue class of
// rows k % 4 (box 132 x 4); offs packs each class's leading floats.
bool make_tmap_b4(const GemmArgs &g, int batch, CUtensorMap maps[4], uint32_t *offs);
// C: N x M fp32 (N innermost), box 128 x 16 (one epilogue chunk).
bool make_tmap_c(const GemmArgs &g, int batch, CUtensorMap *map);
// SGEMM_DEBUG builds: whether a map since the last call was refused because
// it could address bytes outside its operand (clears the flag; this thread).
bool map_range_error();

}  // namespace sg
