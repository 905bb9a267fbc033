// SGEMM on the tcgen05 tensor cores with the 3xTF32 split.
//
// Each fp32 operand x is split into hi = x with the low 13 mantissa bits
// cleared (an exact tf32 value) and lo = tf32(x - hi); the product a*b is
// then accumulated as hi_a*hi_b + hi_a*lo_b + lo_a*hi_b (lo_a*lo_b, below
// 2^-20 |a*b|, is dropped) into one fp32 accumulator in tensor memory.
//
// The kernel computes each C tile transposed: the MMA's M dimension (128
// tensor-memory lanes) runs over C columns n and its N dimension over C rows
// m, so D[n][m] = sum_k B[k][n] * A[m][k].  The epilogue then reads one C
// column per thread and, for each row, a warp stores 32 consecutive floats:
// coalesced for any ldc, including odd row lengths such as N = 14161.
//
// Roles (one persistent CTA per SM, work units strided over the grid):
//   warps 0-3   epilogue: tensor memory -> alpha/beta -> C (or split-K
//               partials); warp w owns tensor-memory lanes 32w..32w+31
//   warps 4..    producers (12 warps in 3 groups when A comes by TMA, else
//               16): the B slab (MMA A operand B^T) -> hi/lo split -> a
//               tensor-memory ring (tcgen05.st), read either from the raw
//               slab a TMA copy left in shared memory (B rows 16-byte
//               aligned) or from their own global loads (any alignment,
//               zero-filled edges, several stages in flight); the A tile
//               (MMA B operand) -> hi/lo in K-major 64-byte-swizzled shared
//               memory: after a TMA copy (A rows 16-byte aligned) the raw
//               tile is the hi operand and only lo is written; otherwise
//               both come from the producers' own loads
//   next warp   tensor-memory allocation and the single MMA-issuing thread
//   last warp   the TMA thread: copies raw A tiles and B slabs into the ring
// Keeping the 128-row operand in tensor memory halves the shared-memory
// traffic per MMA (the tensor core reads only the A tile from shared memory).
// Pipelines: a STAGES-deep ring (full/empty mbarriers; the tensor core frees
// a stage through tcgen05.commit) and one or two accumulators in tensor
// memory (acc_full/acc_empty; with two, a tile's epilogue overlaps the next
// tile's main loop).  Every wait is bounded (see mbar_wait_bounded).
// Launched with programmatic stream serialization: barrier set-up and the
// tensor-memory allocation may run while the previous kernel on the stream
// finishes; griddepcontrol.wait comes before the first global access.
// CTA pairs (PAIR): tiles of 256 columns are shared by the two CTAs of a
// cluster through one cta_group::2 MMA per product and k slice (each CTA
// keeps its 128 columns of B^T and of the accumulator and half the A rows);
// the roles are the same, and the even CTA's MMA thread issues for both.
//
// Operand staging follows the shared-memory tiling, vector-load and
// prefetch ideas of "NVIDIA_SGEMM_PRACTICE" (sections "kernel 2", "kernel 6",
// "kernel 7") and the zero-filled edge tiles of "matmul_opt.cu"
// (matrixMulOptimized), re-done for the tensor core: every element has to
// pass a producer thread for the split, so B^T goes (TMA ->) registers ->
// tensor memory, and A (TMA ->) shared memory, with lo written beside it.
#pragma once
#include <cuda.h>  // CUtensorMap (type only; the library does not link the driver)

#include <cstdint>

#include "common.cuh"

namespace sg {
namespace tf32x3 {

constexpr int kTileN = 128;  // C columns per tile (MMA M, tensor-memory lanes)
constexpr int kBK = 16;      // K per stage: one 64-byte swizzled row per operand row
constexpr int kEpiWarps = 4;
constexpr int kEpiBarrierId = 1;

// Warp roles.  The producer warps form kGroups groups; group g fills the
// k tiles (jobs) g, g + kGroups, g + 2 kGroups, ... of the CTA, so several
// stages are being split at once.  Each group has a multiple of 4 warps (one
// or more per tensor-memory lane quadrant); thread t of a group holds B^T
// column t % 128 and kBtK of the stage's 16 k values.  kPrefetch register
// buffers per producer thread: the loads of kPrefetch - 1 of its jobs are in
// flight while it splits one.  With A arriving by TMA the registers only
// hold B^T; without it they also hold A chunks, so wide tiles use fewer,
// larger groups to stay within the register budget.
template <int TM, bool TMA_A, bool TMA_B>
struct Roles {
    static constexpr bool kTma = TMA_A || TMA_B;  // the TMA thread fills stages
    // With A copied by TMA the producers hold few registers: 12 warps in 3
    // groups leave 96 registers per thread; otherwise 16 warps.
    static constexpr int kProdWarps = TMA_A ? 12 : 16;
    static constexpr int kGroups = TMA_A ? 3 : (TM <= 64 ? 4 : 2);
    static constexpr int kWarpsPerGroup = kProdWarps / kGroups;
    static_assert(kWarpsPerGroup % 4 == 0, "each group covers the four lane quadrants");
    static constexpr int kGroupThreads = kWarpsPerGroup * 32;
    static constexpr int kBtK = kBK * 4 / kWarpsPerGroup;
    static constexpr int kPrefetch = 2;
    static constexpr int kMmaWarp = kEpiWarps + kProdWarps;
    static constexpr int kTmaWarp = kMmaWarp + 1;
    static constexpr int kThreads = (kEpiWarps + kProdWarps + 2) * 32;
};

// Tensor memory (512 columns of 128 lanes x 32 bit): accumulators of TM
// columns each, then a ring of STAGES B^T stages of 32 columns (16 hi + 16 lo
// k values per lane = per C column).
constexpr uint32_t kTmemCols = 512;
constexpr int kRingColsPerStage = 2 * kBK;
constexpr int kMaxStages = 12;
// Short tiles (TM <= 64) pair the products: a tf32 MMA costs at least ~40 ns
// whatever its N up to 128, and in a stage the lo half of the A tile follows
// the hi half with the same row pitch, so [A_hi; A_lo] is one 2TM-row
// operand.  Per 8-deep k slice: B^T_hi x [A_hi; A_lo] (N = 2TM) gives hi*hi
// and hi*lo side by side, then B^T_lo x A_hi (N = TM) adds lo*hi to the first
// half: two MMAs instead of three.  The accumulator is 2TM columns wide and
// the epilogue adds its halves.
__host__ __device__ constexpr bool paired_for(int tm) { return tm <= 64; }
__host__ __device__ constexpr int acc_cols_for(int tm) { return (paired_for(tm) ? 2 : 1) * tm; }
// Accumulators: two (a tile's epilogue overlaps the next tile's MMAs), one
// from TM = 192 up.
__host__ __device__ constexpr int nacc_for(int tm) { return tm >= 192 ? 1 : 2; }
// every tensor-memory column the accumulators leave, up to kMaxStages (short
// tiles stream long B panels and want many copies in flight)
__host__ __device__ constexpr int stages_for(int tm) {
    return (static_cast<int>(kTmemCols) - nacc_for(tm) * acc_cols_for(tm)) / kRingColsPerStage < kMaxStages
               ? (static_cast<int>(kTmemCols) - nacc_for(tm) * acc_cols_for(tm)) / kRingColsPerStage
               : kMaxStages;
}
constexpr int kSmemLimit = 232448;  // dynamic shared memory one CTA may use on sm_103a
// C chunks the epilogue stages in shared memory for TMA copies (16 rows of
// the 128 tile columns each); loads run two chunks ahead of the arithmetic.
constexpr int kEpiBufs = 3;
constexpr int kEpiRows = 16;
constexpr int kEpiChunkBytes = kEpiRows * 128 * 4;
// Shared tiles whose sum a CTA defers to its exit (see fixup_tile); the
// planner gives no CTA more split-K units than this.
constexpr int kMaxDefer = 8;

// B rows that are not 16-byte aligned (ldb % 4 != 0, e.g. N = 14161) still
// come by TMA: rows k with the same k % 4 (a residue class r) lie 4 * ldb
// floats apart, a multiple of 16 bytes, so each class is a tensor of its own
// whose start is rounded down to 16 bytes; its rows then begin o_r = (r *
// ldb) % 4 floats into the copied box.  A stage's slab holds, per class,
// the 4 rows of the class among its 16 k, each kB4Row floats wide (128
// columns plus up to 3 leading floats), in blocks of kB4ClassBytes (a
// multiple of 128 bytes, the TMA destination alignment).
constexpr int kB4Row = kTileN + 4;                     // 132 floats = 528 bytes, a multiple of 16
constexpr int kB4RowBytes = kB4Row * 4;
constexpr int kB4ClassBytes = (4 * kB4RowBytes + 127) / 128 * 128;  // 2176
constexpr int kB4SlabBytes = 4 * kB4ClassBytes;

// TM = C rows per tile (MMA N).  TMA_B: each stage also has a slab for the
// raw B tile (16 k rows x 128 n, copied by TMA) that the producers read and
// split; B4: that slab holds the four residue classes of an unaligned B.
// PAIR: the tile is shared by the two CTAs of a cluster (one cta_group::2
// MMA of M = 256: 128 C columns per CTA); each CTA holds TM / 2 of the A
// tile's rows (the MMA's N rows are split between the pair).
// Shared memory: the stages' A tiles (hi, lo), then the stages' B slabs,
// then the epilogue's C buffers and the barriers.
template <int TM, bool TMA_B = false, bool B4 = false, bool PAIR = false>
struct Cfg {
    static_assert(TM % 16 == 0 && TM >= 16 && TM <= 256, "MMA N for M=128 must be 16..256, step 16");
    static_assert(TMA_B || !B4, "the residue-class form is a TMA form");
    static_assert(!PAIR || TM == 192 || TM == 256, "CTA pairs for tiles of 192 or 256 rows");
    static constexpr int kNacc = nacc_for(TM);
    static constexpr int kAR = PAIR ? TM / 2 : TM;  // A rows held by this CTA
    static constexpr int kABytes = kAR * kBK * 4;  // A tile (MMA B operand), one of hi / lo
    static constexpr int kOffAHi = 0;             // also where TMA lands the raw A tile
    static constexpr int kOffALo = kABytes;
    static constexpr int kAStageBytes = 2 * kABytes;
    static constexpr int kBRawBytes = TMA_B ? (B4 ? kB4SlabBytes : kBK * kTileN * 4) : 0;
    static constexpr int kStageBytes = kAStageBytes + kBRawBytes;  // shared memory per stage, A and B
    // epilogue staging for TMA copies of C: kEpiBufs chunks of 16 rows x 128
    static constexpr int kEpiBufBytes = kEpiBufs * kEpiChunkBytes;
    // as many stages as tensor memory and the 227 KB of shared memory allow
    // (1 KB of alignment slack and up to 528 bytes of barriers and words)
    static constexpr int kStageRoom = kSmemLimit - 1024 - 528 - kEpiBufBytes;
    static constexpr int kStages = stages_for(TM) < kStageRoom / kStageBytes ? stages_for(TM)
                                                                             : kStageRoom / kStageBytes;
    static constexpr int kOffBRegion = kStages * kAStageBytes;  // slab of stage s at + s * kBRawBytes
    static constexpr int kOffEpi = kStages * kStageBytes;
    static_assert(kAStageBytes % 1024 == 0, "A tiles must keep 1 KB alignment (64-byte swizzle atoms)");
    static_assert(kBRawBytes % 512 == 0 || B4, "B slabs keep the 64-byte swizzle's 512-byte alignment");
    static_assert(kBRawBytes % 128 == 0 && kOffEpi % 128 == 0, "TMA destinations 128-byte aligned");
    static constexpr bool kPaired = paired_for(TM);
    static constexpr int kAccCols = acc_cols_for(TM);  // one accumulator (two TM halves when paired)
    static constexpr int kRingCol = kNacc * kAccCols;
    static_assert(kRingCol + kStages * kRingColsPerStage <= static_cast<int>(kTmemCols), "tensor memory");
    static constexpr int kChunk = 16;  // accumulator columns per tensor-memory load in the epilogue
    static constexpr uint32_t kIdesc = umma_idesc_tf32(PAIR ? 2 * kTileN : kTileN, TM);
    static constexpr uint32_t kIdescPair = umma_idesc_tf32(kTileN, 2 * TM);  // N = 2TM: [A_hi; A_lo]
    static_assert(!kPaired || (kABytes % 512 == 0 && 2 * TM <= 256), "[A_hi; A_lo] as one swizzled operand");
    static_assert(!(PAIR && kPaired), "paired products are a single-CTA form");
    // barriers: full[S], empty[S], a_full[S], acc_full[2], acc_empty[2],
    // drain, c_full[kEpiBufs]; then words: tensor-memory address, abort
    // flag, (unused), count of deferred sums, and kMaxDefer entries (tile row,
    // tile column, segment count, first workspace slot)
    static constexpr int kBarBytes = 8 * (3 * kStages + 5 + kEpiBufs) + 4 * (4 + 5 * kMaxDefer);
    static constexpr int kSmemBytes = 1024 + kOffEpi + kEpiBufBytes + kBarBytes;
    static_assert(kBarBytes <= 528, "room kept for the barriers");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory per CTA");
    // a dense convolution's tap table (kConvTabMax ints, 16-byte aligned)
    static constexpr int kConvTabBytes = kConvTabMax * 4 + 16;
    static_assert(TMA_B || kSmemBytes + kConvTabBytes <= kSmemLimit, "shared memory with a tap table");
    static_assert(kStages >= 4, "pipeline depth");
};

// Byte offset of the 16-byte chunk `chunk` (k / 4) of row `row` inside a
// K-major tile with 64-byte rows and the 64-byte swizzle (the layout both the
// tensor core and a TMA copy with 64-byte swizzle use).
__device__ __forceinline__ uint32_t sw64_off(int row, int chunk) {
    return static_cast<uint32_t>(row * 64 + (((chunk ^ (row >> 1)) & 3) << 4));
}

// hi/lo split of one fp32 value: hi = x with the low 13 mantissa bits
// cleared (an exact tf32 value), lo = x - hi (exact in fp32; |lo| < 2^-10
// |x|, the tensor core keeps its top 11 significant bits, an error below
// 2^-20 |x|).  The tensor core reads a tf32 operand as the top 19 bits of
// its 32-bit word and ignores the rest, so the raw fp32 word of x serves as
// hi unchanged: operands copied by TMA keep x in place and only lo is
// written (a GPU test checks that both forms give the same bits).
// Non-finite x gives lo = NaN; the accumulator then comes out NaN and the
// epilogue recomputes that element exactly (recompute_dot), so Inf and NaN
// inputs still produce the IEEE fp32 result.  One logic op and one FADD.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    const uint32_t hu = __float_as_uint(x) & 0xFFFFE000u;
    hi = hu;
    lo = __float_as_uint(x - __uint_as_float(hu));
}

// One k-tile of operands held in a producer thread's registers.
template <int BK_, int AJ>
struct Raw {
    float b[BK_];    // B^T: BK_ consecutive k of one column n
    float a[AJ][4];  // A chunks: 4 consecutive k of one row m
};
template <int BK_>
struct Raw<BK_, 0> {
    float b[BK_];
};
template <int AJ>
struct Raw<0, AJ> {
    float a[AJ][4];
};
template <>
struct Raw<0, 0> {};

// Producer: load one k-tile (K-range [k0, k0+16)) into registers; out-of-range
// elements read as 0.  Thread gt of a group holds B[k0+BtK*h .. +BtK-1][n0+(gt&127)]
// with h = gt >> 7 (its tensor-memory lane is its column), and A chunks
// j = gt + GT * r: row j >> 2, k chunk j & 3 (GT threads per group).
// CONV: B is gathered from the input image (implicit im2col); a warp's 32
// columns are 32 neighbouring output pixels, so each k reads one stretch of
// an input row.  kConvTaps: k = (c * KH + kh) * KW + kw, the filter's own
// (OIHW) order; the tap of k is the same for the whole warp and advances
// with k.  kConvChannels: k = (kh * KW + kw) * C + c (filter staged OHWI,
// C a multiple of 16), so the 16 k of a call are 16 channels at one tap:
// one bounds check, then loads H * W apart, like a plain B column.
// kConvTapsDense: the kConvTaps order on an input where every tap lies in
// the image; element (k, n) is the pixel at the column's window origin plus
// ctab[k] (the tap's offset, a per-CTA table in shared memory).
template <int TM, int BtK, int GT, int AJ, int CONV = kConvNone>
__device__ __forceinline__ void load_raw(const GemmArgs &g, bool vec_a, int bi, int m0, int n0, int k0,
                                         int ptid, Raw<BtK, AJ> &raw, const int *ctab = nullptr) {
    if constexpr (BtK > 0 && CONV == kConvTapsDense) {
        const ConvGeom &cv = g.cv;
        const int n = n0 + (ptid & (kTileN - 1));
        const int kb = k0 + (ptid >> 7) * BtK;
        const bool n_ok = n < g.N;
        const int oh = n_ok ? n / cv.OW : 0;
        const int pix0 = oh * cv.sh * cv.W + (n_ok ? n - oh * cv.OW : 0) * cv.sw;
        const float *xp = g.B + bi * g.sB + pix0;
#pragma unroll
        for (int e = 0; e < BtK; ++e)
            raw.b[e] = (n_ok && kb + e < g.K && SG_IN_B(g, xp + ctab[kb + e], 1)) ? __ldg(xp + ctab[kb + e]) : 0.f;
    } else if constexpr (BtK > 0 && CONV == kConvChannels) {
        const ConvGeom &cv = g.cv;
        const int n = n0 + (ptid & (kTileN - 1));
        const int kb = k0 + (ptid >> 7) * BtK;
        const int tap = kb / cv.C, c0 = kb - tap * cv.C;
        const int kh = tap / cv.KW, kw = tap - kh * cv.KW;
        const int oh = n / cv.OW;
        const int ih = oh * cv.sh - cv.ph + kh * cv.dh;
        const int iw = (n - oh * cv.OW) * cv.sw - cv.pw + kw * cv.dw;
        const bool ok = n < g.N && kb < g.K && static_cast<unsigned>(ih) < static_cast<unsigned>(cv.H) &&
                        static_cast<unsigned>(iw) < static_cast<unsigned>(cv.W);
        const long long plane = static_cast<long long>(cv.H) * cv.W;
        const float *src = g.B + bi * g.sB + c0 * plane + static_cast<long long>(ih) * cv.W + iw;
#pragma unroll
        for (int e = 0; e < BtK; ++e) raw.b[e] = (ok && SG_IN_B(g, src + e * plane, 1)) ? __ldg(src + e * plane) : 0.f;
    } else if constexpr (BtK > 0 && CONV == kConvTaps) {
        const ConvGeom &cv = g.cv;
        const int n = n0 + (ptid & (kTileN - 1));
        const int kb = k0 + (ptid >> 7) * BtK;
        const bool n_ok = n < g.N;
        const int oh = n_ok ? n / cv.OW : 0;
        // first input pixel of this column's window (may lie in the padding)
        const int ih0 = oh * cv.sh - cv.ph;
        const int iw0 = (n_ok ? n - oh * cv.OW : 0) * cv.sw - cv.pw;
        const int pix0 = ih0 * cv.W + iw0;
        // tap of k: (row offset, column offset, offset in the image), the same
        // for the whole warp
        const int khw = cv.KH * cv.KW;
        const int c = kb / khw;
        int kh = (kb - c * khw) / cv.KW;
        int kw = kb - c * khw - kh * cv.KW;
        int coff = c * cv.H * cv.W;
        const float *xb = g.B + bi * g.sB;
#pragma unroll
        for (int e = 0; e < BtK; ++e) {
            const int dy = kh * cv.dh, dx = kw * cv.dw;
            const bool ok = n_ok && kb + e < g.K && static_cast<unsigned>(ih0 + dy) < static_cast<unsigned>(cv.H) &&
                            static_cast<unsigned>(iw0 + dx) < static_cast<unsigned>(cv.W);
            const float *px = xb + (coff + dy * cv.W + dx + pix0);
            raw.b[e] = (ok && SG_IN_B(g, px, 1)) ? __ldg(px) : 0.f;
            if (++kw == cv.KW) {
                kw = 0;
                if (++kh == cv.KH) {
                    kh = 0;
                    coff += cv.H * cv.W;
                }
            }
        }
    } else if constexpr (BtK > 0) {
        const int n = n0 + (ptid & (kTileN - 1));
        const int kb = k0 + (ptid >> 7) * BtK;
        const bool n_ok = n < g.N;
        const float *src = g.B + bi * g.sB + static_cast<long long>(kb) * g.ldb + n;
#pragma unroll
        for (int e = 0; e < BtK; ++e)
            raw.b[e] = (n_ok && kb + e < g.K && SG_IN_B(g, src + e * g.ldb, 1)) ? __ldg(src + e * g.ldb) : 0.f;
    }
    if constexpr (AJ > 0) {
#pragma unroll
        for (int r = 0; r < AJ; ++r) {
            const int j = ptid + r * GT;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (j < TM * 4) {
                const int m = m0 + (j >> 2);
                const int k = k0 + (j & 3) * 4;
                if (m < g.M) {
                    const float *src = g.A + bi * g.sA + static_cast<long long>(m) * g.lda + k;
                    if (vec_a && k + 3 < g.K) {
                        if (SG_IN_A(g, src, 4)) v = __ldg(reinterpret_cast<const float4 *>(src));
                    } else {
                        v.x = (k + 0 < g.K && SG_IN_A(g, src + 0, 1)) ? __ldg(src + 0) : 0.f;
                        v.y = (k + 1 < g.K && SG_IN_A(g, src + 1, 1)) ? __ldg(src + 1) : 0.f;
                        v.z = (k + 2 < g.K && SG_IN_A(g, src + 2, 1)) ? __ldg(src + 2) : 0.f;
                        v.w = (k + 3 < g.K && SG_IN_A(g, src + 3, 1)) ? __ldg(src + 3) : 0.f;
                    }
                }
            }
            raw.a[r][0] = v.x;
            raw.a[r][1] = v.y;
            raw.a[r][2] = v.z;
            raw.a[r][3] = v.w;
        }
    }
}

__device__ __forceinline__ void split_store4(uint32_t hi_addr, uint32_t lo_addr, const float (&x)[4]) {
    uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
    split_tf32(x[0], h0, l0);
    split_tf32(x[1], h1, l1);
    split_tf32(x[2], h2, l2);
    split_tf32(x[3], h3, l3);
    sts128(hi_addr, h0, h1, h2, h3);
    sts128(lo_addr, l0, l1, l2, l3);
}

// Producer: split one k-tile into pipeline stage `s`: B^T hi/lo from
// registers into tensor-memory columns [ring + 32 s, +32) of this warp's
// lanes; A hi/lo into the shared-memory stage at `stage`, from registers
// (AJ > 0) or, after a TMA copy into the hi buffer, lo alone (the raw tile
// is already a valid hi operand).
// TRANS_B: B is stored transposed (N x K, k innermost) and TMA copied the
// slab as 128 n rows of 16 k (64 bytes, 64-byte swizzle): a thread's column
// is one row, read as KB / 4 16-byte chunks (the swizzle spreads the 8
// lanes of each 128-bit load phase over all 32 banks).
// B4: the slab holds the residue classes of an unaligned B (kB4Row floats
// per row); b_offs packs o_r, the leading floats of class r's rows, in bits
// 2r..2r+1.
template <int TM, bool TMA_B, int KB, int BtK, int GT, int AJ, int AJ_TMA, bool TRANS_B = false, bool B4 = false,
          bool PAIR = false>
__device__ __forceinline__ void store_split(uint32_t stage, uint32_t slab, uint32_t ring_taddr, int ptid,
                                            const Raw<BtK, AJ> &raw, uint32_t b_offs = 0) {
    using C = Cfg<TM, TMA_B, B4, PAIR>;
    static_assert(!PAIR || AJ == 0, "a CTA pair copies A by TMA");
    {
        // KB k values of this thread's B^T column: from registers, or from the
        // raw B tile (k rows of 128 floats) that TMA copied into the slab
        uint32_t hi[KB], lo[KB];
        if constexpr (TMA_B && B4) {
            static_assert(KB % 4 == 0, "whole residue classes");
            const int n = ptid & (kTileN - 1);
            const int kb = (ptid >> 7) * KB;  // a multiple of 4: k % 4 == e % 4
#pragma unroll
            for (int e = 0; e < KB; ++e) {
                const int r = e & 3;
                const uint32_t o = (b_offs >> (2 * r)) & 3u;
                const float x = lds32f(slab + static_cast<uint32_t>(r * kB4ClassBytes + ((kb + e) >> 2) * kB4RowBytes) +
                                       (static_cast<uint32_t>(n) + o) * 4u);
                split_tf32(x, hi[e], lo[e]);
                hi[e] = __float_as_uint(x);  // raw word: the tensor core drops the low bits
            }
        } else if constexpr (TMA_B && TRANS_B) {
            static_assert(KB % 4 == 0, "whole 16-byte chunks");
            const int n = ptid & (kTileN - 1);
            const int q0 = ((ptid >> 7) * KB) >> 2;  // first 16-byte chunk (4 k) of this thread
#pragma unroll
            for (int q = 0; q < KB / 4; ++q) {
                const float4 v = lds128(slab + sw64_off(n, q0 + q));
                const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    split_tf32(x[u], hi[4 * q + u], lo[4 * q + u]);
                    hi[4 * q + u] = __float_as_uint(x[u]);  // raw word: the tensor core drops the low bits
                }
            }
        } else if constexpr (TMA_B) {
            const uint32_t col = slab + static_cast<uint32_t>((ptid & (kTileN - 1)) * 4);
            const int kb = (ptid >> 7) * KB;
#pragma unroll
            for (int e = 0; e < KB; ++e) {
                const float x = lds32f(col + static_cast<uint32_t>((kb + e) * kTileN * 4));
                split_tf32(x, hi[e], lo[e]);
                hi[e] = __float_as_uint(x);  // raw word: the tensor core drops the low bits
            }
        } else {
#pragma unroll
            for (int e = 0; e < KB; ++e) split_tf32(raw.b[e], hi[e], lo[e]);
        }
        const uint32_t t = ring_taddr + static_cast<uint32_t>((ptid >> 7) * KB);
        tmem_st_cols<KB>(t, hi);
        tmem_st_cols<KB>(t + kBK, lo);
    }
    if constexpr (AJ > 0) {
#pragma unroll
        for (int r = 0; r < AJ; ++r) {
            const int j = ptid + r * GT;
            if (j < TM * 4) {
                const uint32_t off = sw64_off(j >> 2, j & 3);
                split_store4(stage + C::kOffAHi + off, stage + C::kOffALo + off, raw.a[r]);
            }
        }
    } else {
#pragma unroll
        for (int r = 0; r < AJ_TMA; ++r) {
            const int j = ptid + r * GT;
            if (j < C::kAR * 4) {
                const uint32_t off = sw64_off(j >> 2, j & 3);
                // the raw tile stays in place as hi; only lo is written
                const float4 v = lds128(stage + C::kOffAHi + off);
                uint32_t h, l0, l1, l2, l3;
                split_tf32(v.x, h, l0);
                split_tf32(v.y, h, l1);
                split_tf32(v.z, h, l2);
                split_tf32(v.w, h, l3);
                sts128(stage + C::kOffALo + off, l0, l1, l2, l3);
            }
        }
    }
}

// Exact fp32 dot product of row m of A and column n of B, in k order.  The
// epilogue calls it only for an accumulator that came out NaN: with the
// 3xTF32 split an infinite operand meeting a partner whose lo part is zero
// gives Inf * 0 = NaN where fp32 arithmetic gives +-Inf, so NaN results are
// recomputed on the CUDA cores.  Stops early once the sum itself is NaN.
// TRANS_B: B is stored N x K (element (k, n) at B[n * ldb + k]).
template <int CONV, bool TRANS_B = false>
__device__ __noinline__ float recompute_dot(const GemmArgs &g, int bi, int m, int n) {
    const float *a = g.A + bi * g.sA + static_cast<long long>(m) * g.lda;
    float s = 0.f;
    if constexpr (CONV == kConvChannels) {  // k walks (kh, kw, c) in order
        const ConvGeom &cv = g.cv;
        const int oh = n / cv.OW;
        const int ih0 = oh * cv.sh - cv.ph, iw0 = (n - oh * cv.OW) * cv.sw - cv.pw;
        const long long plane = static_cast<long long>(cv.H) * cv.W;
        const float *x = g.B + bi * g.sB;
        int k = 0;
        for (int kh = 0; kh < cv.KH; ++kh) {
            const int ih = ih0 + kh * cv.dh;
            for (int kw = 0; kw < cv.KW; ++kw) {
                const int iw = iw0 + kw * cv.dw;
                const bool in = static_cast<unsigned>(ih) < static_cast<unsigned>(cv.H) &&
                                static_cast<unsigned>(iw) < static_cast<unsigned>(cv.W);
                const float *px = x + static_cast<long long>(ih) * cv.W + iw;
                for (int c = 0; c < cv.C; ++c, ++k)
                    s = fmaf(SG_IN_A(g, a + k, 1) ? __ldg(a + k) : 0.f,
                             (in && SG_IN_B(g, px + c * plane, 1)) ? __ldg(px + c * plane) : 0.f, s);
            }
            if (s != s) break;
        }
    } else if constexpr (CONV == kConvTaps || CONV == kConvTapsDense) {  // k walks the taps (c, kh, kw) in order
        const ConvGeom &cv = g.cv;
        const int oh = n / cv.OW;
        const int ih0 = oh * cv.sh - cv.ph, iw0 = (n - oh * cv.OW) * cv.sw - cv.pw;
        const float *x = g.B + bi * g.sB;
        int k = 0;
        for (; k < g.K; x += static_cast<long long>(cv.H) * cv.W) {
            for (int kh = 0; kh < cv.KH; ++kh) {
                const int ih = ih0 + kh * cv.dh;
                for (int kw = 0; kw < cv.KW; ++kw, ++k) {
                    const int iw = iw0 + kw * cv.dw;
                    const bool in = static_cast<unsigned>(ih) < static_cast<unsigned>(cv.H) &&
                                    static_cast<unsigned>(iw) < static_cast<unsigned>(cv.W);
                    const float *px = x + static_cast<long long>(ih) * cv.W + iw;
                    s = fmaf(SG_IN_A(g, a + k, 1) ? __ldg(a + k) : 0.f, (in && SG_IN_B(g, px, 1)) ? __ldg(px) : 0.f, s);
                }
            }
            if (s != s) break;
        }
    } else if constexpr (TRANS_B) {
        const float *b = g.B + bi * g.sB + static_cast<long long>(n) * g.ldb;
        for (int k = 0; k < g.K; ++k) {
            s = fmaf(SG_IN_A(g, a + k, 1) ? __ldg(a + k) : 0.f, SG_IN_B(g, b + k, 1) ? __ldg(b + k) : 0.f, s);
            if (s != s) break;
        }
    } else {
        const float *b = g.B + bi * g.sB + n;
        for (int k = 0; k < g.K; ++k) {
            const float *pb = b + static_cast<long long>(k) * g.ldb;
            s = fmaf(SG_IN_A(g, a + k, 1) ? __ldg(a + k) : 0.f, SG_IN_B(g, pb, 1) ? __ldg(pb) : 0.f, s);
            if (s != s) break;
        }
    }
    return s;
}

// The (work unit, k tile) jobs of one CTA, in the order the producers fill
// the pipeline: the CTA's units in next_unit order, each from its first to
// its last k tile.  Keeps only what a producer needs (tile position, k tile,
// end of the unit) to stay light on registers.
struct JobIter {
    int cta, i;
    bool tail, ok;
    int b, mt, nt, kt, ke;
    __device__ __forceinline__ void load(const Schedule &s) {
        UnitCoord c;
        ok = next_unit(s, cta, i, tail, c);
        if (ok) {
            b = c.b;
            mt = c.mt;
            nt = c.nt;
            kt = c.kb;
            ke = c.ke;
        }
    }
    __device__ __forceinline__ void start(const Schedule &s, int cta_) {
        cta = cta_;
        i = 0;
        tail = false;
        load(s);
    }
    __device__ __forceinline__ bool valid(const Schedule &) const { return ok; }
    __device__ __forceinline__ void advance(const Schedule &s) {
        if (++kt >= ke) load(s);
    }
};

// Epilogue-wide vote: all 128 epilogue threads synchronise and agree.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(kEpiBarrierId), "r"(kEpiWarps * 32)
        : "memory");
    return r != 0;
}

// One 16-column chunk of an accumulator: 16 C rows of this thread's column.
// A paired accumulator holds hi*hi + lo*hi in its first TM columns and hi*lo
// in the next TM; the chunk is their sum.
template <int TM>
__device__ __forceinline__ void acc_chunk(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld32x16_issue(taddr, r);
    if constexpr (paired_for(TM)) {
        uint32_t q[16];
        tmem_ld32x16_issue(taddr + static_cast<uint32_t>(TM), q);
        tmem_ld_wait16(r);
        tmem_ld_wait16(q);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]) + __uint_as_float(q[j]);
    } else {
        tmem_ld_wait16(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
    }
}

// Last-arriver sum of a shared tile, by a team of nw warps (wid = this
// warp's index in the team).  The nseg partial tiles (TM x 128, row-major,
// contiguous from wb) and the C tile are read row by row with 16-byte loads:
// a warp covers one 128-column row per load and each thread keeps kFixRows
// rows x (up to kFixSegs segments + C) loads in flight.  The partials are
// added in segment order, starting from zero, whatever order the units
// arrived in, so the bits of C do not depend on timing.
constexpr int kFixRows = 1;
constexpr int kFixSegs = 3;

__device__ __forceinline__ float4 ld4cg(const float *p) {
    return __ldcg(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ float fix_lane(const float4 &v, int q) {
    return q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
}

template <int TM, int CONV, bool TRANS_B>
__device__ __forceinline__ void fixup_tile(const GemmArgs &g, const DeviceCtl &ctl, int bi, const float *wb, int nseg,
                                           int m0, int n0, int wid, int nw, int lane) {
    float *const cmat = g.C + bi * g.sC;  // matrix bi of a batch
    constexpr long long kTileElems = static_cast<long long>(kTileN) * TM;
    const int pass = kFixRows * nw;  // rows per pass
    const int nc = n0 + 4 * lane;    // first of this thread's 4 columns
    if (nc >= g.N) return;
    const bool vec_c = (reinterpret_cast<uintptr_t>(cmat) & 15u) == 0 && (g.ldc & 3) == 0;
    const bool full4 = vec_c && nc + 3 < g.N;
    const bool read_c = g.beta != 0.f;
    const int rows = min(TM, g.M - m0);
#pragma unroll 1
    for (int r0 = wid; r0 < rows; r0 += pass) {
        // rows r0 + nw * j of the tile
        float4 old[kFixRows];
#pragma unroll
        for (int j = 0; j < kFixRows; ++j) {
            const int r = r0 + nw * j;
            old[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (read_c && r < rows) {
                const float *cp = cmat + static_cast<long long>(m0 + r) * g.ldc + nc;
                if (full4) {
                    if (SG_IN_C(g, cp, 4)) old[j] = *reinterpret_cast<const float4 *>(cp);
                } else {
                    if (SG_IN_C(g, cp, 1)) old[j].x = cp[0];
                    if (nc + 1 < g.N && SG_IN_C(g, cp + 1, 1)) old[j].y = cp[1];
                    if (nc + 2 < g.N && SG_IN_C(g, cp + 2, 1)) old[j].z = cp[2];
                    if (nc + 3 < g.N && SG_IN_C(g, cp + 3, 1)) old[j].w = cp[3];
                }
            }
        }
        float4 sum[kFixRows];
#pragma unroll
        for (int j = 0; j < kFixRows; ++j) sum[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int s0 = 0; s0 < nseg; s0 += kFixSegs) {
            float4 v[kFixSegs][kFixRows];
#pragma unroll
            for (int q = 0; q < kFixSegs; ++q)
#pragma unroll
                for (int j = 0; j < kFixRows; ++j)
                    if (s0 + q < nseg && r0 + nw * j < rows) {
                        const float *pw = wb + (s0 + q) * kTileElems + static_cast<long long>(r0 + nw * j) * kTileN +
                                          4 * lane;
                        v[q][j] = SG_IN_WS(ctl, pw, 4) ? ld4cg(pw) : make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
            for (int q = 0; q < kFixSegs; ++q)
                if (s0 + q < nseg)
#pragma unroll
                    for (int j = 0; j < kFixRows; ++j) {
                        sum[j].x += v[q][j].x;
                        sum[j].y += v[q][j].y;
                        sum[j].z += v[q][j].z;
                        sum[j].w += v[q][j].w;
                    }
        }
#pragma unroll
        for (int j = 0; j < kFixRows; ++j) {
            const int r = r0 + nw * j;
            if (r >= rows) continue;
            const int m = m0 + r;
            float res[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float s = fix_lane(sum[j], q);
                if (s != s && nc + q < g.N) s = recompute_dot<CONV, TRANS_B>(g, bi, m, nc + q);
                const float a = g.alpha * s;
                res[q] = read_c ? fmaf(g.beta, fix_lane(old[j], q), a) : a;
            }
            float *cp = cmat + static_cast<long long>(m) * g.ldc + nc;
            if (full4) {
                if (SG_IN_C(g, cp, 4)) *reinterpret_cast<float4 *>(cp) = make_float4(res[0], res[1], res[2], res[3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (nc + q < g.N && SG_IN_C(g, cp + q, 1)) cp[q] = res[q];
            }
        }
    }
}

// Ask L2 for the C tile (rows m0.., columns n0..) that an epilogue will read
// once the accumulator is ready; thread t of the epilogue takes rows t,
// t + 128, ...  Only whole 16-byte pieces inside C are requested.
template <int TM>
__device__ __forceinline__ void prefetch_c_tile(const GemmArgs &g, int bi, int m0, int n0, int t) {
    const int cols = min(kTileN, g.N - n0);
    float *const cmat = g.C + bi * g.sC;
    const bool vec = (reinterpret_cast<uintptr_t>(cmat) & 15u) == 0 && (g.ldc & 3) == 0;
#pragma unroll 1
    for (int r = t; r < TM && m0 + r < g.M; r += kEpiWarps * 32) {
        const float *row = cmat + static_cast<long long>(m0 + r) * g.ldc + n0;
        if (vec) {
            const uint32_t bytes = static_cast<uint32_t>(cols * 4) & ~15u;
            if (bytes && SG_IN_C(g, row, static_cast<int>(bytes / 4))) prefetch_l2_bulk(row, bytes);
        } else {
            for (int q = 0; q < cols; q += 32)
                if (SG_IN_C(g, row + q, 1)) prefetch_l2(row + q);
        }
    }
}

// TMA_A: A rows are 16-byte aligned and tmap_a describes A (K x M, 64-byte
// swizzle, box 16 x TM); otherwise the producers load A themselves.
// TMA_B: B rows are 16-byte aligned and tmap_b describes B (N x K, box
// 128 x 16, no swizzle); otherwise the producers load B^T themselves.
// CONV: implicit-GEMM convolution (kConvTaps, kConvChannels or
// kConvTapsDense; B gathered from the input image by the producers, TMA_B
// false).  kConvTapsDense launches with kConvTabBytes more shared memory for
// the tap table.
// TRANS_B: B is stored N x K (BLAS transb) and tmap_b describes it as K x N
// (box 16 x 128, 64-byte swizzle); needs TMA_B.
// B4: B's rows are not 16-byte aligned; tmap_b, tmap_b1, tmap_b2, tmap_b3
// describe its residue classes k % 4 = 0..3 (each N + o_r floats wide, box
// 132 x 4, no swizzle) and b_offs packs the o_r; needs TMA_B.
// PAIR: launched in clusters of two CTAs that share each 256-column tile
// (sch.pair_shift = 1): CTA r of the pair owns columns 128 r .. 128 r + 127
// of the tile (its B^T slab, its tensor-memory lanes, its C stores) and
// rows kAR r .. kAR r + kAR - 1 of the A tile (tmap_a's box is kAR rows);
// the even CTA's MMA thread issues the pair's MMAs.  Needs TMA_A and TMA_B.
template <int TM, bool TMA_A, bool TMA_B, int CONV = kConvNone, bool TRANS_B = false, bool B4 = false,
          bool PAIR = false>
__global__ void __launch_bounds__(Roles<TM, TMA_A, TMA_B>::kThreads, 1)
    tf32x3_gemm_kernel(const __grid_constant__ GemmArgs g, const __grid_constant__ Schedule sch,
                       const __grid_constant__ DeviceCtl ctl, int vec_a, int tma_c, uint32_t b_offs,
                       const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                       const __grid_constant__ CUtensorMap tmap_c, const __grid_constant__ CUtensorMap tmap_b1,
                       const __grid_constant__ CUtensorMap tmap_b2, const __grid_constant__ CUtensorMap tmap_b3) {
    using C = Cfg<TM, TMA_B, B4, PAIR>;
    using R = Roles<TM, TMA_A, TMA_B>;
    static_assert(CONV == kConvNone || !TMA_B, "a convolution gathers B in the producers");
    static_assert(!PAIR || (TMA_A && TMA_B && CONV == kConvNone), "a CTA pair copies A and B by TMA");
    static_assert(!TRANS_B || (TMA_B && CONV == kConvNone), "a transposed B comes by TMA");
    static_assert(!B4 || (TMA_B && !TRANS_B && CONV == kConvNone), "residue classes of a row-major B");
    constexpr int S = C::kStages;
    constexpr int CH = C::kChunk;
    static_assert(R::kGroups <= S, "a group's next stage must not wrap the ring twice");
    extern __shared__ uint8_t smem_raw[];

    const uint32_t raw_base = smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw_base);
    const uint32_t epi_buf0 = base + C::kOffEpi;                   // C chunk b at epi_buf0 + b * kEpiChunkBytes
    const uint32_t bars = base + C::kOffEpi + C::kEpiBufBytes;  // full[s] = bars + 8s, empty[s] = bars + 8(S+s)
    const uint32_t afull0 = bars + 8u * (2 * S);       // a_full[s]: TMA copy of stage s landed
    const uint32_t acc_full0 = bars + 8u * (3 * S);
    const uint32_t acc_empty0 = acc_full0 + 16u;
    const uint32_t drain_bar = acc_empty0 + 16u;
    const uint32_t cfull0 = drain_bar + 8u;            // c_full[b]: TMA copy of C chunk buffer b landed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(base_ptr + C::kOffEpi + C::kEpiBufBytes +
                                                       8 * (3 * S + 5 + kEpiBufs));
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *s_ndefer = reinterpret_cast<volatile int *>(tmem_slot + 3);
    volatile int *s_defer = reinterpret_cast<volatile int *>(tmem_slot + 4);  // [kMaxDefer][mt, nt, nseg, slot0, b]
    // tap offsets of a dense convolution, after the barriers (16-byte aligned)
    int *ctab = reinterpret_cast<int *>(base_ptr + ((C::kOffEpi + C::kEpiBufBytes + C::kBarBytes + 15) & ~15));
    if constexpr (CONV == kConvTapsDense) {
        const ConvGeom &cv = g.cv;
        const int khw = cv.KH * cv.KW;
        for (int k = threadIdx.x; k < g.K; k += blockDim.x) {
            const int c = k / khw, r = k - c * khw, kh = r / cv.KW, kw = r - kh * cv.KW;
            ctab[k] = (c * cv.H + kh * cv.dh) * cv.W + kw * cv.dw;
        }
    }

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pair: this CTA's rank, the pair's index among the walkers of the
    // schedule, and the column tile (of 128) this CTA owns in a unit's tile
    const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
    const int walker = PAIR ? static_cast<int>(blockIdx.x) >> 1 : static_cast<int>(blockIdx.x);
    auto col_tile = [&](int nt) { return PAIR ? 2 * nt + rank : nt; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // full: every thread of the filling group; of a pair, one arrive
            // per warp of each CTA's group (on the even CTA's barrier)
            mbar_init(bars + 8u * s, PAIR ? 2 * R::kWarpsPerGroup : R::kGroupThreads);
            mbar_init(bars + 8u * (S + s), 1);       // empty: one tcgen05.commit
            mbar_init(afull0 + 8u * s, 1);           // a_full: the TMA thread's expect_tx arrive
        }
        mbar_init(acc_full0, 1);
        mbar_init(acc_full0 + 8u, 1);
        // acc_empty: every epilogue thread; of a pair, one arrive per
        // epilogue warp of each CTA
        mbar_init(acc_empty0, PAIR ? 2 * kEpiWarps : kEpiWarps * 32);
        mbar_init(acc_empty0 + 8u, PAIR ? 2 * kEpiWarps : kEpiWarps * 32);
        mbar_init(drain_bar, 1);
        for (int b = 0; b < kEpiBufs; ++b) mbar_init(cfull0 + 8u * b, 1);
        *abort_flag = 0;
        *s_ndefer = 0;
        fence_mbar_init();
    }
    if (warp == R::kMmaWarp) {
        if constexpr (PAIR) {
            tmem_alloc2(smem_u32(tmem_slot), kTmemCols);  // collective over the pair
            tmem_relinquish2();
        } else {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    // a pair: the other CTA's barriers are initialised before any arrive on them
    if constexpr (PAIR) cluster_sync();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // of a pair, the even CTA's barriers that both CTAs arrive on
    const uint32_t lead_full0 = PAIR ? mapa_shared(bars, 0) : bars;
    const uint32_t lead_acc_empty0 = PAIR ? mapa_shared(acc_empty0, 0) : acc_empty0;
    // this warp has read the accumulator `acc` out: free it for the MMA
    auto release_acc = [&](int acc) {
        tc_fence_before();
        if constexpr (PAIR) {
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lead_acc_empty0 + 8u * acc);
        } else {
            mbar_arrive(acc_empty0 + 8u * acc);
        }
    };
    // Everything above is on chip.  Launched after another kernel of this
    // library, that kernel may still be running: wait for it here, before
    // any global memory is read or written, then let the next one start.
    grid_dep_wait();
    grid_dep_trigger();

    if (warp < kEpiWarps) {
        // ------------------------------------------------------ epilogue
        const int nl = warp * 32 + lane;  // tensor-memory lane = column within the tile
        int it = 0;
        uint32_t cpar = 0;      // per C buffer: parity of its next c_full phase
        uint32_t inflight = 0;  // per C buffer: a TMA copy into it not yet waited for
        UnitIter ui;
        for (ui.start(sch, walker); ui.ok; ui.next(sch), ++it) {
            const UnitCoord &c = ui.c;
            const int acc = it % C::kNacc;
            const uint32_t aph = (it / C::kNacc) & 1;
            const int ct = col_tile(c.nt);  // this CTA's column tile
            if (c.nseg == 1 && g.beta != 0.f) prefetch_c_tile<TM>(g, c.b, c.mt * TM, ct * kTileN, threadIdx.x);
            if (c.nseg == 1 && tma_c) {
                // the previous tile's stores have read their buffers; copy the
                // first C chunks of this tile while the accumulator is computed
                if (threadIdx.x == 0) bulk_wait_group_read<0>();
                if (g.beta != 0.f) {
                    // chunks that start at or beyond row M are never copied
                    const int nch = min(TM / CH, (g.M - c.mt * TM + CH - 1) / CH);
#pragma unroll
                    for (int ch = 0; ch < kEpiBufs - 1 && ch < nch; ++ch) {
                        if (threadIdx.x == 0) {
                            mbar_arrive_expect_tx(cfull0 + 8u * ch, kEpiChunkBytes);
                            tma_load_3d(epi_buf0 + ch * kEpiChunkBytes, &tmap_c, ct * kTileN, c.mt * TM + ch * CH,
                                        c.b, cfull0 + 8u * ch);
                        }
                        inflight |= 1u << ch;
                    }
                }
            }
            const bool w = mbar_wait_bounded(acc_full0 + 8u * acc, aph, abort_flag, ctl,
                                             kStatusTimeoutEpilogue);
            if (!epi_all(w)) break;
            tc_fence_after();
            const int n = ct * kTileN + nl;
            const int m0 = c.mt * TM;
            const uint32_t t0 = tmem_base + (static_cast<uint32_t>(warp * 32) << 16) +
                                static_cast<uint32_t>(acc * C::kAccCols);
            if (c.nseg == 1 && tma_c) {
                // Chunks of CH accumulator columns (C rows) staged in shared
                // memory: C copied in by TMA (two chunks ahead), alpha/beta
                // applied in place, the chunk copied out by one TMA store.
                // Buffer b of chunk ch = ch % kEpiBufs; before a buffer is
                // written again, the store that last read it has finished.
                static_assert(CH == kEpiRows, "one C chunk per tensor-memory load");
                const bool read_c = g.beta != 0.f;
                const bool n_ok = n < g.N;
                const int n0 = ct * kTileN;
                const int nch = min(TM / CH, (g.M - m0 + CH - 1) / CH);  // chunks with rows below M
                bool ok = true;
#pragma unroll 1
                for (int ch = 0; ch < nch; ++ch) {
                    const int b = ch % kEpiBufs;
                    const uint32_t col = epi_buf0 + b * kEpiChunkBytes + nl * 4;
                    if (read_c) {
                        const bool wc = mbar_wait_bounded(cfull0 + 8u * b, (cpar >> b) & 1u, abort_flag, ctl,
                                                          kStatusTimeoutEpilogue);
                        if (!epi_all(wc)) {
                            ok = false;
                            break;
                        }
                        cpar ^= 1u << b;
                        inflight &= ~(1u << b);
                    }
                    const int mb = m0 + ch * CH;
                    float v[CH];
                    acc_chunk<TM>(t0 + ch * CH, v);
                    bool nan = false;
#pragma unroll
                    for (int j = 0; j < CH; ++j) nan |= v[j] != v[j];
                    if (nan && n_ok) {
#pragma unroll 1
                        for (int j = 0; j < CH; ++j)
                            if (v[j] != v[j] && mb + j < g.M) v[j] = recompute_dot<CONV, TRANS_B>(g, c.b, mb + j, n);
                    }
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const uint32_t a = col + static_cast<uint32_t>(j * kTileN * 4);
                        sts32(a, read_c ? fmaf(g.beta, lds32f(a), g.alpha * v[j]) : g.alpha * v[j]);
                    }
                    fence_proxy_async_smem();
                    // the store of chunk ch - 2 has read its buffer (next iteration's)
                    if (threadIdx.x == 0) bulk_wait_group_read<kEpiBufs - 2>();
                    named_bar_sync(kEpiBarrierId, kEpiWarps * 32);
                    if (threadIdx.x == 0) {
                        tma_store_3d(&tmap_c, epi_buf0 + b * kEpiChunkBytes, n0, mb, c.b);
                        bulk_commit_group();
                    }
                    if (read_c && ch + kEpiBufs - 1 < nch) {
                        // chunk ch + 2 goes where chunk ch - 1 was: wait for its store
                        const int nb = (ch + kEpiBufs - 1) % kEpiBufs;
                        if (threadIdx.x == 0) {
                            bulk_wait_group_read<1>();
                            mbar_arrive_expect_tx(cfull0 + 8u * nb, kEpiChunkBytes);
                            tma_load_3d(epi_buf0 + nb * kEpiChunkBytes, &tmap_c, n0, mb + (kEpiBufs - 1) * CH,
                                        c.b, cfull0 + 8u * nb);
                        }
                        inflight |= 1u << nb;
                    }
                }
                if (!ok) break;
                release_acc(acc);
            } else if (c.nseg == 1) {
                // Chunks of CH accumulator columns (C rows): each chunk's C
                // loads are issued before its tensor-memory load and are in
                // flight together with it (C was requested into L2 while
                // the accumulator was being computed).
                static_assert(CH == 16, "the epilogue loads 16 columns at a time");
                const bool read_c = g.beta != 0.f;
                const bool n_ok = n < g.N;
                float *cbase = g.C + c.b * g.sC + static_cast<long long>(m0) * g.ldc + n;
#pragma unroll 1
                for (int ch = 0; ch < TM / CH; ++ch) {
                    const int mb = m0 + ch * CH;
                    float *cp = cbase + static_cast<long long>(ch * CH) * g.ldc;
                    float old[CH];
                    if (read_c) {
#pragma unroll
                        for (int j = 0; j < CH; ++j)
                            old[j] = (n_ok && mb + j < g.M && SG_IN_C(g, cp + j * g.ldc, 1)) ? cp[j * g.ldc] : 0.f;
                    }
                    float v[CH];
                    acc_chunk<TM>(t0 + ch * CH, v);
                    bool nan = false;
#pragma unroll
                    for (int j = 0; j < CH; ++j) nan |= v[j] != v[j];
                    if (nan && n_ok) {
                        // a non-finite input reached this chunk: exact dot products
#pragma unroll 1
                        for (int j = 0; j < CH; ++j)
                            if (v[j] != v[j] && mb + j < g.M) v[j] = recompute_dot<CONV, TRANS_B>(g, c.b, mb + j, n);
                    }
                    if (n_ok) {
                        if (read_c) {
#pragma unroll
                            for (int j = 0; j < CH; ++j)
                                if (mb + j < g.M && SG_IN_C(g, cp + j * g.ldc, 1))
                                    cp[j * g.ldc] = fmaf(g.beta, old[j], g.alpha * v[j]);
                        } else {
#pragma unroll
                            for (int j = 0; j < CH; ++j)
                                if (mb + j < g.M && SG_IN_C(g, cp + j * g.ldc, 1)) cp[j * g.ldc] = g.alpha * v[j];
                        }
                    }
                }
                release_acc(acc);
            } else if (ctl.ws == nullptr || ctl.counters == nullptr) {
                // a shared tile without a workspace: report, never dereference
                release_acc(acc);
                if (threadIdx.x == 0) atomicOr(ctl.status, kStatusNoWorkspace);
            } else {
                // shared tile: write this unit's partial tile, then the last
                // unit to arrive adds all partials in segment order.  Of a
                // pair, each CTA's half of the tile counts and sums on its
                // own: the tile's 2 nseg slots from 2 slot0 hold half r's
                // segments at 2 slot0 + r nseg, its counter is 2 tile + r.
                constexpr int kTileElems = kTileN * TM;
                const long long slot_first = PAIR ? 2 * c.slot0 + rank * c.nseg : c.slot0;
                const int counter = PAIR ? 2 * c.tile + rank : c.tile;
                float *wt = ctl.ws + (slot_first + c.seg) * kTileElems;
#pragma unroll 1
                for (int ch = 0; ch < TM / CH; ++ch) {
                    float v[CH];
                    acc_chunk<TM>(t0 + ch * CH, v);
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        if (SG_IN_WS(ctl, wt + (ch * CH + j) * kTileN + nl, 1)) __stcg(wt + (ch * CH + j) * kTileN + nl, v[j]);
                }
                release_acc(acc);
                __threadfence();
                named_bar_sync(kEpiBarrierId, kEpiWarps * 32);
                if (threadIdx.x == 0) {
                    // the last unit to arrive queues the tile's sum for the
                    // CTA's exit, where every warp of the CTA is free for it
                    const bool cnt_ok = !kDebugBounds || (counter >= 0 && counter < ctl.n_counters);
                    if (!cnt_ok) atomicOr(ctl.status, kStatusOutOfBounds);
                    const int prev = cnt_ok ? atomicAdd(ctl.counters + counter, 1) : -1;
                    if (prev == c.nseg - 1) {
                        ctl.counters[counter] = 0;
                        const int nd = *s_ndefer;
                        if (nd < kMaxDefer) {
                            s_defer[5 * nd + 0] = c.mt;
                            s_defer[5 * nd + 1] = ct;
                            s_defer[5 * nd + 2] = c.nseg;
                            s_defer[5 * nd + 3] = static_cast<int>(slot_first);
                            s_defer[5 * nd + 4] = c.b;
                            *s_ndefer = nd + 1;
                        } else {
                            atomicOr(ctl.status, kStatusDeferOverflow);
                        }
                    }
                }
            }
        }
        if (tma_c && threadIdx.x == 0) {
            // C stores finished and every C copy into shared memory landed
            // before the CTA may exit
            bulk_wait_group<0>();
            volatile int no_abort = 0;
            for (int b = 0; b < kEpiBufs; ++b)
                if (inflight & (1u << b))
                    mbar_wait_bounded(cfull0 + 8u * b, (cpar >> b) & 1u, &no_abort, ctl, kStatusTimeoutDrain);
        }
    } else if (warp < R::kMmaWarp) {
        // ------------------------------------------------------ producers
        // Group g fills the jobs (unit, k tile) q = g, g + G, g + 2G, ... of
        // this CTA (G = kGroups), job q into stage q % S.  kPrefetch register
        // buffers rotate: while one job is split and stored, the loads of the
        // group's next kPrefetch-1 jobs are in flight.
        constexpr int G = R::kGroups;
        constexpr int GT = R::kGroupThreads;
        constexpr int KB = R::kBtK;                  // B^T k values per thread and job
        constexpr int BtK = TMA_B ? 0 : KB;          // ... held in registers
        constexpr int AJ_ALL = (C::kAR * 4 + GT - 1) / GT;
        constexpr int AJ = TMA_A ? 0 : AJ_ALL;
        constexpr int NB = R::kPrefetch;
        const int group = (warp - kEpiWarps) / R::kWarpsPerGroup;
        const int gt = threadIdx.x - kEpiWarps * 32 - group * GT;  // thread index within the group
        int s = group;  // stage of the group's current job (q % S, with G <= S)
        uint32_t ph = 0;
        JobIter next;
        next.start(sch, walker);
        for (int i = 0; i < group && next.valid(sch); ++i) next.advance(sch);
        Raw<BtK, AJ> buf[NB];
        int loaded = 0, done = 0;
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            if (next.valid(sch)) {
                load_raw<TM, BtK, GT, AJ, CONV>(g, vec_a != 0, next.b, next.mt * TM, next.nt * kTileN, next.kt * kBK, gt,
                                          buf[i], ctab);
                for (int t = 0; t < G && next.valid(sch); ++t) next.advance(sch);
                ++loaded;
            }
        }
        // this warp's tensor-memory lanes hold the B^T columns of its threads
        const uint32_t ring_lane = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                                   static_cast<uint32_t>(C::kRingCol);
        bool ok = true;
#pragma unroll 1
        while (ok && done < loaded) {
#pragma unroll
            for (int i = 0; i < NB; ++i) {
                if (done < loaded) {
                    // warp-uniform decision: tcgen05.st below is warp-collective
                    bool w = mbar_wait_bounded(bars + 8u * (S + s), ph ^ 1u, abort_flag, ctl,
                                               kStatusTimeoutProducer);
                    if (R::kTma && w)
                        w = mbar_wait_bounded(afull0 + 8u * s, ph, abort_flag, ctl, kStatusTimeoutProducer);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    store_split<TM, TMA_B, KB, BtK, GT, AJ, AJ_ALL, TRANS_B, B4, PAIR>(
                        base + s * C::kAStageBytes, base + C::kOffBRegion + s * C::kBRawBytes,
                        ring_lane + static_cast<uint32_t>(s * kRingColsPerStage), gt, buf[i], b_offs);
                    // the lo tile was written to this CTA's own shared memory:
                    // the proxy fence orders it for the tensor core (of a pair,
                    // also for the even CTA's MMA, which reads it here)
                    fence_proxy_async_smem();
                    tmem_st_wait();
                    tc_fence_before();
                    const bool withhold =
                        done == 0 && group == 0 && gt == 0 && (ctl.debug_flags & kDebugWithholdArrive);
                    if constexpr (PAIR) {
                        // one arrive per warp, on the even CTA's barrier
                        __syncwarp();
                        if (lane == 0 && !withhold) mbar_arrive_cluster(lead_full0 + 8u * s);
                    } else {
                        if (!withhold) mbar_arrive(bars + 8u * s);
                    }
                    ++done;
                    s += G;
                    if (s >= S) {
                        s -= S;
                        ph ^= 1u;
                    }
                    if (next.valid(sch)) {
                        load_raw<TM, BtK, GT, AJ, CONV>(g, vec_a != 0, next.b, next.mt * TM, next.nt * kTileN, next.kt * kBK,
                                                  gt, buf[i], ctab);
                        for (int t = 0; t < G && next.valid(sch); ++t) next.advance(sch);
                        ++loaded;
                    }
                }
            }
        }
    } else if (R::kTma && warp == R::kTmaWarp) {
        // ------------------------------------------------------ TMA thread
        if (lane == 0) {
            if (TMA_A) prefetch_tmap(&tmap_a);
            if (TMA_B) prefetch_tmap(&tmap_b);
            if (B4) {
                prefetch_tmap(&tmap_b1);
                prefetch_tmap(&tmap_b2);
                prefetch_tmap(&tmap_b3);
            }
            constexpr uint32_t kTx =
                (TMA_A ? C::kAR * kBK * 4 : 0) + (TMA_B ? (B4 ? kBK * kB4RowBytes : kBK * kTileN * 4) : 0);
            int s = 0;
            uint32_t ph = 0;
            uint32_t used = 0, last_ph = 0;  // per stage: copy issued / its phase parity
            JobIter it;
            it.start(sch, walker);
            while (it.valid(sch)) {
                if (!mbar_wait_bounded(bars + 8u * (S + s), ph ^ 1u, abort_flag, ctl, kStatusTimeoutProducer))
                    break;
                mbar_arrive_expect_tx(afull0 + 8u * s, kTx);
                const uint32_t slab = base + C::kOffBRegion + s * C::kBRawBytes;
                const int bn = col_tile(it.nt) * kTileN;  // this CTA's first B column
                if (TMA_A)
                    tma_load_3d(base + s * C::kAStageBytes + C::kOffAHi, &tmap_a, it.kt * kBK,
                                it.mt * TM + rank * C::kAR, g.sA != 0 ? it.b : 0, afull0 + 8u * s);
                if (TMA_B && TRANS_B) {
                    tma_load_3d(slab, &tmap_b, it.kt * kBK, bn, g.sB != 0 ? it.b : 0, afull0 + 8u * s);
                } else if (TMA_B && B4) {
                    // rows k0 + 4i + r of the stage (i < 4) are rows 4 kt + i of class r
                    const CUtensorMap *maps[4] = {&tmap_b, &tmap_b1, &tmap_b2, &tmap_b3};
#pragma unroll
                    for (int r = 0; r < 4; ++r)
                        tma_load_3d(slab + r * kB4ClassBytes, maps[r], bn, it.kt * (kBK / 4),
                                    g.sB != 0 ? it.b : 0, afull0 + 8u * s);
                } else if (TMA_B) {
                    tma_load_3d(slab, &tmap_b, bn, it.kt * kBK, g.sB != 0 ? it.b : 0, afull0 + 8u * s);
                }
                used |= 1u << s;
                last_ph = (last_ph & ~(1u << s)) | (ph << s);
                it.advance(sch);
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // every copy this thread issued has landed before the CTA can exit
            volatile int no_abort = 0;
            for (int t = 0; t < S; ++t)
                if (used & (1u << t))
                    mbar_wait_bounded(afull0 + 8u * t, (last_ph >> t) & 1u, &no_abort, ctl, kStatusTimeoutDrain);
        }
    } else if (warp == R::kMmaWarp && lane == 0) {
        // ------------------------------------------------------ MMA issuer
        // Of a pair, the even CTA's thread issues the pair's MMAs and its
        // commits arrive on the barriers of both CTAs; the odd CTA's thread
        // only waits for the drain.
        if (!PAIR || rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            int it = 0;
            bool ok = true;
            auto commit = [&](uint32_t bar) {
                if constexpr (PAIR) mma_commit2(bar, 3);
                else mma_commit(bar);
            };
            auto mma = [&](uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
                if constexpr (PAIR) mma_tf32_ts2(d, a, b, idesc, accumulate);
                else mma_tf32_ts(d, a, b, idesc, accumulate);
            };
            UnitIter ui;
            for (ui.start(sch, walker); ui.ok && ok; ui.next(sch), ++it) {
                const UnitCoord &c = ui.c;
                const int acc = it % C::kNacc;
                const uint32_t aph = (it / C::kNacc) & 1;
                if (!mbar_wait_bounded<PAIR>(acc_empty0 + 8u * acc, aph ^ 1u, abort_flag, ctl, kStatusTimeoutMma)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
                for (int kt = c.kb; kt < c.ke; ++kt) {
                    if (!mbar_wait_bounded<PAIR>(bars + 8u * s, ph, abort_flag, ctl, kStatusTimeoutMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = base + s * C::kAStageBytes;
                    const uint32_t ring = tmem_base + static_cast<uint32_t>(C::kRingCol + s * kRingColsPerStage);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint32_t a_hi = ring + static_cast<uint32_t>(j * 8);
                        const uint32_t a_lo = a_hi + static_cast<uint32_t>(kBK);
                        const uint64_t b_hi = umma_desc_kmajor_sw64(st + C::kOffAHi + j * 32);
                        if constexpr (C::kPaired) {
                            // b_hi spans A_hi then A_lo: 2TM rows at the same pitch
                            mma(d, a_hi, b_hi, C::kIdescPair, (kt != c.kb || j != 0) ? 1u : 0u);
                            mma(d, a_lo, b_hi, C::kIdesc, 1u);
                        } else {
                            const uint64_t b_lo = umma_desc_kmajor_sw64(st + C::kOffALo + j * 32);
                            mma(d, a_lo, b_hi, C::kIdesc, (kt != c.kb || j != 0) ? 1u : 0u);
                            mma(d, a_hi, b_lo, C::kIdesc, 1u);
                            mma(d, a_hi, b_hi, C::kIdesc, 1u);
                        }
                    }
                    commit(bars + 8u * (S + s));
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                commit(acc_full0 + 8u * acc);
            }
            // every MMA this thread issued has finished once the drain arrives
            commit(drain_bar);
        }
        volatile int no_abort = 0;
        mbar_wait_bounded(drain_bar, 0u, &no_abort, ctl, kStatusTimeoutDrain);
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) {
        // both CTAs are done with the pair's tensor memory, shared memory and
        // barriers; the allocation is released by the pair together
        cluster_sync();
        if (warp == R::kMmaWarp) {
            tc_fence_after();
            tmem_dealloc2(tmem_base, kTmemCols);
        }
        cluster_sync();
    } else {
        if (warp == R::kMmaWarp) {
            tc_fence_after();
            tmem_dealloc(tmem_base, kTmemCols);
        }
    }
    // deferred sums of shared tiles, by every warp of the CTA
    const int nd = *s_ndefer;
    if (nd > 0 && !*abort_flag) {
        __threadfence();
#pragma unroll 1
        for (int e = 0; e < nd; ++e)
            fixup_tile<TM, CONV, TRANS_B>(g, ctl, s_defer[5 * e + 4], ctl.ws + static_cast<long long>(s_defer[5 * e + 3]) * (kTileN * TM),
                           s_defer[5 * e + 2], s_defer[5 * e] * TM, s_defer[5 * e + 1] * kTileN, warp,
                           R::kThreads / 32, lane);
    }
}

}  // namespace tf32x3
}  // namespace sg
