// C ABI of the library (declared in include/sgemm_gb300.h): argument
// checks, quick returns, the planner, library-owned device memory and the
// launches.  The problem statement is mysgemm(M,N,K,alpha,A,B,beta,C) of
// "NVIDIA_SGEMM_PRACTICE" (section "kernel 1") with leading dimensions; the
// pages' error handling (print and exit, "matmul_opt.cu" CHECK_CUDA_ERROR)
// is replaced by status codes: nothing here exits the process.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>

#include "sgemm_gb300.h"
#include "launch.h"

namespace {

using sg::DeviceCtl;
using sg::GemmArgs;
using sg::Schedule;

constexpr int kVersion = 100;              // 0.1.0
constexpr int kMaxDevices = 64;
constexpr long long kWaitBudget = 20000000000LL;  // ~10 s of SM clock: only a broken pipeline waits that long
constexpr long long kDebugWaitBudget = 2000000LL;  // ~1 ms, test-only withheld-arrive mode

struct Workspace {
    float *ws = nullptr;
    size_t ws_bytes = 0;
    int *counters = nullptr;
    size_t n_counters = 0;
    float *tr = nullptr;  // transposed operands of sgemm_t
    size_t tr_bytes = 0;
    float *ap = nullptr;  // A with rows padded to 16 bytes (3xTF32 path)
    size_t ap_bytes = 0;
};

constexpr int kHostMaxBlocks = 12;  // row (or column) blocks of a pipelined sgemm_host

// Sizes of the blocks a pipelined sgemm_host cuts `total` rows (or columns)
// into, in multiples of `quantum`: blocks of about total / 5 while more than
// two of them remain, then halving blocks down to two quanta.  The call's
// time is the upload of every block plus the last block's GEMM and its
// download, so the last blocks are made small; the first ones stay large
// enough for the GEMMs to keep up with the uploads.  Returns the count.
int host_blocks(int total, int quantum, int sizes[kHostMaxBlocks]) {
    const int big = std::max(quantum, (total / 5 + quantum - 1) / quantum * quantum);
    int n = 0, left = total;
    while (left > 0 && n < kHostMaxBlocks - 1) {
        int take;
        if (left > 2 * big) {
            take = big;
        } else {
            take = std::max(2 * quantum, (left / 2 + quantum - 1) / quantum * quantum);
            if (take >= left) take = left;
        }
        sizes[n++] = take;
        left -= take;
    }
    if (left > 0) sizes[n++] = left;
    return n;
}

struct HostBuffers {
    float *A = nullptr, *B = nullptr, *C = nullptr;
    size_t a_bytes = 0, b_bytes = 0, c_bytes = 0;
    cudaStream_t stream = nullptr;           // GEMMs
    cudaStream_t up = nullptr, down = nullptr;  // host->device and device->host copies
    cudaEvent_t b_in = nullptr, in[kHostMaxBlocks] = {}, out[kHostMaxBlocks] = {};
};

struct DevState {
    bool ready = false;
    int sms = 0;
    int pair_slots = 0;  // CTA pairs of the 3xTF32 pair form resident at once
    int major = 0, minor = 0;
    int *status = nullptr;
    std::map<cudaStream_t, Workspace> ws;
    HostBuffers host;
};

std::mutex g_mu;  // guards g_dev (setup, workspace growth, host buffers)
DevState g_dev[kMaxDevices];

// The device status word of sgemm / sgemm_ex / sgemm_t / the batched and
// convolution calls: a __device__ variable (one per GPU, zero when the
// library's device code is loaded), so that reading and clearing it in
// sgemm_check_status allocates nothing.  Host code reaches it only through
// the address cudaGetSymbolAddress gives for the current device.
__device__ int g_status_word;

int from_cuda(cudaError_t e) { return e == cudaSuccess ? 0 : static_cast<int>(e); }

// Initialise per-device state; caller holds g_mu.
int device_state(DevState **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e == cudaErrorNoDevice || e == cudaErrorInsufficientDriver
                                     ? SGEMM_ERR_NO_DEVICE : from_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_NO_DEVICE;
    DevState &d = g_dev[dev];
    if (!d.ready) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return from_cuda(e);
        d.major = prop.major;
        d.minor = prop.minor;
        d.sms = prop.multiProcessorCount;
        if (!(d.major == 10 && d.minor == 3)) return SGEMM_ERR_UNSUPPORTED_DEVICE;
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_status_word);
        if (e != cudaSuccess) return from_cuda(e);
        d.status = static_cast<int *>(p);
        d.pair_slots = sg::tf32x3_pair_slots();
        d.ready = true;
    }
    *out = &d;
    return 0;
}

// ------------------------------------------------------------------ planner

struct Plan {
    int path = 0;
    int tile_m = 0, tile_n = 0;
    Schedule sch{};
    int grid = 0;
    int stages = 0;
    int vec_a = 0, vec_b = 0, vec_c = 0;
    size_t ws_bytes = 0;
    bool wide = false;  // FFMA path: the wide-N kernel (A resident, B streamed)
};

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

bool aligned16(const void *p, long long ld) {
    return (reinterpret_cast<uintptr_t>(p) % 16u) == 0 && (ld % 4) == 0;
}

// K slices for a grid of `tiles` tiles on `slots` resident CTAs, keeping at
// least `min_kt` K tiles per slice.
int choose_splits(int tiles, int k_tiles, int slots, int splits_req, int min_kt) {
    if (splits_req > 0) return std::max(1, std::min(splits_req, k_tiles));
    if (tiles >= slots) return 1;
    int s = std::min(slots / std::max(tiles, 1), k_tiles / std::max(min_kt, 1));
    s = std::min(s, 16);
    return std::max(s, 1);
}

int forced_tile_rows(int flags) { return ((flags >> 8) & 0xFF) * 16; }

// Run-time model of the 3xTF32 kernel (microseconds), fitted to GB300
// measurements of square, ragged, K-heavy and wide shapes over every tile
// height and split count: a launch cost, per unit a fixed cost plus a cost
// per 16-deep K tile (both growing with the tile height), and for a shared
// tile a sum whose cost grows with its partial tiles.  Waves count the
// units of the busiest CTA, and CTA waves when there are more CTAs than SMs.
struct TileCost {
    double per_k_tile, per_unit, per_unit_c;  // per_unit_c: added when C is read (beta != 0)
};

TileCost tile_cost(int tm) {
    if (tm <= 64) return {0.302, 1.69, 0.0};
    if (tm <= 128) return {0.365, 2.43, 1.43};
    if (tm <= 192) return {0.391, 6.03, 0.0};
    return {0.431, 9.95, 0.44};
}

constexpr double kLaunchUs = 7.8;
constexpr double kSumUsPer256Rows = 0.93;  // per partial tile (and C) of a shared tile

struct Tf32x3Choice {
    int tm = 0, splits = 1, tail_splits = 0;
    double us = 0;
};

// Split-K (or whole tiles when s == 1) with tile height tm.
// A strided batch multiplies the tiles by its matrix count.
double model_split_k(int M, int N, int K, int tm, int s, int sms, bool read_c, long long batch = 1) {
    const TileCost c = tile_cost(tm);
    const double unit = c.per_unit + (read_c ? c.per_unit_c : 0.0);
    const long long tiles = static_cast<long long>(ceil_div(M, tm)) * ceil_div(N, sg::kTf32x3TileN) * batch;
    const int kt = ceil_div(std::max(K, 1), sg::kTf32x3BK);
    s = std::max(1, std::min(s, kt));
    const long long units = tiles * s;
    long long grid = std::min<long long>(units, sms);
    if (s > 1) grid = std::max(grid, (units + sg::kTf32x3MaxDefer - 1) / sg::kTf32x3MaxDefer);
    const long long waves = ((units + grid - 1) / grid) * ((grid + sms - 1) / sms);
    double us = kLaunchUs + waves * (ceil_div(kt, s) * c.per_k_tile + unit);
    if (s > 1) us += kSumUsPer256Rows * waves * (s + 1) * tm / 256.0;
    return us;
}

// Whole waves of whole tiles, then the leftover tiles in ts K slices each.
double model_split_tail(int M, int N, int K, int tm, int ts, int sms, bool read_c, long long batch = 1) {
    const TileCost c = tile_cost(tm);
    const double unit = c.per_unit + (read_c ? c.per_unit_c : 0.0);
    const long long tiles = static_cast<long long>(ceil_div(M, tm)) * ceil_div(N, sg::kTf32x3TileN) * batch;
    const int kt = ceil_div(std::max(K, 1), sg::kTf32x3BK);
    const long long waves = tiles / sms;
    return kLaunchUs + waves * (kt * c.per_k_tile + unit) + ceil_div(kt, ts) * c.per_k_tile + unit +
           kSumUsPer256Rows * (ts + 1) * tm / 256.0;
}

// K slices per leftover tile of a split tail (0: no split tail possible).
int tail_splits_for(long long tiles, int kt, int sms) {
    const long long rem = tiles % sms;
    if (tiles < sms || rem == 0) return 0;
    const int ts = static_cast<int>(std::min<long long>(sms / rem, kt / 8));
    return ts >= 2 ? ts : 0;
}

// Tile heights the planner may use for M rows: the smallest supported height
// that covers M (at most 256) and, for M > 64, the lower ones from 64 up.
int tm_candidates(int M, int out[6]) {
    static const int kAll[] = {16, 32, 64, 128, 192, 256};
    int cover = 256;
    for (int tm : kAll)
        if (tm >= M) { cover = tm; break; }
    int n = 0;
    if (cover <= 64) {
        out[n++] = cover;
    } else {
        for (int tm : kAll)
            if (tm >= 64 && tm <= cover) out[n++] = tm;
    }
    return n;
}

Tf32x3Choice choose_tf32x3(int M, int N, int K, int sms, int forced_tm, int splits_req, int flags, bool read_c,
                           long long batch = 1) {
    int tms[6];
    int ntm = forced_tm > 0 ? (tms[0] = forced_tm, 1) : tm_candidates(M, tms);
    const int kt = ceil_div(std::max(K, 1), sg::kTf32x3BK);
    Tf32x3Choice best, best_tail;
    best.us = best_tail.us = 1e300;
    for (int i = 0; i < ntm; ++i) {
        const int tm = tms[i];
        const long long tiles = static_cast<long long>(ceil_div(M, tm)) * ceil_div(N, sg::kTf32x3TileN) * batch;
        if (splits_req > 0) {
            const int s = std::max(1, std::min(splits_req, kt));
            const double us = model_split_k(M, N, K, tm, s, sms, read_c, batch);
            if (us < best.us) best = {tm, s, 0, us};
            continue;
        }
        // split-K: at least 4 K tiles per slice, at most 16 slices, and
        // only while the slices still fit in one wave
        for (int s = 1; s <= 16; ++s) {
            if (s > 1 && (kt / s < 4 || tiles * s > sms)) break;
            const double us = model_split_k(M, N, K, tm, s, sms, read_c, batch);
            if (us < best.us) best = {tm, s, 0, us};
        }
        if (!(flags & SGEMM_FLAG_WHOLE_TILES)) {
            const int ts = tail_splits_for(tiles, kt, sms);
            if (ts > 0) {
                const double us = model_split_tail(M, N, K, tm, ts, sms, read_c, batch);
                if (us < best.us) best = {tm, 1, ts, us};
                if (us < best_tail.us) best_tail = {tm, 1, ts, us};
            }
        }
    }
    // SPLIT_TAIL: the fastest plan that has a split tail, if any has one
    if ((flags & SGEMM_FLAG_SPLIT_TAIL) && !(flags & SGEMM_FLAG_WHOLE_TILES) && best_tail.tm > 0) return best_tail;
    return best;
}

// Run-time model of the CTA-pair form: a 256 x 256 tile over two SMs costs
// kPairKTile times the single-CTA 256-row tile per K tile and kPairUnitUs
// more per unit; tiles of 256 columns are walked by `slots` pairs.  Least-
// squares fit to GB300 kernel times of 21 shapes from 2560 x 2560 x 1024
// to 12288^3 (each within 6 %, most within 2 %).  *tail: the split-tail
// schedule is the faster one (K slices per leftover tile from
// tail_splits_for).
constexpr double kPairKTile = 0.94;
constexpr double kPairUnitUs = 0.5;

double model_pairs(int M, int N, int K, int tm, int slots, bool read_c, long long batch, int flags, bool *tail) {
    const TileCost c = tile_cost(tm);
    const double unit = c.per_unit + (read_c ? c.per_unit_c : 0.0) + kPairUnitUs;
    const double per_k = c.per_k_tile * kPairKTile;
    const long long tiles = static_cast<long long>(ceil_div(M, tm)) * ceil_div(N, 2 * sg::kTf32x3TileN) * batch;
    const int kt = ceil_div(std::max(K, 1), sg::kTf32x3BK);
    const double whole = kLaunchUs + static_cast<double>((tiles + slots - 1) / slots) * (kt * per_k + unit);
    *tail = false;
    if (flags & SGEMM_FLAG_WHOLE_TILES) return whole;
    const int ts = tail_splits_for(tiles, kt, slots);
    if (ts == 0) return whole;
    const double split = kLaunchUs + static_cast<double>(tiles / slots) * (kt * per_k + unit) +
                         ceil_div(kt, ts) * per_k + unit + kSumUsPer256Rows * (ts + 1) * tm / 256.0;
    if (split < whole || (flags & SGEMM_FLAG_SPLIT_TAIL)) {
        *tail = true;
        return split;
    }
    return whole;
}

// A tile of 192 or 256 rows on CTA pairs (SGEMM_FLAG_PAIRS): tiles of 256
// columns walked by `slots` pairs (the pairs resident at once), each pair
// two CTAs of the grid.  Whole waves of tiles plus a split tail, or split-K
// when a split count is forced.  Counters: two per tile (one per CTA half).
void plan_pairs(int M, int N, int K, int tm, int slots, int splits_req, int flags, bool read_c, Plan &p, int batch) {
    constexpr int kPairN = 2 * sg::kTf32x3TileN;
    p.tile_m = tm;
    p.tile_n = kPairN;
    Schedule &s = p.sch;
    s = Schedule{};
    s.pair_shift = 1;
    s.m_tiles = ceil_div(M, tm);
    s.n_tiles = ceil_div(N, kPairN);
    s.k_tiles = ceil_div(K, sg::kTf32x3BK);
    s.tpb = batch > 1 ? s.m_tiles * s.n_tiles : 0;
    const int tiles = s.m_tiles * s.n_tiles * batch;
    s.splits = splits_req > 0 ? std::max(1, std::min(splits_req, s.k_tiles)) : 1;
    s.units = tiles * s.splits;
    s.group_m = std::min(8, s.m_tiles);
    int walkers = std::min(s.units, slots);
    // a CTA finishes at most kTf32x3MaxDefer shared tiles (one half each)
    if (s.splits > 1) walkers = std::max(walkers, ceil_div(s.units, sg::kTf32x3MaxDefer));
    p.grid = 2 * walkers;
    p.stages = sg::tf32x3_stages(tm, true);
    const size_t tile_bytes = static_cast<size_t>(kPairN) * tm * sizeof(float);
    p.ws_bytes = s.splits > 1 ? static_cast<size_t>(s.units) * tile_bytes : 0;
    bool tail = false;
    if (s.splits == 1) model_pairs(M, N, K, tm, slots, read_c, batch, flags, &tail);
    const int ts = tail ? tail_splits_for(tiles, s.k_tiles, slots) : 0;
    if (ts > 0) {
        const int rem = tiles % slots;
        s.dp_tiles = tiles - rem;
        s.tail_tiles = rem;
        s.tail_splits = ts;
        p.grid = 2 * slots;
        p.ws_bytes = static_cast<size_t>(rem) * ts * tile_bytes;
    }
}

// Whether a tile of tm rows runs on CTA pairs, given the single-CTA plan
// (split count and estimated time).  SGEMM_FLAG_PAIRS forces them for tiles
// of 192 or 256 rows; otherwise 256-row plans without split-K take them when
// the model above estimates them faster.  Measured on GB300 (TF/s, single
// CTAs -> pairs): 4096^3 311 -> 330, 5120^3 321 -> 342, 8192^3 349 -> 374,
// 12288^3 343 -> 380, 3000^3 283 -> 302, 2304 x 2304 x 8192 297 -> 314,
// 256 x 50176 x 1024 206 -> 223; the model keeps single CTAs where they win
// clearly: 10000 x 600 x 3000 254 against 204 (N padded to 256-column tiles,
// 1.6 waves).  It misjudges near-ties: 2560 x 2560 x 1024 runs on pairs at
// 197 against 203, 512 x 20000 x 1024 at 198 against 200.
// Where the single-CTA plan splits K to fill the SMs, pairs (half as many
// tiles) lose: 1536^3 174 -> 130, 1024^3 57-61 against 73.  Tiles of 192
// rows gained nothing (384 x 14161 x 1152: 178 both).
bool use_pairs(int M, int N, int K, const Tf32x3Choice &ch, int flags, int pair_slots, bool read_c,
               long long batch) {
    if (pair_slots <= 0 || (flags & SGEMM_FLAG_NO_PAIRS) || !sg::tf32x3_pair_tm(ch.tm)) return false;
    if (flags & SGEMM_FLAG_PAIRS) return true;
    if (ch.tm != 256 || ch.splits != 1) return false;
    bool tail = false;
    return model_pairs(M, N, K, ch.tm, pair_slots, read_c, batch, flags, &tail) < ch.us;
}

// batch > 1: one launch over the tiles of every matrix (Schedule::tpb).
// pair_slots > 0: CTA pairs are possible for this call (operands copied by
// TMA) and that many fit on the device (use_pairs decides).
void plan_tf32x3(int M, int N, int K, int sms, int splits_req, int flags, bool read_c, Plan &p, int batch = 1,
                 int pair_slots = 0) {
    p.path = SGEMM_ALGO_TF32X3;
    const Tf32x3Choice ch = choose_tf32x3(M, N, K, sms, forced_tile_rows(flags), splits_req, flags, read_c, batch);
    const int tm = ch.tm;
    if (use_pairs(M, N, K, ch, flags, pair_slots, read_c, batch)) {
        plan_pairs(M, N, K, tm, pair_slots, splits_req, flags, read_c, p, batch);
        return;
    }
    p.tile_m = tm;
    p.tile_n = sg::kTf32x3TileN;
    Schedule &s = p.sch;
    s.m_tiles = ceil_div(M, tm);
    s.n_tiles = ceil_div(N, p.tile_n);
    s.k_tiles = ceil_div(K, sg::kTf32x3BK);
    s.tpb = batch > 1 ? s.m_tiles * s.n_tiles : 0;
    const int tiles = s.m_tiles * s.n_tiles * batch;
    s.splits = ch.splits;
    s.units = tiles * s.splits;
    s.group_m = std::min(8, s.m_tiles);
    p.grid = std::min(s.units, sms);
    // a CTA finishes at most kTf32x3MaxDefer shared tiles: with more units
    // than that per SM (forced split counts), run more CTAs than SMs
    if (s.splits > 1) p.grid = std::max(p.grid, ceil_div(s.units, sg::kTf32x3MaxDefer));
    p.stages = sg::tf32x3_stages(tm);
    p.ws_bytes = s.splits > 1 ? static_cast<size_t>(s.units) * p.tile_n * tm * sizeof(float) : 0;
    if (ch.tail_splits > 0) {
        // whole waves keep whole tiles; the leftover tiles are cut into K
        // slices so that the last wave keeps (almost) every SM busy
        const int rem = tiles % sms;
        s.dp_tiles = tiles - rem;
        s.tail_tiles = rem;
        s.tail_splits = ch.tail_splits;
        p.grid = sms;
        p.ws_bytes = static_cast<size_t>(rem) * ch.tail_splits * p.tile_n * tm * sizeof(float);
    }
}

// The wide-N kernel takes short, shallow A (M <= 32, K <= 64) on the FFMA
// path unless a split count is forced.  AUTO sends it the shapes where it
// beats the tensor path's narrow tiles, measured at M = 32, N = 1.6 M:
// K = 28 98 vs 189 us, K = 32 107 vs 137, K = 48 149 vs 151, K = 64 191 vs
// 181; streaming B and C needs only part of the CUDA cores there.
constexpr int kWideAutoMaxK = 48;
bool use_wide(int M, int K, int splits_req) { return splits_req <= 1 && sg::ffma_wide_fits(M, K); }
bool auto_wide(int M, int K, int splits_req) { return use_wide(M, K, splits_req) && K <= kWideAutoMaxK; }

void plan_ffma(int M, int N, int K, int sms, int splits_req, Plan &p) {
    p.path = SGEMM_ALGO_FFMA;
    if (use_wide(M, K, splits_req)) {
        p.wide = true;
        p.tile_m = 32;
        p.tile_n = 512;
        Schedule &s = p.sch;
        s.m_tiles = 1;
        s.n_tiles = sg::ffma_wide_blocks(N);
        s.k_tiles = ceil_div(K, sg::kFfmaBK);
        s.splits = 1;
        s.units = s.n_tiles;
        s.group_m = 1;
        p.grid = std::min(s.units, 2 * sms);
        p.stages = 3;
        p.ws_bytes = 0;
        return;
    }
    // 128 x 256 tiles, one CTA per SM, when they fill at least 80 % of a
    // wave; else 128 x 128 (two CTAs per SM), or wide tiles for short A
    const bool big = M > 64 && static_cast<long long>(ceil_div(M, 128)) * ceil_div(N, 256) * 5 >= 4LL * sms;
    if (M <= 32) { p.tile_m = 32; p.tile_n = 512; }
    else if (M <= 64) { p.tile_m = 64; p.tile_n = 256; }
    else if (big) { p.tile_m = 128; p.tile_n = 256; }
    else { p.tile_m = 128; p.tile_n = 128; }
    Schedule &s = p.sch;
    s.m_tiles = ceil_div(M, p.tile_m);
    s.n_tiles = ceil_div(N, p.tile_n);
    s.k_tiles = ceil_div(K, sg::kFfmaBK);
    const int tiles = s.m_tiles * s.n_tiles;
    s.splits = choose_splits(tiles, s.k_tiles, big ? sms : 2 * sms, splits_req, 4);
    s.units = tiles * s.splits;
    s.group_m = std::min(8, s.m_tiles);
    p.grid = s.units;
    p.stages = sg::ffma_stages(p.tile_m, p.tile_n);
    p.ws_bytes = s.splits > 1
                     ? static_cast<size_t>(s.units) * p.tile_m * p.tile_n * sizeof(float) : 0;
    // 128 x 256 tiles beyond whole waves: the leftover tiles of the partly
    // empty last wave are cut into K slices (each at least 8 K tiles), so
    // that the last wave is short instead of mostly idle
    const int ts = big && splits_req == 0 ? tail_splits_for(tiles, s.k_tiles, sms) : 0;
    if (ts > 0) {
        const int rem = tiles % sms;
        s.splits = 1;
        s.dp_tiles = tiles - rem;
        s.tail_tiles = rem;
        s.tail_splits = ts;
        s.units = s.dp_tiles + rem * ts;
        p.grid = s.units;
        p.ws_bytes = static_cast<size_t>(rem) * ts * p.tile_m * p.tile_n * sizeof(float);
    }
}

// The path AUTO takes: the tensor path, except for the shapes the wide-N
// FFMA kernel streams.
int resolve_path(int M, int K, int algo, int splits) {
    return (algo == SGEMM_ALGO_AUTO) ? (auto_wide(M, K, splits) ? SGEMM_ALGO_FFMA : SGEMM_ALGO_TF32X3) : algo;
}

// batch > 1 (3xTF32 path only): matrix b of each operand starts b * stride
// elements after the first; 16-byte copies need 16-byte strides too.
// Whether run() copies an A whose rows are not 16-byte aligned into aligned
// rows before the 3xTF32 kernel (then its tiles come by TMA): A far smaller
// than B (M * 32 <= N, the im2col shapes), one matrix or one shared by the
// batch, unless SGEMM_FLAG_NO_A_COPY.
bool a_gets_staged(int M, int N, int flags, int batch, long long sA) {
    return !(flags & SGEMM_FLAG_NO_A_COPY) && (batch <= 1 || sA == 0) && static_cast<long long>(M) * 32 <= N;
}

// pair_slots: CTA pairs the device holds at once (0: no pair form).
int make_plan(int M, int N, int K, const void *A, int lda, const void *B, int ldb, const void *C, int ldc,
              int algo, int splits, int flags, int sms, bool read_c, Plan &p, int batch = 1, long long sA = 0,
              long long sB = 0, long long sC = 0, int pair_slots = 0) {
    const int path = resolve_path(M, K, algo, splits);
    if (batch > 1 && path != SGEMM_ALGO_TF32X3) return SGEMM_ERR_INTERNAL;
    const bool va = aligned16(A, lda) && sA % 4 == 0;
    const bool vb = aligned16(B, ldb) && sB % 4 == 0;
    // the pair form copies A and B by TMA: B's rows aligned, or an aligned
    // start with whole residue classes (K >= 4, batch stride of 4 floats)
    const bool b_tma = vb || ((reinterpret_cast<uintptr_t>(B) & 15u) == 0 && K >= 4 && sB % 4 == 0 &&
                              !(flags & SGEMM_FLAG_B_ROWS_LOADED));
    // an unaligned A that run() stages into aligned rows comes by TMA too
    const bool a_staged = !va && a_gets_staged(M, N, flags, batch, sA);
    const int slots = ((va || a_staged) && b_tma) ? pair_slots : 0;
    if (path == SGEMM_ALGO_TF32X3) plan_tf32x3(M, N, K, sms, splits, flags, read_c, p, batch, slots);
    else plan_ffma(M, N, K, sms, splits, p);
    p.vec_a = va;
    p.vec_b = vb;
    p.vec_c = aligned16(C, ldc) && sC % 4 == 0;
    // the wide kernel's bulk-copy form runs one CTA per SM
    if (p.wide && p.vec_b && N % 4 == 0) p.grid = std::min(p.sch.units, sms);
    if (p.sch.units <= 0 || p.grid <= 0) return SGEMM_ERR_INTERNAL;
    return 0;
}

// --------------------------------------------------------- argument checks

bool overlaps(const void *a, size_t a_bytes, const void *b, size_t b_bytes) {
    if (!a || !b || a_bytes == 0 || b_bytes == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_bytes && b0 < a0 + a_bytes;
}

size_t span_bytes(int rows, int cols, long long ld) {
    if (rows <= 0 || cols <= 0) return 0;
    return static_cast<size_t>((static_cast<long long>(rows) - 1) * ld + cols) * sizeof(float);
}

bool flags_valid(int flags) {
    if (flags & ~(SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE | SGEMM_FLAG_WHOLE_TILES | SGEMM_FLAG_SPLIT_TAIL | 0xFF00 |
                  SGEMM_FLAG_NO_A_COPY | SGEMM_FLAG_B_ROWS_LOADED | SGEMM_FLAG_PAIRS | SGEMM_FLAG_NO_PAIRS))
        return false;
    const int tm = forced_tile_rows(flags);
    return tm == 0 || sg::tf32x3_supported_tm(tm);
}

int check_args(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
               float *C, int ldc, int algo, int splits, int flags) {
    (void)beta;
    if (M < 0) return -1;
    if (N < 0) return -2;
    if (K < 0) return -3;
    if (lda < std::max(1, K)) return -6;
    if (ldb < std::max(1, N)) return -8;
    if (ldc < std::max(1, N)) return -11;
    if (algo < SGEMM_ALGO_AUTO || algo > SGEMM_ALGO_TF32X3) return -13;
    if (splits < 0) return -14;
    if (!flags_valid(flags)) return -15;
    if (M == 0 || N == 0) return 0;
    const bool use_ab = alpha != 0.f && K > 0;
    if (use_ab && A == nullptr) return -5;
    if (use_ab && B == nullptr) return -7;
    if (C == nullptr) return -10;
    const size_t c_bytes = span_bytes(M, N, ldc);
    if (use_ab && (overlaps(C, c_bytes, A, span_bytes(M, K, lda)) ||
                   overlaps(C, c_bytes, B, span_bytes(K, N, ldb))))
        return -10;
    return 0;
}

// Grow the split-K workspace of (device, stream); caller holds g_mu.
int get_workspace(DevState &d, cudaStream_t stream, size_t bytes, size_t counters, Workspace **out) {
    Workspace &w = d.ws[stream];
    if (w.ws_bytes < bytes) {
        if (w.ws) {
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return from_cuda(e);
            cudaFree(w.ws);
            w.ws = nullptr;
            w.ws_bytes = 0;
        }
        if (cudaMalloc(reinterpret_cast<void **>(&w.ws), bytes) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_WORKSPACE;
        }
        w.ws_bytes = bytes;
    }
    if (w.n_counters < counters) {
        const size_t n = std::max<size_t>(counters, 1024);
        if (w.counters) {
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return from_cuda(e);
            cudaFree(w.counters);
            w.counters = nullptr;
            w.n_counters = 0;
        }
        if (cudaMalloc(reinterpret_cast<void **>(&w.counters), n * sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_WORKSPACE;
        }
        cudaError_t e = cudaMemsetAsync(w.counters, 0, n * sizeof(int), stream);
        if (e != cudaSuccess) return from_cuda(e);
        w.n_counters = n;
    }
    *out = &w;
    return 0;
}

// Room for transposed copies of the operands, grown like the split-K
// workspace (after the stream's earlier work is done with the old buffer).
int get_transpose_ws(DevState &d, cudaStream_t stream, size_t bytes, float **out) {
    Workspace &w = d.ws[stream];
    if (w.tr_bytes < bytes) {
        if (w.tr) {
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return from_cuda(e);
            cudaFree(w.tr);
            w.tr = nullptr;
            w.tr_bytes = 0;
        }
        if (cudaMalloc(reinterpret_cast<void **>(&w.tr), bytes) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_WORKSPACE;
        }
        w.tr_bytes = bytes;
    }
    *out = w.tr;
    return 0;
}

// batch > 1: a strided batch in one launch of the 3xTF32 kernel (the caller
// has checked the strides and that the path is the tensor path).
// trans_b: B is stored N x K (ldb >= K) and read in place by the 3xTF32
// kernel's transposed-B form; the caller has checked the arguments, chosen
// the tensor path, and made sure A and B are 16-byte aligned.
// A per-stream buffer for a padded copy of A (grown like the transpose buffer).
int get_apad_ws(DevState &d, cudaStream_t stream, size_t bytes, float **out) {
    Workspace &w = d.ws[stream];
    if (w.ap_bytes < bytes) {
        if (w.ap) {
            cudaError_t e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return from_cuda(e);
            cudaFree(w.ap);
            w.ap = nullptr;
            w.ap_bytes = 0;
        }
        if (cudaMalloc(reinterpret_cast<void **>(&w.ap), bytes) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_WORKSPACE;
        }
        w.ap_bytes = bytes;
    }
    *out = w.ap;
    return 0;
}

int run(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
        float *C, int ldc, cudaStream_t stream, int algo, int splits, int flags, int batch = 1, long long sA = 0,
        long long sB = 0, long long sC = 0, bool trans_b = false) {
    int rc = trans_b ? 0 : check_args(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, algo, splits, flags);
    if (rc != 0) return rc;
    if (M == 0 || N == 0) return 0;

    DevState *d = nullptr;
    DeviceCtl ctl{};
    Plan p;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        rc = device_state(&d);
        if (rc != 0) return rc;
        if (alpha == 0.f || K == 0) {
            if (beta == 1.f) return 0;
            return from_cuda(sg::scale_c_launch(C, ldc, M, N, beta, d->sms, stream));
        }
        rc = make_plan(M, N, K, A, lda, B, ldb, C, ldc, algo, splits, flags, d->sms, beta != 0.f, p, batch, sA, sB,
                       sC, trans_b ? 0 : d->pair_slots);
        if (rc != 0) return rc;
        ctl.status = d->status;
        ctl.wait_budget = (flags & SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE) ? kDebugWaitBudget : kWaitBudget;
        ctl.debug_flags = (flags & SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE) ? sg::kDebugWithholdArrive : 0;
        if (p.ws_bytes > 0) {  // split-K or split tail: tiles shared by several units
            Workspace *w = nullptr;
            rc = get_workspace(*d, stream, p.ws_bytes,
                               static_cast<size_t>(p.sch.m_tiles) * p.sch.n_tiles * std::max(batch, 1)
                                   << p.sch.pair_shift, &w);
            if (rc != 0) return rc;
            ctl.ws = w->ws;
            ctl.counters = w->counters;
            ctl.ws_end = w->ws + p.ws_bytes / sizeof(float);
            ctl.n_counters = static_cast<long long>(w->n_counters);
        }
        // A whose rows are not 16-byte aligned (one matrix, or one shared by
        // the batch) and that is far smaller than B (M * 32 <= N, the im2col
        // shapes: every column tile re-reads it) is copied once into rows
        // padded to 4 floats, so that the 3xTF32 kernel copies its tiles by
        // TMA: 12 producer warps with 96 registers instead of 16 loading A
        // themselves with 80.  Measured: 64 x 1605632 x 147 from 74.7 to
        // 90.0 TF/s; at 1023 x 1021 x 1025 the copy cost more than it saved.
        // The two forms give the same bits.
        if (p.path == SGEMM_ALGO_TF32X3 && !p.vec_a && a_gets_staged(M, N, flags, batch, sA)) {
            const int K4 = (K + 3) / 4 * 4;
            float *apad = nullptr;
            rc = get_apad_ws(*d, stream, static_cast<size_t>(M) * K4 * sizeof(float), &apad);
            if (rc != 0) return rc;
            cudaError_t e = cudaMemcpy2DAsync(apad, static_cast<size_t>(K4) * sizeof(float), A,
                                              static_cast<size_t>(lda) * sizeof(float), static_cast<size_t>(K) * sizeof(float),
                                              static_cast<size_t>(M), cudaMemcpyDeviceToDevice, stream);
            if (e != cudaSuccess) return from_cuda(e);
            A = apad;
            lda = K4;
            p.vec_a = 1;
        }
    }
    GemmArgs g{M, N, K, alpha, beta, A, lda, B, ldb, C, ldc, sA, sB, sC};
    sg::set_extents(g, batch, trans_b, ctl.status);
    cudaError_t e;
    if (trans_b && (p.path != SGEMM_ALGO_TF32X3 || !p.vec_a || !p.vec_b))
        return SGEMM_ERR_INTERNAL;
    if (trans_b)
        e = sg::tf32x3_launch_tb(p.tile_m, g, p.sch, ctl, p.vec_a, p.vec_c, p.grid, stream, batch);
    else if (p.path == SGEMM_ALGO_TF32X3)
        e = sg::tf32x3_launch(p.tile_m, g, p.sch, ctl, p.vec_a, p.vec_b, p.vec_c, p.grid, stream, batch,
                              (flags & SGEMM_FLAG_B_ROWS_LOADED) != 0);
    else if (p.wide)
        e = sg::ffma_wide_launch(g, p.vec_b, p.grid, stream, sg::kConvNone, &ctl);
    else
        e = sg::ffma_launch(p.tile_m, p.tile_n, g, p.sch, ctl, p.vec_a, p.vec_b, p.vec_c, stream);
    return from_cuda(e);
}

// op(X) = X or X^T (BLAS transa / transb, row-major storage): with transa
// A is stored K x M (lda >= M), with transb B is stored N x K (ldb >= K).
// A transposed operand is first copied, transposed, into a workspace of this
// stream; then the planned GEMM runs on the copies.  Returns 0 or -i, i the
// position of the offending argument in sgemm_t.
int check_t(int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
            int ldb, const float *C, int ldc, int algo) {
    if (transa != 0 && transa != 1) return -1;
    if (transb != 0 && transb != 1) return -2;
    if (M < 0) return -3;
    if (N < 0) return -4;
    if (K < 0) return -5;
    if (lda < std::max(1, transa ? M : K)) return -8;
    if (ldb < std::max(1, transb ? K : N)) return -10;
    if (ldc < std::max(1, N)) return -13;
    if (algo != SGEMM_ALGO_AUTO && algo != SGEMM_ALGO_FFMA && algo != SGEMM_ALGO_TF32X3) return -15;
    if (M == 0 || N == 0) return 0;
    const bool use_ab = alpha != 0.f && K > 0;
    if (use_ab && A == nullptr) return -7;
    if (use_ab && B == nullptr) return -9;
    if (C == nullptr) return -12;
    const size_t c_bytes = span_bytes(M, N, ldc);
    if (use_ab && (overlaps(C, c_bytes, A, transa ? span_bytes(K, M, lda) : span_bytes(M, K, lda)) ||
                   overlaps(C, c_bytes, B, transb ? span_bytes(N, K, ldb) : span_bytes(K, N, ldb))))
        return -12;
    return 0;
}

int run_t(int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
          int ldb, float beta, float *C, int ldc, cudaStream_t stream, int algo) {
    int rc0 = check_t(transa, transb, M, N, K, alpha, A, lda, B, ldb, C, ldc, algo);
    if (rc0 != 0 || M == 0 || N == 0) return rc0;
    const bool use_ab = alpha != 0.f && K > 0;
    if (!use_ab)  // C = beta * C; A and B are not read
        return run(M, N, K, alpha, nullptr, std::max(1, K), nullptr, std::max(1, N), beta, C, ldc, stream, algo, 0, 0);
    if (!transa && !transb) return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, algo, 0, 0);
    // A transposed B is read in place (the kernel's transposed-B form) on the
    // tensor path when B and A (or A's transposed copy) are 16-byte aligned;
    // otherwise it is copied.  Copies: A^T at offset 0 in rows of K rounded
    // up to 4 floats (16-byte aligned rows), B^T after it on a 256-byte
    // boundary in rows of N rounded up to 4.
    const int K4 = (K + 3) / 4 * 4, N4 = (N + 3) / 4 * 4;
    const bool fuse_b = transb && resolve_path(M, K, algo, 0) == SGEMM_ALGO_TF32X3 && aligned16(B, ldb) &&
                        (transa || aligned16(A, lda));
    if (fuse_b && !transa)
        return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, algo, 0, 0, 1, 0, 0, 0, true);
    const size_t a_floats = transa ? static_cast<size_t>(M) * K4 : 0;
    const size_t b_off = (a_floats + 63) / 64 * 64;
    const size_t floats = b_off + ((transb && !fuse_b) ? static_cast<size_t>(K) * N4 : 0);
    float *ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DevState *d = nullptr;
        int rc = device_state(&d);
        if (rc != 0) return rc;
        rc = get_transpose_ws(*d, stream, floats * sizeof(float), &ws);
        if (rc != 0) return rc;
    }
    cudaError_t e = cudaSuccess;
    if (transa) e = sg::transpose_launch(A, lda, K, M, ws, K4, stream);  // K x M -> M x K
    if (e == cudaSuccess && transb && !fuse_b)
        e = sg::transpose_launch(B, ldb, N, K, ws + b_off, N4, stream);  // N x K -> K x N
    if (e != cudaSuccess) return from_cuda(e);
    if (fuse_b)
        return run(M, N, K, alpha, ws, K4, B, ldb, beta, C, ldc, stream, algo, 0, 0, 1, 0, 0, 0, true);
    return run(M, N, K, alpha, transa ? ws : A, transa ? K4 : lda, transb ? ws + b_off : B, transb ? N4 : ldb,
               beta, C, ldc, stream, algo, 0, 0);
}

// One launch for a whole strided batch on the 3xTF32 path: transposed
// operands are first copied, transposed, matrix by matrix into this stream's
// workspace.  Returns 1 where the batch has to run matrix by matrix: the FFMA
// path, alpha = 0 or K = 0, more tiles than the schedule's 32-bit unit index
// holds, or C's matrices overlapping A's or B's (each matrix is then checked
// on its own); else 0 or -i as run_t.
int run_batched_one_launch(int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda,
                           long long sA, const float *B, int ldb, long long sB, float beta, float *C, int ldc,
                           long long sC, int batch, cudaStream_t stream, int algo) {
    if (alpha == 0.f || K == 0 || resolve_path(M, K, algo, 0) != SGEMM_ALGO_TF32X3) return 1;
    // units: at most 16 K slices of tiles 16 rows high
    if (static_cast<long long>(ceil_div(M, 16)) * ceil_div(N, sg::kTf32x3TileN) * batch * 16 > INT32_MAX) return 1;
    const long long nA = sA ? batch : 1, nB = sB ? batch : 1;
    const size_t a_span = (nA - 1) * sA * sizeof(float) + (transa ? span_bytes(K, M, lda) : span_bytes(M, K, lda));
    const size_t b_span = (nB - 1) * sB * sizeof(float) + (transb ? span_bytes(N, K, ldb) : span_bytes(K, N, ldb));
    const size_t c_span = (batch - 1) * sC * sizeof(float) + span_bytes(M, N, ldc);
    if (overlaps(C, c_span, A, a_span) || overlaps(C, c_span, B, b_span)) return 1;
    if (!transa && !transb)
        return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, algo, 0, 0, batch, sA, sB, sC);
    // a transposed B is read in place when B and A (or A's copy) are 16-byte
    // aligned, batch strides included (as in run_t)
    const bool fuse_b = transb && aligned16(B, ldb) && sB % 4 == 0 && (transa || (aligned16(A, lda) && sA % 4 == 0));
    // transposed copies, each matrix on a 256-byte boundary, rows rounded up
    // to 4 floats: A^T (M x K) first, then B^T (K x N)
    const int K4 = (K + 3) / 4 * 4, N4 = (N + 3) / 4 * 4;
    const long long a_str = transa ? (static_cast<long long>(M) * K4 + 63) / 64 * 64 : 0;
    const long long b_str = (transb && !fuse_b) ? (static_cast<long long>(K) * N4 + 63) / 64 * 64 : 0;
    const long long b_off = a_str * (transa ? nA : 0);
    if (fuse_b && !transa)
        return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream, algo, 0, 0, batch, sA, sB, sC, true);
    float *ws = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        DevState *d = nullptr;
        int rc = device_state(&d);
        if (rc != 0) return rc;
        rc = get_transpose_ws(*d, stream, static_cast<size_t>(b_off + b_str * (b_str ? nB : 0)) * sizeof(float),
                              &ws);
        if (rc != 0) return rc;
    }
    cudaError_t e = cudaSuccess;
    if (transa) e = sg::transpose_launch(A, lda, K, M, ws, K4, stream, static_cast<int>(nA), sA, a_str);
    if (e == cudaSuccess && transb && !fuse_b)
        e = sg::transpose_launch(B, ldb, N, K, ws + b_off, N4, stream, static_cast<int>(nB), sB, b_str);
    if (e != cudaSuccess) return from_cuda(e);
    if (fuse_b)
        return run(M, N, K, alpha, ws, K4, B, ldb, beta, C, ldc, stream, algo, 0, 0, batch, sA ? a_str : 0, sB, sC,
                   true);
    return run(M, N, K, alpha, transa ? ws : A, transa ? K4 : lda, transb ? ws + b_off : B, transb ? N4 : ldb, beta,
               C, ldc, stream, algo, 0, 0, batch, transa ? (sA ? a_str : 0) : sA, transb ? (sB ? b_str : 0) : sB,
               sC);
}

// Strided batch of run_t calls: matrix b of each operand starts stride * b
// elements after the first.  A zero stride shares one operand across the
// batch; the C matrices must not overlap.  Returns 0 or -i, i the position
// in sgemm_strided_batched.
int run_batched(int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda, long long sA,
                const float *B, int ldb, long long sB, float beta, float *C, int ldc, long long sC, int batch,
                cudaStream_t stream, int algo) {
    static const int kPos[16] = {0, 1, 2, 3, 4, 5, 6, 7, 8, 10, 11, 13, 14, 15, 18, 19};  // sgemm_t -> batched
    const int rc0 = check_t(transa, transb, M, N, K, alpha, A, lda, B, ldb, C, ldc, algo);
    if (rc0 < 0) return -kPos[-rc0];
    if (sA < 0) return -9;
    if (sB < 0) return -12;
    if (batch < 0) return -17;
    if (batch > 1 && M > 0 && N > 0 && (sC < 0 || static_cast<size_t>(sC) * sizeof(float) < span_bytes(M, N, ldc)))
        return -16;
    if (batch > 1 && M > 0 && N > 0) {
        const int rc = run_batched_one_launch(transa, transb, M, N, K, alpha, A, lda, sA, B, ldb, sB, beta, C, ldc,
                                              sC, batch, stream, algo);
        if (rc <= 0) return rc < 0 ? -kPos[-rc] : 0;
    }
    for (int b = 0; b < batch; ++b) {
        const long long ob = b;
        const int rc = run_t(transa, transb, M, N, K, alpha, A ? A + ob * sA : A, lda, B ? B + ob * sB : B, ldb,
                             beta, C + ob * sC, ldc, stream, algo);
        if (rc < 0) return -kPos[-rc];
        if (rc > 0) return rc;
    }
    return 0;
}

// ------------------------------------------------------------ convolution

// Y = alpha * conv2d(X, Wt) + beta * Y (NCHW input and output, OIHW filter)
// as one implicit GEMM per image: M = F filters, K = C * KH * KW taps,
// N = OH * OW output pixels, with the images as the kernel's strided batch.
// The filter is the A operand, always read through its tensor map:
//  - C % 16 == 0: k runs over the channels at each tap (kConvChannels), so
//    the filter is first reordered to OHWI rows in this stream's transpose
//    buffer;
//  - otherwise k runs over the taps of each channel (kConvTaps, the OIHW
//    order); a filter whose rows are not 16-byte aligned is copied into rows
//    padded to 4 floats there.
// Returns 0, -i for the i-th argument of sgemm_conv2d, or a positive error.
constexpr long long kPadCopyMaxBytes = 1LL << 30;  // largest zero-bordered input copy a call makes

int run_conv(int nb, int C, int H, int W, int F, int KH, int KW, int sh, int sw, int ph, int pw, int dh, int dw,
             float alpha, const float *X, const float *Wt, float beta, float *Y, cudaStream_t stream, int algo,
             int flags) {
    if (nb < 0) return -1;
    if (C < 0) return -2;
    if (H < 1) return -3;
    if (W < 1) return -4;
    if (F < 0) return -5;
    if (KH < 1) return -6;
    if (KW < 1) return -7;
    if (sh < 1) return -8;
    if (sw < 1) return -9;
    if (ph < 0) return -10;
    if (pw < 0) return -11;
    if (dh < 1) return -12;
    if (dw < 1) return -13;
    if (algo != SGEMM_ALGO_AUTO && algo != SGEMM_ALGO_TF32X3 && algo != SGEMM_ALGO_FFMA) return -20;
    if (flags & ~SGEMM_CONV_NO_PAD_COPY) return -21;
    const long long span_h = static_cast<long long>(H) + 2LL * ph, span_w = static_cast<long long>(W) + 2LL * pw;
    const long long reach_h = static_cast<long long>(dh) * (KH - 1) + 1, reach_w = static_cast<long long>(dw) * (KW - 1) + 1;
    if (span_h < reach_h) return -6;  // the filter is taller than the padded image
    if (span_w < reach_w) return -7;
    const long long OH = (span_h - reach_h) / sh + 1, OW = (span_w - reach_w) / sw + 1;
    const long long Kl = static_cast<long long>(C) * KH * KW, Nl = OH * OW;
    // 32-bit offsets inside one padded image (the gather) and 32-bit GEMM sizes
    if ((static_cast<long long>(C) + 1) * (span_h + reach_h) * (span_w + reach_w) >= (1LL << 31) || Kl >= (1LL << 31))
        return -2;
    if (Nl >= (1LL << 31)) return -3;
    if (nb == 0 || F == 0) return 0;
    const bool use_ab = alpha != 0.f && C > 0;
    if (use_ab && X == nullptr) return -15;
    if (use_ab && Wt == nullptr) return -16;
    if (Y == nullptr) return -18;
    const int K = static_cast<int>(Kl), N = static_cast<int>(Nl);
    // the wide-N FFMA kernel's convolution form: up to 32 filters of up to 64
    // taps; AUTO takes it where its GEMM form beats the tensor path (K <= 48)
    const bool wide = sg::ffma_wide_fits(F, K) && (algo == SGEMM_ALGO_FFMA || (algo == SGEMM_ALGO_AUTO &&
                                                                               K <= kWideAutoMaxK));
    if (algo == SGEMM_ALGO_FFMA && !wide) return -20;
    const long long img_in = static_cast<long long>(C) * H * W, img_out = static_cast<long long>(F) * N;
    const size_t y_bytes = static_cast<size_t>(nb) * img_out * sizeof(float);
    if (use_ab && (overlaps(Y, y_bytes, X, static_cast<size_t>(nb) * img_in * sizeof(float)) ||
                   overlaps(Y, y_bytes, Wt, static_cast<size_t>(F) * K * sizeof(float))))
        return -18;

    DevState *d = nullptr;
    float *wpad = nullptr, *xpad = nullptr;
    const int lda = (K + 3) / 4 * 4;
    // k order: channels at each tap when C % 16 == 0 (tensor path), else the
    // filter's taps; those gather without bounds checks (a tap table) when
    // every tap lies in the image: no padding, or a zero-bordered copy
    int order = (!wide && C % 16 == 0) ? sg::kConvChannels : sg::kConvTaps;
    const long long pad_elems = (ph || pw) ? static_cast<long long>(nb) * C * span_h * span_w : 0;
    bool copy_pad = false;
    if (order == sg::kConvTaps && K <= sg::kConvTabMax &&
        (pad_elems == 0 ||
         (!(flags & SGEMM_CONV_NO_PAD_COPY) && pad_elems * static_cast<long long>(sizeof(float)) <= kPadCopyMaxBytes))) {
        order = sg::kConvTapsDense;
        copy_pad = pad_elems > 0;
    }
    const bool stage_filter = !wide && (order == sg::kConvChannels || !aligned16(Wt, K));
    const size_t filter_bytes = stage_filter ? (static_cast<size_t>(F) * lda * sizeof(float) + 255) / 256 * 256 : 0;
    if (use_ab && (filter_bytes > 0 || copy_pad)) {
        std::lock_guard<std::mutex> lk(g_mu);
        int rc = device_state(&d);
        if (rc != 0) return rc;
        float *ws = nullptr;
        rc = get_transpose_ws(*d, stream, filter_bytes + (copy_pad ? pad_elems * sizeof(float) : 0), &ws);
        if (rc != 0) return rc;
        if (stage_filter) wpad = ws;
        if (copy_pad) xpad = ws + filter_bytes / sizeof(float);
    } else {
        std::lock_guard<std::mutex> lk(g_mu);
        const int rc = device_state(&d);
        if (rc != 0) return rc;
    }
    if (!use_ab) {  // Y = beta * Y, image by image (F x N each)
        if (beta == 1.f) return 0;
        for (int b = 0; b < nb; ++b) {
            cudaError_t e = sg::scale_c_launch(Y + b * img_out, N, F, N, beta, d->sms, stream);
            if (e != cudaSuccess) return from_cuda(e);
        }
        return 0;
    }
    if (wpad && order == sg::kConvChannels) {
        cudaError_t e = sg::filter_ohwi_launch(Wt, F, C, KH, KW, wpad, lda, stream);
        if (e != cudaSuccess) return from_cuda(e);
    } else if (wpad) {
        cudaError_t e = cudaMemcpy2DAsync(wpad, static_cast<size_t>(lda) * sizeof(float), Wt,
                                          static_cast<size_t>(K) * sizeof(float), static_cast<size_t>(K) * sizeof(float),
                                          static_cast<size_t>(F), cudaMemcpyDeviceToDevice, stream);
        if (e != cudaSuccess) return from_cuda(e);
    }
    const float *A = wpad ? wpad : Wt;
    const int ldA = wpad ? lda : K;
    // the gather's view of the input: the zero-bordered copy, with no padding left
    const float *Xg = X;
    long long g_img = img_in;
    int gH = H, gW = W, gph = ph, gpw = pw;
    if (copy_pad) {
        cudaError_t e = sg::pad_planes_launch(X, static_cast<long long>(nb) * C, H, W, ph, pw, xpad, stream);
        if (e != cudaSuccess) return from_cuda(e);
        Xg = xpad;
        gH = static_cast<int>(span_h);
        gW = static_cast<int>(span_w);
        gph = gpw = 0;
        g_img = static_cast<long long>(C) * gH * gW;
    }
    const sg::ConvGeom geom{C, gH, gW, static_cast<int>(OW), KH, KW, sh, sw, gph, gpw, dh, dw};
    if (wide) {
        // columns = the pixels of all images of a launch (fewer than 2^31)
        const int imgs = static_cast<int>(std::max(1LL, std::min<long long>(nb, INT32_MAX / Nl)));
        for (int b0 = 0; b0 < nb; b0 += imgs) {
            const int nbc = std::min(imgs, nb - b0);
            const int Nt = nbc * N;
            GemmArgs g{F, Nt, K, alpha, beta, Wt, K, Xg + b0 * g_img, 1, Y + b0 * img_out, N, 0, g_img, img_out};
            g.cv = geom;
            g.a_end = Wt + static_cast<long long>(F) * K;
            g.b_end = Xg + (b0 + nbc) * g_img;
            g.c_end = Y + (b0 + nbc) * img_out;
            g.dbg_status = d->status;
            const int grid = std::min(sg::ffma_wide_blocks(Nt), 2 * d->sms);
            cudaError_t e = sg::ffma_wide_launch(g, 0, grid, stream, order);
            if (e != cudaSuccess) return from_cuda(e);
        }
        return 0;
    }
    // images per launch: the schedule's unit index is 32-bit (at most 16 K
    // slices of tiles 16 rows high)
    const long long per_img = static_cast<long long>(ceil_div(F, 16)) * ceil_div(N, sg::kTf32x3TileN) * 16;
    const int chunk = static_cast<int>(std::max(1LL, std::min<long long>(nb, INT32_MAX / per_img)));
    for (int b0 = 0; b0 < nb; b0 += chunk) {
        const int nbc = std::min(chunk, nb - b0);
        Plan p;
        DeviceCtl ctl{};
        {
            std::lock_guard<std::mutex> lk(g_mu);
            plan_tf32x3(F, N, K, d->sms, 0, 0, beta != 0.f, p, nbc);
            if (p.sch.units <= 0 || p.grid <= 0) return SGEMM_ERR_INTERNAL;
            ctl.status = d->status;
            ctl.wait_budget = kWaitBudget;
            if (p.ws_bytes > 0) {
                Workspace *w = nullptr;
                const int rc = get_workspace(*d, stream, p.ws_bytes,
                                             static_cast<size_t>(p.sch.m_tiles) * p.sch.n_tiles * nbc, &w);
                if (rc != 0) return rc;
                ctl.ws = w->ws;
                ctl.counters = w->counters;
                ctl.ws_end = w->ws + p.ws_bytes / sizeof(float);
                ctl.n_counters = static_cast<long long>(w->n_counters);
            }
        }
        float *Yb = Y + b0 * img_out;
        const int vec_c = aligned16(Yb, N) && img_out % 4 == 0;
        GemmArgs g{F, N, K, alpha, beta, A, ldA, Xg + b0 * g_img, N, Yb, N, 0, g_img, img_out};
        g.cv = geom;
        g.a_end = A + static_cast<long long>(F - 1) * ldA + K;
        g.b_end = Xg + (b0 + nbc) * g_img;
        g.c_end = Yb + nbc * img_out;
        g.dbg_status = ctl.status;
        cudaError_t e = sg::tf32x3_conv_launch(p.tile_m, g, p.sch, ctl, order, vec_c, p.grid, stream, nbc);
        if (e != cudaSuccess) return from_cuda(e);
    }
    return 0;
}

// ------------------------------------------------- host-buffer pipeline

// Assumed host <-> device copy rate of pinned memory, each direction, and
// the gap between a block's rows landing and its GEMM starting.  They only
// shape the choice of block sizes below; every block is an ordinary planned
// GEMM, so the result does not depend on them.
constexpr double kHostLinkGBs = 200.0;
constexpr double kHostGemmGapUs = 8.0;
constexpr int kHostRowQuantum = 128;

// The planner's run-time estimate (us) of a 3xTF32 call: the single-CTA
// choice, or the CTA-pair form where the planner would take it.
double model_tf32x3_us(int M, int N, int K, int sms, int pair_slots, bool read_c) {
    const Tf32x3Choice ch = choose_tf32x3(M, N, K, sms, 0, 0, 0, read_c);
    if (use_pairs(M, N, K, ch, 0, pair_slots, read_c, 1)) {
        bool tail = false;
        return model_pairs(M, N, K, ch.tm, pair_slots, read_c, 1, 0, &tail);
    }
    return ch.us;
}

// Row blocks of a pipelined 3xTF32 call, chosen by simulating its timeline:
// B goes up first, then each block's rows of A (and of C when beta != 0);
// a block's GEMM starts once its rows have landed and the previous GEMM is
// done (its time from the planner's model); its rows of C go down after
// it, one block after another.  The call ends with the last download.
// Candidates: a first block of 1..8 quanta (the GEMMs start early), a last
// block of 1..4 quanta (little work after the last upload), and 1..10
// equal middle blocks, plus the fixed policy of host_blocks.  Returns the
// count.
int host_row_blocks_tf32x3(int M, int N, int K, int lda, int ldb, int ldc, bool use_ab, bool read_c, int sms,
                           int pair_slots, int sizes[kHostMaxBlocks]) {
    constexpr int q = kHostRowQuantum;
    // the pair form needs operands that come by TMA (as make_plan decides
    // for the library's own, 256-byte aligned device buffers)
    const bool va = lda % 4 == 0, b_tma = ldb % 4 == 0 || K >= 4;
    std::map<int, double> gemm_us;
    auto gemm = [&](int rows) {
        auto it = gemm_us.find(rows);
        if (it != gemm_us.end()) return it->second;
        const bool a_tma = va || a_gets_staged(rows, N, 0, 1, 0);
        const double us = model_tf32x3_us(rows, N, K, sms, (a_tma && b_tma) ? pair_slots : 0, read_c);
        gemm_us.emplace(rows, us);
        return us;
    };
    const double bytes_per_us = kHostLinkGBs * 1e3;
    auto simulate = [&](const int *sz, int n) {
        double up = use_ab ? static_cast<double>(span_bytes(K, N, ldb)) / bytes_per_us : 0.0;
        double g_end = 0.0, d_end = 0.0;
        for (int i = 0; i < n; ++i) {
            double in = use_ab ? static_cast<double>(span_bytes(sz[i], K, lda)) : 0.0;
            const double c = static_cast<double>(span_bytes(sz[i], N, ldc));
            if (read_c) in += c;
            up += in / bytes_per_us;
            g_end = std::max(up, g_end) + kHostGemmGapUs + gemm(sz[i]);
            d_end = std::max(g_end, d_end) + c / bytes_per_us;
        }
        return d_end;
    };
    int n_best = host_blocks(M, q, sizes);
    double t_best = simulate(sizes, n_best);
    int cand[kHostMaxBlocks];
    const int r = M % q;
    for (int f = q; f <= 8 * q; f += q) {
        for (int l = q; l <= 4 * q; l += q) {
            const int mid = M - f - (l + r);
            if (mid < 0 || f > M / 3) continue;
            for (int nm = (mid > 0 ? 1 : 0); nm <= kHostMaxBlocks - 2 && nm <= mid / q; ++nm) {
                int n = 0;
                cand[n++] = f;
                if (nm > 0) {
                    const int base = mid / q / nm * q;
                    int extra = (mid - base * nm) / q;
                    for (int i = 0; i < nm; ++i, --extra) cand[n++] = base + (extra > 0 ? q : 0);
                }
                cand[n++] = l + r;
                const double t = simulate(cand, n);
                if (t < t_best) {
                    t_best = t;
                    n_best = n;
                    std::copy(cand, cand + n, sizes);
                }
                if (mid == 0) break;
            }
        }
    }
    return n_best;
}

// How sgemm_host cuts a call: returns the block count (1: one GEMM) and
// sets *axis (0: row blocks of C, 1: column blocks).  From 64 MB of traffic
// up, calls of 512 rows or more run as row blocks (3xTF32: chosen by
// host_row_blocks_tf32x3; FFMA: host_blocks), shorter ones of at least
// 8192 columns as column blocks of 1024-column multiples.
int host_split(int M, int N, int K, int lda, int ldb, int ldc, float alpha, float beta, int algo, int sms,
               int pair_slots, int *axis, int sizes[kHostMaxBlocks]) {
    *axis = 0;
    sizes[0] = M;
    const bool use_ab = alpha != 0.f && K > 0;
    const bool read_c = beta != 0.f;
    const size_t a_bytes = use_ab ? span_bytes(M, K, lda) : 0;
    const size_t b_bytes = use_ab ? span_bytes(K, N, ldb) : 0;
    const size_t c_bytes = span_bytes(M, N, ldc);
    const size_t in_bytes = a_bytes + b_bytes + (read_c ? c_bytes : 0);
    if (in_bytes + c_bytes < (64u << 20)) return 1;
    if (M >= 512) {
        if (resolve_path(kHostRowQuantum, K, algo, 0) == SGEMM_ALGO_TF32X3)
            return host_row_blocks_tf32x3(M, N, K, lda, ldb, ldc, use_ab, read_c, sms, pair_slots, sizes);
        return host_blocks(M, kHostRowQuantum, sizes);
    }
    if (N >= 8192) {
        *axis = 1;
        return host_blocks(N, 1024, sizes);
    }
    return 1;
}

}  // namespace

extern "C" {

int sgemm(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
          float *C, int ldc, sgemm_stream_t stream) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, reinterpret_cast<cudaStream_t>(stream),
               SGEMM_ALGO_AUTO, 0, 0);
}

int sgemm_ex(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
             float *C, int ldc, sgemm_stream_t stream, int algo, int splits, int flags) {
    return run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, reinterpret_cast<cudaStream_t>(stream), algo,
               splits, flags);
}

int sgemm_host(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb, float beta,
               float *C, int ldc, int algo) {
    int rc = check_args(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, algo, 0, 0);
    if (rc != 0) return rc;
    if (M == 0 || N == 0) return 0;
    std::unique_lock<std::mutex> lk(g_mu);
    DevState *d = nullptr;
    rc = device_state(&d);
    if (rc != 0) return rc;
    HostBuffers &h = d->host;
    cudaError_t e;
    if (!h.stream) {
        e = cudaStreamCreateWithFlags(&h.stream, cudaStreamNonBlocking);
        if (e != cudaSuccess) return from_cuda(e);
        if ((e = cudaStreamCreateWithFlags(&h.up, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&h.down, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaEventCreateWithFlags(&h.b_in, cudaEventDisableTiming)) != cudaSuccess)
            return from_cuda(e);
        for (int i = 0; i < kHostMaxBlocks; ++i)
            if ((e = cudaEventCreateWithFlags(&h.in[i], cudaEventDisableTiming)) != cudaSuccess ||
                (e = cudaEventCreateWithFlags(&h.out[i], cudaEventDisableTiming)) != cudaSuccess)
                return from_cuda(e);
    }
    const bool use_ab = alpha != 0.f && K > 0;
    const size_t a_bytes = use_ab ? span_bytes(M, K, lda) : 0;
    const size_t b_bytes = use_ab ? span_bytes(K, N, ldb) : 0;
    const size_t c_bytes = span_bytes(M, N, ldc);
    auto grow = [&](float *&buf, size_t &cap, size_t need) -> int {
        if (cap >= need) return 0;
        if (buf) {
            cudaStreamSynchronize(h.stream);
            cudaFree(buf);
            buf = nullptr;
            cap = 0;
        }
        if (cudaMalloc(reinterpret_cast<void **>(&buf), need) != cudaSuccess) {
            cudaGetLastError();
            return SGEMM_ERR_WORKSPACE;
        }
        cap = need;
        return 0;
    };
    if ((rc = grow(h.A, h.a_bytes, std::max<size_t>(a_bytes, 16))) != 0) return rc;
    if ((rc = grow(h.B, h.b_bytes, std::max<size_t>(b_bytes, 16))) != 0) return rc;
    if ((rc = grow(h.C, h.c_bytes, c_bytes)) != 0) return rc;
    // Large calls run as row blocks of C, so that copies overlap the GEMMs:
    // B goes up first, then each block's rows of A (and C when beta != 0) on
    // the upload stream; a block's GEMM runs once its rows have landed, and
    // its rows of C come back on the download stream while the next blocks
    // compute.  Each block is a planned GEMM of its own (the same arithmetic
    // per element; a block's schedule may differ from the whole call's).
    int sizes[kHostMaxBlocks];
    int axis = 0;
    // row blocks; short and wide (the im2col shapes): column blocks instead,
    // A goes up first and each block's columns of B (and C) move as pitched
    // copies
    const int nb = host_split(M, N, K, lda, ldb, ldc, alpha, beta, algo, d->sms, d->pair_slots, &axis, sizes);
    const int nblk = axis == 0 ? nb : 1;
    const int ncb = axis == 1 ? nb : 1;
    if (ncb > 1) {
        float *dA = h.A, *dB = h.B, *dC = h.C;
        cudaStream_t st = h.stream, up = h.up, down = h.down;
        cudaEvent_t a_in = h.b_in, ev_in[kHostMaxBlocks], ev_out[kHostMaxBlocks];
        for (int i = 0; i < ncb; ++i) {
            ev_in[i] = h.in[i];
            ev_out[i] = h.out[i];
        }
        lk.unlock();
        if (a_bytes && (e = cudaMemcpyAsync(dA, A, a_bytes, cudaMemcpyHostToDevice, up)) != cudaSuccess)
            return from_cuda(e);
        if ((e = cudaEventRecord(a_in, up)) != cudaSuccess || (e = cudaStreamWaitEvent(st, a_in, 0)) != cudaSuccess)
            return from_cuda(e);
        int first_rc = 0;
        for (int i = 0, c0 = 0; i < ncb; c0 += sizes[i], ++i) {
            const int nc = sizes[i];
            const size_t w = static_cast<size_t>(nc) * sizeof(float);
            if (use_ab && (e = cudaMemcpy2DAsync(dB + c0, static_cast<size_t>(ldb) * sizeof(float), B + c0,
                                                 static_cast<size_t>(ldb) * sizeof(float), w, static_cast<size_t>(K),
                                                 cudaMemcpyHostToDevice, up)) != cudaSuccess)
                return from_cuda(e);
            if (beta != 0.f && (e = cudaMemcpy2DAsync(dC + c0, static_cast<size_t>(ldc) * sizeof(float), C + c0,
                                                      static_cast<size_t>(ldc) * sizeof(float), w,
                                                      static_cast<size_t>(M), cudaMemcpyHostToDevice, up)) !=
                                    cudaSuccess)
                return from_cuda(e);
            if ((e = cudaEventRecord(ev_in[i], up)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(st, ev_in[i], 0)) != cudaSuccess)
                return from_cuda(e);
            rc = run(M, nc, K, alpha, use_ab ? dA : nullptr, lda, use_ab ? dB + c0 : nullptr, ldb, beta, dC + c0, ldc,
                     st, algo, 0, 0);
            if (rc != 0 && first_rc == 0) first_rc = rc;
            if ((e = cudaEventRecord(ev_out[i], st)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(down, ev_out[i], 0)) != cudaSuccess)
                return from_cuda(e);
            if ((e = cudaMemcpy2DAsync(C + c0, static_cast<size_t>(ldc) * sizeof(float), dC + c0,
                                       static_cast<size_t>(ldc) * sizeof(float), w, static_cast<size_t>(M),
                                       cudaMemcpyDeviceToHost, down)) != cudaSuccess)
                return from_cuda(e);
        }
        e = cudaStreamSynchronize(down);
        const cudaError_t e2 = cudaStreamSynchronize(st);
        if (first_rc != 0) return first_rc;
        return from_cuda(e != cudaSuccess ? e : e2);
    }
    if (nblk > 1) {
        float *dA = h.A, *dB = h.B, *dC = h.C;
        cudaStream_t st = h.stream, up = h.up, down = h.down;
        cudaEvent_t b_in = h.b_in, ev_in[kHostMaxBlocks], ev_out[kHostMaxBlocks];
        for (int i = 0; i < nblk; ++i) {
            ev_in[i] = h.in[i];
            ev_out[i] = h.out[i];
        }
        lk.unlock();
        // the previous call's copies and GEMMs on these streams are finished
        // (it synchronised), so the buffers are free
        if (b_bytes && (e = cudaMemcpyAsync(dB, B, b_bytes, cudaMemcpyHostToDevice, up)) != cudaSuccess)
            return from_cuda(e);
        if ((e = cudaEventRecord(b_in, up)) != cudaSuccess || (e = cudaStreamWaitEvent(st, b_in, 0)) != cudaSuccess)
            return from_cuda(e);
        int first_rc = 0;
        for (int i = 0, r0 = 0; i < nblk; r0 += sizes[i], ++i) {
            const int mr = sizes[i];
            const size_t ao = static_cast<size_t>(r0) * lda, co = static_cast<size_t>(r0) * ldc;
            const size_t cb = span_bytes(mr, N, ldc);
            if (use_ab && (e = cudaMemcpyAsync(dA + ao, A + ao, span_bytes(mr, K, lda), cudaMemcpyHostToDevice,
                                               up)) != cudaSuccess)
                return from_cuda(e);
            if (beta != 0.f && (e = cudaMemcpyAsync(dC + co, C + co, cb, cudaMemcpyHostToDevice, up)) != cudaSuccess)
                return from_cuda(e);
            if ((e = cudaEventRecord(ev_in[i], up)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(st, ev_in[i], 0)) != cudaSuccess)
                return from_cuda(e);
            rc = run(mr, N, K, alpha, use_ab ? dA + ao : nullptr, lda, use_ab ? dB : nullptr, ldb, beta, dC + co, ldc,
                     st, algo, 0, 0);
            if (rc != 0 && first_rc == 0) first_rc = rc;
            if ((e = cudaEventRecord(ev_out[i], st)) != cudaSuccess ||
                (e = cudaStreamWaitEvent(down, ev_out[i], 0)) != cudaSuccess)
                return from_cuda(e);
            if ((e = cudaMemcpyAsync(C + co, dC + co, cb, cudaMemcpyDeviceToHost, down)) != cudaSuccess)
                return from_cuda(e);
        }
        e = cudaStreamSynchronize(down);
        const cudaError_t e2 = cudaStreamSynchronize(st);
        if (first_rc != 0) return first_rc;
        return from_cuda(e != cudaSuccess ? e : e2);
    }
    if (a_bytes && (e = cudaMemcpyAsync(h.A, A, a_bytes, cudaMemcpyHostToDevice, h.stream)) != cudaSuccess)
        return from_cuda(e);
    if (b_bytes && (e = cudaMemcpyAsync(h.B, B, b_bytes, cudaMemcpyHostToDevice, h.stream)) != cudaSuccess)
        return from_cuda(e);
    if (beta != 0.f &&
        (e = cudaMemcpyAsync(h.C, C, c_bytes, cudaMemcpyHostToDevice, h.stream)) != cudaSuccess)
        return from_cuda(e);
    float *dA = h.A, *dB = h.B, *dC = h.C;
    cudaStream_t st = h.stream;
    lk.unlock();
    rc = run(M, N, K, alpha, use_ab ? dA : nullptr, lda, use_ab ? dB : nullptr, ldb, beta, dC, ldc, st, algo,
             0, 0);
    if (rc != 0) return rc;
    if ((e = cudaMemcpyAsync(C, dC, c_bytes, cudaMemcpyDeviceToHost, st)) != cudaSuccess) return from_cuda(e);
    return from_cuda(cudaStreamSynchronize(st));
}

int sgemm_plan_info(int M, int N, int K, const void *A, int lda, const void *B, int ldb, const void *C, int ldc,
                    int algo, int splits, int flags, float alpha, float beta, int num_sms, int *info,
                    int ninfo) {
    if (M < 0) return -1;
    if (N < 0) return -2;
    if (K < 0) return -3;
    if (lda < std::max(1, K)) return -5;
    if (ldb < std::max(1, N)) return -7;
    if (ldc < std::max(1, N)) return -9;
    if (algo < SGEMM_ALGO_AUTO || algo > SGEMM_ALGO_TF32X3) return -10;
    if (splits < 0) return -11;
    if (!flags_valid(flags)) return -12;
    if (num_sms < 0) return -15;
    if (info == nullptr && ninfo > 0) return -16;
    if (ninfo < 0) return -17;
    (void)alpha;
    (void)beta;
    int sms = num_sms, pair_slots = num_sms / 2;
    if (sms == 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        DevState *d = nullptr;
        int rc = device_state(&d);
        if (rc != 0) return rc;
        sms = d->sms;
        pair_slots = d->pair_slots;
    }
    int vals[13] = {0};
    if (M > 0 && N > 0 && K > 0) {
        Plan p;
        int rc = make_plan(M, N, K, A, lda, B, ldb, C, ldc, algo, splits, flags, sms, beta != 0.f, p, 1, 0, 0, 0,
                           pair_slots);
        if (rc != 0) return rc;
        vals[0] = p.path;
        vals[1] = p.tile_m;
        vals[2] = p.tile_n;
        vals[3] = p.sch.splits;
        vals[4] = p.sch.units;
        vals[5] = p.grid;
        vals[6] = p.stages;
        vals[7] = p.vec_a;
        vals[8] = p.vec_b;
        vals[9] = static_cast<int>(std::min<size_t>(p.ws_bytes, 0x7fffffff));
        vals[10] = p.sch.tail_tiles;
        vals[11] = p.wide ? 1 : 0;
        vals[12] = p.sch.pair_shift;
    }
    for (int i = 0; i < ninfo && i < 13; ++i) info[i] = vals[i];
    return 0;
}

int sgemm_host_blocks(int M, int N, int K, int lda, int ldb, int ldc, float alpha, float beta, int algo,
                      int num_sms, int *axis, int *sizes, int max_sizes) {
    if (M < 0) return -1;
    if (N < 0) return -2;
    if (K < 0) return -3;
    if (lda < std::max(1, K)) return -4;
    if (ldb < std::max(1, N)) return -5;
    if (ldc < std::max(1, N)) return -6;
    if (algo < SGEMM_ALGO_AUTO || algo > SGEMM_ALGO_TF32X3) return -9;
    if (num_sms < 0) return -10;
    if (axis == nullptr) return -11;
    if (sizes == nullptr && max_sizes > 0) return -12;
    if (max_sizes < 0) return -13;
    int sms = num_sms, pair_slots = num_sms / 2;
    if (sms == 0) {
        std::lock_guard<std::mutex> lk(g_mu);
        DevState *d = nullptr;
        int rc = device_state(&d);
        if (rc != 0) return rc;
        sms = d->sms;
        pair_slots = d->pair_slots;
    }
    int sz[kHostMaxBlocks];
    int n = 1;
    *axis = 0;
    if (M > 0 && N > 0) n = host_split(M, N, K, lda, ldb, ldc, alpha, beta, algo, sms, pair_slots, axis, sz);
    else sz[0] = M;
    for (int i = 0; i < n && i < max_sizes; ++i) sizes[i] = sz[i];
    return n;
}

int sgemm_check_status(sgemm_stream_t stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    std::lock_guard<std::mutex> lk(g_mu);
    DevState *d = nullptr;
    int rc = device_state(&d);
    if (rc != 0) return rc;
    int word = 0;
    e = cudaMemcpy(&word, d->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (word != 0) {
        // a kernel that gave up may have left split-K arrival counters
        // non-zero: wait for the device and clear them all
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return from_cuda(e);
        for (auto &kv : d->ws)
            if (kv.second.counters) cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(int));
        e = cudaMemset(d->status, 0, sizeof(int));
        if (e != cudaSuccess) return from_cuda(e);
    }
    // the status word of sgemm_noalloc on this device (it clears its own
    // arrival counters when the word is set)
    const int na = sg::noalloc_take_status();
    if (na < 0) return -na;  // a CUDA error, as a positive code
    if (word & sg::kStatusOutOfBounds) return SGEMM_ERR_OUT_OF_BOUNDS;
    return (word != 0 || na > 0) ? SGEMM_ERR_DEVICE_TIMEOUT : 0;
}

const char *sgemm_status_string(int status) {
    if (status == 0) return "success";
    if (status < 0) {
        switch (-status) {
            case 1: return "invalid argument 1 (M < 0)";
            case 2: return "invalid argument 2 (N < 0)";
            case 3: return "invalid argument 3 (K < 0)";
            case 5: return "invalid argument 5 (A is NULL)";
            case 6: return "invalid argument 6 (lda < max(1, K))";
            case 7: return "invalid argument 7 (B is NULL)";
            case 8: return "invalid argument 8 (ldb < max(1, N))";
            case 10: return "invalid argument 10 (C is NULL or overlaps A or B)";
            case 11: return "invalid argument 11 (ldc < max(1, N))";
            case 13: return "invalid argument 13 (unknown algo)";
            case 14: return "invalid argument 14 (splits < 0)";
            case 15: return "invalid argument 15 (unknown flags)";
            default: return "invalid argument";
        }
    }
    switch (status) {
        case SGEMM_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait gave up (result unspecified)";
        case SGEMM_ERR_NO_DEVICE: return "no usable CUDA device";
        case SGEMM_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (sm_103a)";
        case SGEMM_ERR_WORKSPACE: return "could not allocate library-owned device memory";
        case SGEMM_ERR_INTERNAL: return "internal planner error";
        case SGEMM_ERR_OUT_OF_BOUNDS:
            return "SGEMM_DEBUG build: a kernel address outside its matrix was found and skipped (result unspecified)";
        case SGEMM_ERR_SCRATCH_LIMIT:
            return "the problem needs more split-K scratch than sgemm_noalloc's fixed array "
                   "(16 MiB of partial tiles, 4096 tiles): use sgemm_ex or fewer splits";
        default: break;
    }
    if (status > 0 && status < 10000) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

int sgemm_release(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int rc = 0;
    for (int dev = 0; dev < kMaxDevices; ++dev) {
        DevState &d = g_dev[dev];
        if (!d.ready) continue;
        cudaSetDevice(dev);
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess && rc == 0) rc = from_cuda(e);
        for (auto &kv : d.ws) {
            cudaFree(kv.second.ws);
            cudaFree(kv.second.counters);
            cudaFree(kv.second.tr);
            cudaFree(kv.second.ap);
        }
        d.ws.clear();
        cudaFree(d.host.A);
        cudaFree(d.host.B);
        cudaFree(d.host.C);
        d.host.A = d.host.B = d.host.C = nullptr;
        d.host.a_bytes = d.host.b_bytes = d.host.c_bytes = 0;
    }
    cudaSetDevice(cur);
    return rc;
}

int sgemm_t(int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda, const float *B,
            int ldb, float beta, float *C, int ldc, sgemm_stream_t stream, int algo) {
    return run_t(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, reinterpret_cast<cudaStream_t>(stream),
                 algo);
}

int sgemm_strided_batched(int transa, int transb, int M, int N, int K, float alpha, const float *A, int lda,
                          long long strideA, const float *B, int ldb, long long strideB, float beta, float *C,
                          int ldc, long long strideC, int batch, sgemm_stream_t stream, int algo) {
    return run_batched(transa, transb, M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc, strideC,
                       batch, reinterpret_cast<cudaStream_t>(stream), algo);
}

int sgemm_conv2d(int nb, int C, int H, int W, int F, int KH, int KW, int stride_h, int stride_w, int pad_h,
                 int pad_w, int dil_h, int dil_w, float alpha, const float *X, const float *Wt, float beta, float *Y,
                 sgemm_stream_t stream, int algo) {
    return run_conv(nb, C, H, W, F, KH, KW, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, alpha, X, Wt, beta, Y,
                    reinterpret_cast<cudaStream_t>(stream), algo, 0);
}

int sgemm_conv2d_ex(int nb, int C, int H, int W, int F, int KH, int KW, int stride_h, int stride_w, int pad_h,
                    int pad_w, int dil_h, int dil_w, float alpha, const float *X, const float *Wt, float beta,
                    float *Y, sgemm_stream_t stream, int algo, int flags) {
    return run_conv(nb, C, H, W, F, KH, KW, stride_h, stride_w, pad_h, pad_w, dil_h, dil_w, alpha, X, Wt, beta, Y,
                    reinterpret_cast<cudaStream_t>(stream), algo, flags);
}

int sgemm_version(void) { return kVersion; }

}  // extern "C"

// ---------------------------------------------------------------- internal
// Used by sgemm_noalloc (noalloc.cu): the same checks and planner as
// sgemm_ex with algo = SGEMM_ALGO_TF32X3 and flags = 0.
namespace sg {

int check_tensor_call(int M, int N, int K, float alpha, const float *A, int lda, const float *B, int ldb,
                      float beta, const float *C, int ldc, int splits) {
    const int rc = check_args(M, N, K, alpha, A, lda, B, ldb, beta, const_cast<float *>(C), ldc,
                              SGEMM_ALGO_TF32X3, splits, 0);
    return rc == -15 ? SGEMM_ERR_INTERNAL : rc;  // flags are fixed here
}

int plan_tensor_call(int M, int N, int K, const float *A, int lda, const float *B, int ldb, float beta,
                     const float *C, int ldc, int splits, int sms, int pair_slots, size_t max_ws_floats,
                     TensorPlan *out) {
    Plan p;
    int rc = make_plan(M, N, K, A, lda, B, ldb, C, ldc, SGEMM_ALGO_TF32X3, splits, 0, sms, beta != 0.f, p, 1, 0, 0,
                       0, pair_slots);
    if (rc != 0) return rc;
    if (p.sch.tail_tiles > 0 && p.ws_bytes / sizeof(float) > max_ws_floats) {
        // the split tail is an optimisation: drop it rather than exceed the scratch
        p = Plan();
        rc = make_plan(M, N, K, A, lda, B, ldb, C, ldc, SGEMM_ALGO_TF32X3, splits, SGEMM_FLAG_WHOLE_TILES, sms,
                       beta != 0.f, p, 1, 0, 0, 0, pair_slots);
        if (rc != 0) return rc;
    }
    out->tile_m = p.tile_m;
    out->sch = p.sch;
    out->grid = p.grid;
    out->vec_a = p.vec_a;
    out->vec_b = p.vec_b;
    out->vec_c = p.vec_c;
    out->ws_floats = p.ws_bytes / sizeof(float);
    out->tiles = (p.sch.m_tiles * p.sch.n_tiles) << p.sch.pair_shift;
    return 0;
}

}  // namespace sg
