"""Host-side checks of the C ABI that need no GPU.

The library must load and export every function the header declares;
invalid arguments are rejected with -i (1-based, LAPACK style) before any
CUDA call; empty problems return 0 without touching the device; the planner
(sgemm_plan_info with an explicit SM count) makes the documented choices.
"""
from __future__ import annotations

import ctypes

import pytest

import dense_fp32_matrix_05_gb300 as pkg


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return pkg.library()


def test_exports_every_declared_symbol(lib):
    declared = pkg.declared_functions()
    assert {"sgemm", "sgemm_ex", "sgemm_host", "sgemm_plan_info", "sgemm_check_status",
            "sgemm_status_string", "sgemm_release", "sgemm_version"} <= set(declared)
    raw = ctypes.CDLL(pkg.lib_path())
    for name in declared:
        assert hasattr(raw, name), f"{name} declared in the header but not exported"


def test_version(lib):
    assert pkg.sgemm_version() >= 100


FAKE = 1 << 20  # never dereferenced: every call below returns before any CUDA call


@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -1),
    ((4, -1, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -2),
    ((4, 4, -1, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -3),
    ((4, 4, 4, 1.0, FAKE, 3, FAKE, 4, 0.0, FAKE, 4), -6),
    ((4, 4, 0, 1.0, FAKE, 0, FAKE, 4, 0.0, FAKE, 4), -6),
    ((4, 4, 4, 1.0, FAKE, 4, FAKE, 3, 0.0, FAKE, 4), -8),
    ((4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 3), -11),
    ((4, 4, 4, 1.0, None, 4, FAKE, 4, 0.0, FAKE + 4096, 4), -5),
    ((4, 4, 4, 1.0, FAKE, 4, None, 4, 0.0, FAKE + 4096, 4), -7),
    ((4, 4, 4, 1.0, FAKE, 4, FAKE + 4096, 4, 0.0, None, 4), -10),
    # C overlapping A / B
    ((4, 4, 4, 1.0, FAKE, 4, FAKE + 4096, 4, 0.0, FAKE + 16, 4), -10),
    ((4, 4, 4, 1.0, FAKE, 4, FAKE + 4096, 4, 0.0, FAKE + 4096 + 60, 4), -10),
])
def test_invalid_arguments(lib, args, code):
    assert pkg.sgemm(*args) == code
    assert pkg.sgemm_ex(*args, None, 0, 0, 0) == code


def test_invalid_extended_arguments(lib):
    base = (4, 4, 4, 1.0, FAKE, 4, FAKE + 4096, 4, 0.0, FAKE + 8192, 4, None)
    assert pkg.sgemm_ex(*base, 3, 0, 0) == -13
    assert pkg.sgemm_ex(*base, -1, 0, 0) == -13
    assert pkg.sgemm_ex(*base, 0, -1, 0) == -14
    assert pkg.sgemm_ex(*base, 0, 0, 8) == -15
    assert pkg.sgemm_ex(*base, 0, 0, pkg.SGEMM_FLAG_TILE_ROWS(48)) == -15
    assert pkg.sgemm_ex(*base, 0, 0, 1 << 20) == -15


def test_empty_problems_need_no_device(lib):
    assert pkg.sgemm(0, 5, 5, 1.0, None, 5, None, 5, 0.0, None, 5) == 0
    assert pkg.sgemm(5, 0, 5, 1.0, None, 5, None, 1, 0.0, None, 1) == 0
    assert pkg.sgemm_host(0, 5, 5, 1.0, None, 5, None, 5, 0.0, None, 5) == 0


def test_no_ab_needed_when_alpha_zero_validation(lib):
    # alpha == 0: A and B may be NULL; with M == 0 the call is a no-op
    assert pkg.sgemm(0, 4, 4, 0.0, None, 4, None, 4, 1.0, None, 4) == 0


def test_status_strings(lib):
    assert pkg.sgemm_status_string(0) == "success"
    assert "argument 6" in pkg.sgemm_status_string(-6)
    assert "wait" in pkg.sgemm_status_string(pkg.SGEMM_ERR_DEVICE_TIMEOUT)
    assert pkg.sgemm_status_string(987654) == "unknown status"


SMS = 152


def plan(M, N, K, **kw):
    kw.setdefault("num_sms", SMS)
    return pkg.sgemm_plan_info(M, N, K, A=0x100000, B=0x200000, C=0x300000, **kw)


def test_plan_large_square_uses_tensor_path_without_split():
    p = plan(5120, 5120, 5120)
    assert p["path"] == pkg.SGEMM_ALGO_TF32X3
    # 256-row tiles run on CTA pairs: 256 x 256 tiles, two CTAs each
    assert (p["tile_m"], p["tile_n"], p["pairs"]) == (256, 256, 1)
    assert p["splits"] == 1 and p["units"] == 20 * 20 and p["grid"] == SMS
    assert p["vec_a"] == 1 and p["vec_b"] == 1
    q = plan(5120, 5120, 5120, flags=pkg.SGEMM_FLAG_NO_PAIRS)
    assert (q["tile_m"], q["tile_n"], q["pairs"]) == (256, 128, 0)
    assert q["units"] == 20 * 40 and q["grid"] == SMS


def test_plan_cta_pairs():
    """When the planner runs tiles on CTA pairs: 256-row tiles by default,
    192-row tiles only with SGEMM_FLAG_PAIRS, never with SGEMM_FLAG_NO_PAIRS
    or when an operand cannot come by TMA (A rows not 16-byte aligned; a B
    whose start is misaligned or whose residue classes are turned off)."""
    P, NP = pkg.SGEMM_FLAG_PAIRS, pkg.SGEMM_FLAG_NO_PAIRS
    assert plan(256, 43264, 1152)["pairs"] == 1
    assert plan(384, 14161, 1152)["pairs"] == 0  # 192-row tiles
    p = plan(384, 14161, 1152, flags=P)
    assert (p["pairs"], p["tile_m"], p["tile_n"]) == (1, 192, 256)
    assert plan(384, 14161, 1152, flags=P | NP)["pairs"] == 0
    assert plan(1024, 1024, 1024, flags=P)["pairs"] == 0  # 128-row tiles have no pair form
    # where the single-CTA plan splits K to fill the SMs, pairs (half the tiles) stay off
    q = plan(1536, 1536, 1536)
    assert q["pairs"] == 0 and q["splits"] > 1 and q["tile_m"] == 256
    assert plan(1536, 1536, 1536, flags=P)["pairs"] == 1
    # the pair model keeps single CTAs where 256-column tiles waste a wave:
    # N = 600 pads to 768 columns and 120 pair tiles fill 1.6 waves
    assert plan(10000, 600, 3000)["pairs"] == 0
    assert plan(10000, 600, 3000, flags=P)["pairs"] == 1
    # unaligned A rows: no TMA for A, no pairs (not even when asked for)
    assert pkg.sgemm_plan_info(5120, 5120, 5121, A=0x100000, B=0x200000, C=0x300000, num_sms=SMS,
                               flags=P)["pairs"] == 0
    # unaligned B rows with an aligned start come by TMA as residue classes
    q = pkg.sgemm_plan_info(5120, 5121, 5120, A=0x100000, B=0x200000, C=0x300000, num_sms=SMS, flags=P)
    assert q["pairs"] == 1 and q["vec_b"] == 0
    assert pkg.sgemm_plan_info(5120, 5121, 5120, A=0x100000, B=0x200004, C=0x300000, num_sms=SMS,
                               flags=P)["pairs"] == 0
    assert pkg.sgemm_plan_info(5120, 5121, 5120, A=0x100000, B=0x200000, C=0x300000, num_sms=SMS,
                               flags=P | pkg.SGEMM_FLAG_B_ROWS_LOADED)["pairs"] == 0
    # the FFMA path never pairs
    assert plan(5120, 5120, 5120, algo=pkg.SGEMM_ALGO_FFMA)["pairs"] == 0


def test_plan_small_square_splits_k():
    p = plan(1024, 1024, 1024)
    assert p["splits"] > 1
    assert p["units"] <= SMS
    assert p["ws_bytes"] == p["units"] * p["tile_m"] * p["tile_n"] * 4


def test_plan_skinny_shapes_pick_matching_tile_rows():
    assert plan(32, 1605632, 27)["tile_m"] == 32
    assert plan(64, 559104, 147)["tile_m"] == 64
    assert plan(384, 14161, 1152)["tile_m"] == 192
    assert plan(256, 50176, 1024)["tile_m"] == 256


def test_plan_alignment_detection():
    p = pkg.sgemm_plan_info(64, 64, 27, A=0x100000, lda=27, B=0x200004, C=0x300000,
                            num_sms=SMS)
    assert p["vec_a"] == 0 and p["vec_b"] == 0
    p = pkg.sgemm_plan_info(64, 64, 28, A=0x100000, lda=28, B=0x200000, C=0x300000,
                            num_sms=SMS)
    assert p["vec_a"] == 1 and p["vec_b"] == 1


def test_plan_forced_splits_are_clamped():
    p = plan(512, 512, 64, splits=100)
    assert p["splits"] == 4  # 64 / 16 K tiles
    p = plan(512, 512, 64, splits=100, algo=pkg.SGEMM_ALGO_FFMA)
    assert p["splits"] == 4


def test_plan_forced_splits_bound_units_per_cta():
    """A CTA finishes at most 8 shared tiles, so many forced K slices get a
    grid larger than the SM count."""
    p = plan(4096, 4096, 4096, splits=16)
    assert p["splits"] == 16 and p["units"] == -(-4096 // p["tile_m"]) * 32 * 16
    assert p["grid"] == -(-p["units"] // 8) and p["grid"] > SMS
    q = plan(1024, 1024, 1024, splits=2)
    assert q["grid"] == min(q["units"], SMS)


def test_plan_ffma_tiles():
    assert (plan(32, 4096, 64, algo=1)["tile_m"], plan(32, 4096, 64, algo=1)["tile_n"]) == (32, 512)
    assert plan(64, 4096, 64, algo=1)["tile_n"] == 256
    # 128 x 256 tiles (one CTA per SM) once they fill 80 % of a wave, else 128 x 128
    big = plan(4096, 4096, 4096, algo=1)  # 512 tiles: 3 waves, then 56 tiles in 2 K slices each
    assert (big["tile_m"], big["tile_n"], big["tail_tiles"], big["grid"]) == (128, 256, 56, 3 * SMS + 56 * 2)
    assert plan(1024, 1024, 1024, algo=1)["tile_n"] == 128
    assert plan(2048, 2048, 2048, algo=1, num_sms=152)["tile_n"] == 256  # 16 x 8 = 128 tiles >= 0.8 x 152
    assert plan(2048, 1536, 2048, algo=1, num_sms=152)["tile_n"] == 128  # 16 x 6 = 96 tiles


def test_plan_split_tail():
    """Tiles beyond many whole waves: the whole waves keep whole tiles, the
    leftover tiles are cut into K slices over the otherwise idle SMs (single
    CTAs here; CTA pairs: test_plan_cta_pairs)."""
    p = plan(8192, 8192, 8192, flags=pkg.SGEMM_FLAG_NO_PAIRS)  # 2048 tiles = 13 waves of 152 + 72
    assert p["tail_tiles"] == 72 and p["grid"] == SMS
    assert p["ws_bytes"] == 72 * (SMS // 72) * 256 * 128 * 4
    q = plan(8192, 8192, 8192, flags=pkg.SGEMM_FLAG_WHOLE_TILES | pkg.SGEMM_FLAG_NO_PAIRS)
    assert q["tail_tiles"] == 0 and q["ws_bytes"] == 0
    p5 = plan(5120, 5120, 5120, flags=pkg.SGEMM_FLAG_NO_PAIRS)  # 800 tiles = 5 waves + 40
    assert p5["tail_tiles"] == 40 and p5["tile_m"] == 256
    assert p5["ws_bytes"] == 40 * (SMS // 40) * 256 * 128 * 4
    assert plan(4864, 4096, 4096, flags=pkg.SGEMM_FLAG_NO_PAIRS)["tail_tiles"] == 0  # 19 x 32 = 608 tiles: 4 whole waves
    assert plan(1024, 1024, 1024)["tail_tiles"] == 0    # fewer tiles than SMs: split-K instead
    assert plan(8192, 8192, 8192, splits=1, flags=pkg.SGEMM_FLAG_NO_PAIRS)["tail_tiles"] == 0  # explicit split count wins
    # a forced split tail where the estimate prefers whole tiles
    f = plan(4096, 24576, 256, flags=pkg.SGEMM_FLAG_SPLIT_TAIL | pkg.SGEMM_FLAG_NO_PAIRS)
    assert f["tail_tiles"] > 0 and f["grid"] == SMS
    assert f["tail_tiles"] == (-(-4096 // f["tile_m"]) * 192) % SMS
    assert plan(3072, 3072, 3072, flags=pkg.SGEMM_FLAG_SPLIT_TAIL | pkg.SGEMM_FLAG_NO_PAIRS)["tail_tiles"] == 0  # none possible


@pytest.mark.parametrize("rows", [16, 32, 64, 128, 192, 256])
def test_plan_forced_tile_rows(rows):
    p = plan(5120, 5120, 5120, flags=pkg.SGEMM_FLAG_TILE_ROWS(rows) | pkg.SGEMM_FLAG_NO_PAIRS)
    assert p["tile_m"] == rows
    assert p["units"] == -(-5120 // rows) * 40


def test_plan_info_rejects_bad_arguments():
    with pytest.raises(pkg.SgemmError):
        pkg.sgemm_plan_info(-1, 4, 4, num_sms=SMS)
    with pytest.raises(pkg.SgemmError):
        pkg.sgemm_plan_info(4, 4, 4, algo=7, num_sms=SMS)
    with pytest.raises(pkg.SgemmError):
        pkg.sgemm_plan_info(4, 4, 4, flags=pkg.SGEMM_FLAG_TILE_ROWS(80), num_sms=SMS)


def test_tf32_mma_rate_rejects_bad_arguments(lib):
    """Argument checks come before any device query, so they run here."""
    import ctypes
    out = ctypes.c_double(0.0)
    f = pkg.library().sgemm_tf32_mma_rate
    assert f(8, 100, None, ctypes.byref(out)) == -1      # n below 16
    assert f(264, 100, None, ctypes.byref(out)) == -1    # n above 256
    assert f(72, 100, None, ctypes.byref(out)) == -1     # not a multiple of 16
    assert f(256, 0, None, ctypes.byref(out)) == -2
    assert f(256, 100, None, None) == -4


def test_plan_wide_kernel_for_short_shallow_a():
    """M <= 32 and K <= 64 go to the FFMA path's wide-N kernel under AUTO."""
    p = plan(32, 1605632, 27)
    assert p["path"] == pkg.SGEMM_ALGO_FFMA and p["wide"] == 1
    # aligned B rows and N: the bulk-copy form, one CTA per SM; else two
    assert p["units"] == -(-1605632 // 512) and p["grid"] == min(p["units"], SMS)
    q = plan(32, 1605630, 27)
    assert q["wide"] == 1 and q["grid"] == min(q["units"], 2 * SMS)
    assert plan(1, 7, 1)["wide"] == 1
    assert plan(32, 4096, 48)["wide"] == 1
    assert plan(32, 4096, 64)["path"] == pkg.SGEMM_ALGO_TF32X3      # AUTO: the tensor path wins at K = 64
    assert plan(32, 4096, 64, algo=pkg.SGEMM_ALGO_FFMA)["wide"] == 1
    assert plan(32, 4096, 65, algo=pkg.SGEMM_ALGO_FFMA)["wide"] == 0
    assert plan(33, 4096, 27)["path"] == pkg.SGEMM_ALGO_TF32X3      # more than 32 rows
    assert plan(32, 4096, 27, algo=pkg.SGEMM_ALGO_TF32X3)["wide"] == 0
    forced = plan(32, 4096, 64, algo=pkg.SGEMM_ALGO_FFMA, splits=2)
    assert forced["wide"] == 0 and forced["splits"] == 2             # a forced split keeps the tiled kernel


def test_transposed_and_batched_argument_checks(lib):
    """sgemm_t and sgemm_strided_batched reject bad arguments, numbered by
    position, before touching a device."""
    A, B, C = FAKE, FAKE + (1 << 20), FAKE + (2 << 20)
    t = pkg.sgemm_t
    assert t(2, 0, 4, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4) == -1
    assert t(0, -1, 4, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4) == -2
    assert t(0, 0, -1, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4) == -3
    assert t(1, 0, 8, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4) == -8     # A stored K x M needs lda >= M
    assert t(0, 1, 4, 4, 8, 1.0, A, 8, B, 4, 0.0, C, 4) == -10    # B stored N x K needs ldb >= K
    assert t(0, 0, 4, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 3) == -13
    assert t(0, 0, 4, 4, 4, 1.0, A, 4, B, 4, 0.0, C, 4, None, 7) == -15
    assert t(0, 0, 4, 4, 4, 1.0, None, 4, B, 4, 0.0, C, 4) == -7
    assert t(1, 1, 0, 4, 4, 1.0, A, 1, B, 4, 0.0, C, 4) == 0      # M = 0: nothing to do
    b = pkg.sgemm_strided_batched
    base = (0, 0, 4, 4, 4, 1.0, A, 4)
    assert b(*base, -1, B, 4, 0, 0.0, C, 4, 16, 2) == -9
    assert b(*base, 0, B, 4, -1, 0.0, C, 4, 16, 2) == -12
    assert b(*base, 0, B, 4, 0, 0.0, C, 4, 15, 2) == -16         # C matrices would overlap
    assert b(*base, 0, B, 4, 0, 0.0, C, 4, 16, -1) == -17
    assert b(*base, 0, B, 4, 0, 0.0, C, 3, 16, 2) == -15          # ldc, renumbered
    assert b(0, 0, 4, 4, 4, 1.0, A, 4, 0, B, 4, 0, 0.0, C, 4, 16, 2, None, 9) == -19
    assert b(*base, 0, B, 4, 0, 0.0, C, 4, 16, 0) == 0            # empty batch



def test_conv2d_argument_checks(lib):
    """sgemm_conv2d rejects bad geometry, numbered by position, before
    touching a device; an empty batch or no filters is a no-op."""
    X, W, Y = FAKE, FAKE + (1 << 24), FAKE + (2 << 24)

    def conv(nb=2, C=3, H=8, W_=8, F=4, KH=3, KW=3, sh=1, sw=1, ph=1, pw=1, dh=1, dw=1,
             x=X, w=W, y=Y, algo=0, alpha=1.0):
        return pkg.sgemm_conv2d(x, w, y, alpha=alpha, stride=(sh, sw), pad=(ph, pw), dil=(dh, dw), algo=algo,
                                shape=(nb, C, H, W_, F, KH, KW))

    assert conv(nb=-1) == -1
    assert conv(C=-1) == -2
    assert conv(H=0) == -3
    assert conv(W_=0) == -4
    assert conv(F=-1) == -5
    assert conv(KH=0) == -6
    assert conv(KW=0) == -7
    assert conv(sh=0) == -8
    assert conv(sw=0) == -9
    assert conv(ph=-1) == -10
    assert conv(pw=-1) == -11
    assert conv(dh=0) == -12
    assert conv(dw=0) == -13
    assert conv(KH=11, ph=1) == -6                     # dilated filter taller than the padded image
    assert conv(KW=3, dw=5, pw=0) == -7
    assert conv(F=33, algo=pkg.SGEMM_ALGO_FFMA) == -20     # the FFMA form takes at most 32 filters
    assert conv(C=8, algo=pkg.SGEMM_ALGO_FFMA) == -20      # ... and at most 64 taps (8 x 3 x 3 = 72)
    assert conv(algo=7) == -20
    assert conv(x=None) == -15
    assert conv(w=None) == -16
    assert conv(y=None) == -18
    assert conv(y=X + 64) == -18                       # Y overlaps X
    assert conv(C=70000, H=200, W_=200) == -2         # 32-bit offsets inside one image
    assert conv(nb=0) == 0 and conv(F=0) == 0
    assert pkg.sgemm_conv2d(X, W, Y, shape=(2, 3, 8, 8, 4, 3, 3), flags=2) == -21   # unknown flag bit
    assert pkg.conv2d_out_size(224, 224, 7, 7, (2, 2), (3, 3)) == (112, 112)
    assert pkg.conv2d_out_size(10, 9, 3, 2, (1, 2), (0, 1), (2, 3)) == (6, 4)


def _walk_units(p, M, N, K, sms):
    """The 3xTF32 kernel's unit sequence as its schedule documents it, per
    CTA: split-K units u = cta + i * grid (tile u / S, slice u % S, slice s
    covering K tiles [s*KT/S, (s+1)*KT/S)); or, with a split tail, whole
    tiles t = cta + i * grid below the whole waves, then one K slice of a
    tail tile for each of the first tail * slices CTAs.  Returns the
    (tile, k tile) pairs of every CTA."""
    tm, tn = p["tile_m"], p["tile_n"]
    tiles = -(-M // tm) * -(-N // tn)
    kt = -(-K // 16)
    grid = p["grid"] // 2 if p.get("pairs") else p["grid"]  # CTA pairs walk the units together
    per_cta = [[] for _ in range(grid)]
    if p["tail_tiles"] == 0:
        s = p["splits"]
        for cta in range(grid):
            for u in range(cta, p["units"], grid):
                t, sl = divmod(u, s)
                per_cta[cta].append([(t, k) for k in range(sl * kt // s, (sl + 1) * kt // s)])
    else:
        tail = p["tail_tiles"]
        ts = p["ws_bytes"] // (tail * tm * tn * 4)
        dp = tiles - tail
        for cta in range(grid):
            for t in range(cta, dp, grid):
                per_cta[cta].append([(t, k) for k in range(kt)])
            if cta < tail * ts:
                t, sl = divmod(cta, ts)
                per_cta[cta].append([(dp + t, k) for k in range(sl * kt // ts, (sl + 1) * kt // ts)])
    return tiles, kt, per_cta


@pytest.mark.parametrize("sms", [152, 148, 132])
def test_plan_schedules_cover_every_k_tile_once(sms):
    """Over a spread of shapes, forced split counts and both last-wave
    treatments, the planner's schedule covers every (tile, k tile) of C
    exactly once, hands no CTA more than 8 shared tiles (the sums a CTA can
    defer to its exit), and sizes the workspace to one slot per partial
    tile; whole-wave schedules run one CTA per SM."""
    import itertools
    shapes = [(1, 1, 1), (5, 7, 3), (64, 64, 16), (100, 300, 17), (256, 256, 256), (1023, 1021, 1025),
              (1024, 1024, 1024), (384, 14161, 1152), (256, 50176, 1024), (64, 559104, 147),
              (5120, 5120, 5120), (2048, 8192, 64), (130, 4000, 4096), (16, 100000, 512)]
    variants = [{}, {"splits": 2}, {"splits": 7}, {"splits": 16}, {"flags": pkg.SGEMM_FLAG_WHOLE_TILES},
                {"flags": pkg.SGEMM_FLAG_SPLIT_TAIL}]
    checked = 0
    for (M, N, K), kw in itertools.product(shapes, variants):
        p = plan(M, N, K, algo=pkg.SGEMM_ALGO_TF32X3, num_sms=sms, **kw)
        tiles, kt, per_cta = _walk_units(p, M, N, K, sms)
        seen = {}
        for units in per_cta:
            for unit in units:
                for tk in unit:
                    seen[tk] = seen.get(tk, 0) + 1
        assert len(seen) == tiles * kt and set(seen.values()) == {1}, (M, N, K, kw, p)
        if p["splits"] > 1:  # every unit is a partial tile
            assert max(len(u) for u in per_cta) <= 8, (M, N, K, kw, p)
        # walkers: CTAs, or CTA pairs (two CTAs of the grid each, sms / 2 of them)
        pw = 2 if p["pairs"] else 1
        walkers, slots = p["grid"] // pw, sms // pw
        if p["pairs"]:
            assert p["tile_m"] == 256 and p["tile_n"] == 256 and p["grid"] % 2 == 0
        if p["tail_tiles"] == 0:
            assert p["units"] == tiles * p["splits"]
            assert p["ws_bytes"] == (p["units"] * p["tile_m"] * p["tile_n"] * 4 if p["splits"] > 1 else 0)
            assert 1 <= walkers <= max(p["units"], 1)
            if p["splits"] == 1:
                assert walkers == min(p["units"], slots)
        else:
            tail = p["tail_tiles"]
            ts = p["ws_bytes"] // (tail * p["tile_m"] * p["tile_n"] * 4)
            assert walkers == slots and 0 < tail < slots and (tiles - tail) % slots == 0
            assert ts >= 2 and tail * ts <= slots and ts <= kt
            assert p["ws_bytes"] == tail * ts * p["tile_m"] * p["tile_n"] * 4
        checked += 1
    assert checked == len(shapes) * len(variants)


def test_binding_constants_match_the_header():
    """Every integer constant the header #defines (algorithms, flags, status
    codes) has the same value in the Python binding."""
    import re
    text = open(pkg.HEADER).read()
    defs = {}
    for name, expr in re.findall(r"^#define\s+(SGEMM_\w+)\s+(\(?[0-9][0-9 <()]*\)?)", text, re.M):
        shift = re.fullmatch(r"\(\s*(\d+)\s*<<\s*(\d+)\s*\)", expr.strip())
        defs[name] = int(shift.group(1)) << int(shift.group(2)) if shift else int(expr)
    assert len(defs) >= 12
    for name, value in defs.items():
        assert hasattr(pkg, name), f"{name} is in the header but not in the binding"
        assert getattr(pkg, name) == value, f"{name}: header {value}, binding {getattr(pkg, name)}"
    assert pkg.SGEMM_FLAG_TILE_ROWS(192) == (192 // 16) << 8


def test_binding_signatures_match_the_header():
    """The ctypes argument lists of the binding have one entry per parameter
    of each prototype in the header, with the matching C type class (int,
    float, 64-bit integer, pointer or stream), so no argument is marshalled
    into the wrong slot."""
    import re
    text = re.sub(r"/\*.*?\*/", "", open(pkg.HEADER).read(), flags=re.S)
    protos = dict(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sgemm\w*)\s*\(([^)]*)\)\s*;", text, flags=re.M))
    assert set(protos) == set(pkg.declared_functions())

    def kind(param: str) -> str:
        p = " ".join(param.split())
        if "*" in p or p.startswith("sgemm_stream_t"):
            return "ptr"
        if p.startswith("long long"):
            return "i64"
        if p.startswith("float"):
            return "f32"
        if p.startswith("int"):
            return "i32"
        raise AssertionError(f"unexpected parameter type: {param!r}")

    ct_kind = {ctypes.c_int: "i32", ctypes.c_float: "f32", ctypes.c_longlong: "i64", ctypes.c_void_p: "ptr"}
    for name, params in protos.items():
        assert name in pkg._SIGS, f"{name} has no ctypes signature"
        want = [] if params.strip() in ("", "void") else [kind(p) for p in params.split(",")]
        got = [ct_kind.get(a, "ptr") for a in pkg._SIGS[name][1]]
        assert got == want, f"{name}: binding {got}, header {want}"


@pytest.mark.parametrize("sms", [152, 132])
def test_ffma_plans_cover_every_k_tile_once(sms):
    """The FFMA path's plans under the same walk: the tiled kernel runs one
    unit per CTA (split-K slices included), the wide-N kernel strides its
    CTAs over 512-column blocks with the whole K; every (tile, k tile) is
    covered once and the split workspace holds one slot per partial tile."""
    import itertools
    shapes = [(1, 1, 1), (5, 7, 3), (32, 4096, 27), (32, 1605632, 64), (64, 559104, 147), (100, 300, 17),
              (1023, 1021, 1025), (1024, 1024, 1024), (5120, 5120, 5120), (129, 257, 4096), (4096, 4096, 4096),
              (2048, 2048, 2048), (3000, 5000, 700)]
    for (M, N, K), splits in itertools.product(shapes, (0, 2, 5)):
        p = plan(M, N, K, algo=pkg.SGEMM_ALGO_FFMA, splits=splits, num_sms=sms)
        assert p["path"] == pkg.SGEMM_ALGO_FFMA
        if p["tail_tiles"]:
            # 128 x 256 tiles with a split tail: one unit per CTA, whole
            # tiles first, then the K slices of the leftover tiles
            assert (p["tile_m"], p["tile_n"]) == (128, 256) and splits == 0
            tiles = -(-M // 128) * -(-N // 256)
            kt = -(-K // 16)
            tail = p["tail_tiles"]
            ts = p["ws_bytes"] // (tail * 128 * 256 * 4)
            dp = tiles - tail
            assert dp % sms == 0 and 0 < tail < sms and ts >= 2 and p["grid"] == p["units"] == dp + tail * ts
            per_cta = [[[(t, k) for k in range(kt)]] for t in range(dp)]
            per_cta += [[[(dp + u // ts, k) for k in range((u % ts) * kt // ts, (u % ts + 1) * kt // ts)]]
                        for u in range(tail * ts)]
            seen = {}
            for units in per_cta:
                for unit in units:
                    for tk in unit:
                        seen[tk] = seen.get(tk, 0) + 1
            assert len(seen) == tiles * kt and set(seen.values()) == {1}, (M, N, K, p)
            continue
        tiles, kt, per_cta = _walk_units(p, M, N, K, sms)
        seen = {}
        for units in per_cta:
            for unit in units:
                for tk in unit:
                    seen[tk] = seen.get(tk, 0) + 1
        assert len(seen) == tiles * kt and set(seen.values()) == {1}, (M, N, K, splits, p)
        if p["wide"]:
            # the bulk-copy form (aligned B rows and N) runs one CTA per SM
            per_sm = 1 if N % 4 == 0 else 2
            assert p["splits"] == 1 and p["grid"] == min(p["units"], per_sm * sms) and p["ws_bytes"] == 0
        else:
            assert p["grid"] == p["units"] == tiles * p["splits"]
            assert p["ws_bytes"] == (p["units"] * p["tile_m"] * p["tile_n"] * 4 if p["splits"] > 1 else 0)


def test_host_blocks_pipeline_policy():
    """sgemm_host's blocks: one GEMM below 64 MB; row blocks of 128-row
    multiples (the last one takes the remainder) that cover M, at most 12;
    column blocks for short, wide calls.  On the 3xTF32 path the timeline
    simulation with the planner's model picks, for 5120^3 with beta != 0 on
    152 SMs, a 256-row first block, six of 768 rows (60 CTA-pair tiles: one
    wave on 76 pairs) and a 256-row last block; the FFMA path keeps the
    fixed policy."""
    assert pkg.sgemm_host_blocks(1000, 1000, 1000, num_sms=152) == (0, [1000])
    assert pkg.sgemm_host_blocks(5120, 5120, 5120, beta=0.5, num_sms=152) == (0, [256] + [768] * 6 + [256])
    assert pkg.sgemm_host_blocks(5120, 5120, 5120, beta=0.5, algo=pkg.SGEMM_ALGO_FFMA, num_sms=152) == \
        (0, [1024, 1024, 1024, 1024, 512, 256, 256])
    for M, N, K, beta in [(2000, 3000, 2500, -0.75), (8192, 8192, 8192, 0.0), (4097, 5000, 3000, 1.0),
                          (16384, 16384, 16384, 0.0), (100000, 1024, 1024, 0.0), (600, 20000, 512, 0.0),
                          (513, 40000, 1024, 0.5)]:
        for algo in (pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA):
            axis, sizes = pkg.sgemm_host_blocks(M, N, K, beta=beta, algo=algo, num_sms=152)
            assert axis == 0 and 1 < len(sizes) <= 12 and sum(sizes) == M, (M, N, K, algo, sizes)
            assert all(s % 128 == 0 and s > 0 for s in sizes[:-1]) and sizes[-1] > 0, sizes
    axis, sizes = pkg.sgemm_host_blocks(200, 40000, 700, ldb=40008, ldc=40012, beta=0.5, num_sms=152)
    assert axis == 1 and sum(sizes) == 40000 and len(sizes) <= 12
    assert all(s % 1024 == 0 for s in sizes[:-1])
    assert pkg.library().sgemm_host_blocks(-1, 5, 5, 5, 5, 5, 1.0, 0.0, 0, 152, None, None, 0) == -1
    with pytest.raises(pkg.SgemmError):
        pkg.sgemm_host_blocks(10, 10, 10, lda=5, num_sms=152)
