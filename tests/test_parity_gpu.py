"""GPU parity: every path, through the C ABI, against the float64 oracle.

Acceptance rule (per element, both paths):
    |gpu - ref| <= 1e-4 * (|alpha| * sum_k |a_mk b_kn| + |beta c_mn|)
Small cases (ragged, several tiles, alignment and leading-dimension
variants) are checked on every element; the full-size workloads (square
5120, the six im2col shapes, the square sweep) on sampled rows, in the same
launch configuration the benchmark times.  Guard bands around A, B, C and
the ld padding of C must stay untouched; A and B must not change.
"""
from __future__ import annotations

import numpy as np
import pytest

import dense_fp32_matrix_05_gb300 as pkg
import oracle
from dense_fp32_matrix_05_gb300.workloads import (SKINNY_SHAPES, SWEEP_SIZES, WORKLOADS,
                                                  make_problem, random_problem, uniform)
from gpu_util import check_against_oracle, run_sgemm, sample_rows

pytestmark = pytest.mark.gpu

ALGOS = [pkg.SGEMM_ALGO_TF32X3, pkg.SGEMM_ALGO_FFMA]
ALGO_IDS = ["tf32x3", "ffma"]


@pytest.fixture(scope="module", autouse=True)
def gpu_ready():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    torch.cuda.synchronize()


def _with_c(p, seed=99):
    if p.beta != 0:
        p.C[:, :p.N] = uniform(np.random.default_rng(seed), p.M * p.N).reshape(p.M, p.N)
    return p


SMALL_SHAPES = [(1, 1, 1), (2, 3, 4), (7, 9, 5), (16, 16, 16), (17, 15, 33), (31, 33, 17),
                (63, 65, 64), (65, 63, 129), (127, 129, 31), (128, 128, 128), (129, 127, 65),
                (200, 300, 77), (257, 130, 160), (33, 515, 20), (300, 1, 40), (1, 300, 40)]


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
@pytest.mark.parametrize("shape", SMALL_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SMALL_SHAPES])
def test_small_ragged_shapes(algo, shape):
    M, N, K = shape
    p = _with_c(random_problem(M, N, K, alpha=1.5, beta=0.5, seed=M * 10007 + N * 101 + K))
    C, st = run_sgemm(p, algo)
    assert st == 0
    check_against_oracle(p, C, what=f"{shape} algo={algo}")


LAYOUTS = {
    "packed": dict(ld=(0, 0, 0), off=(0, 0, 0)),
    "odd_ld": dict(ld=(1, 3, 5), off=(0, 0, 0)),
    "ld_plus4": dict(ld=(4, 4, 4), off=(0, 0, 0)),
    "misaligned_ptrs": dict(ld=(0, 0, 0), off=(1, 3, 2)),
    "odd_ld_misaligned": dict(ld=(3, 1, 7), off=(2, 1, 3)),
}


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("shape", [(100, 130, 36), (130, 260, 129), (33, 700, 27)])
def test_leading_dimensions_and_alignment(algo, layout, shape):
    M, N, K = shape
    L = LAYOUTS[layout]
    p = _with_c(random_problem(M, N, K, alpha=-0.75, beta=1.25, seed=M + N + K,
                               lda=K + L["ld"][0], ldb=N + L["ld"][1], ldc=N + L["ld"][2]))
    C, st = run_sgemm(p, algo, offsets=L["off"])
    assert st == 0
    check_against_oracle(p, C, what=f"{shape} {layout} algo={algo}")


BIG_FFMA_CASES = [  # (M, N, K, ld pads, offsets, splits, beta): >= 0.8 of a wave of 128 x 256 tiles
    (1100, 3900, 333, (0, 0, 0), (0, 0, 0), 0, 0.5), (1100, 3900, 333, (1, 3, 5), (0, 0, 0), 0, 1.25),
    (1030, 4000, 200, (0, 0, 0), (1, 3, 2), 0, 0.5), (1100, 3900, 160, (0, 0, 0), (0, 0, 0), 3, 0.5),
    (1024, 4096, 64, (0, 0, 0), (0, 0, 0), 0, 0.0)]


@pytest.mark.parametrize("case", BIG_FFMA_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-ld{c[3]}-off{c[4]}-s{c[5]}"
                                                      for c in BIG_FFMA_CASES])
def test_ffma_large_tiles(case):
    """The FFMA path's 128 x 256 tiles (one CTA per SM, A transposed into
    shared memory): every element against the oracle over ragged edges in
    M, N and K, odd leading dimensions, misaligned pointers (4-byte copies),
    forced split-K and beta = 0 with NaN in the old C."""
    M, N, K, ld, off, splits, beta = case
    p = _with_c(random_problem(M, N, K, alpha=0.5, beta=beta, seed=M + N + K + splits, lda=K + ld[0],
                               ldb=N + ld[1], ldc=N + ld[2]))
    plan = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_FFMA, splits=splits, num_sms=0)
    assert (plan["tile_m"], plan["tile_n"]) == (128, 256), plan
    C, st = run_sgemm(p, pkg.SGEMM_ALGO_FFMA, splits=splits, offsets=off)
    assert st == 0
    check_against_oracle(p, C, what=f"{case} FFMA 128 x 256")


WIDE_CASES = [(32, 1605632 // 64, 27), (24, 1500 * 4, 27), (17, 5000, 64), (32, 4096 + 512 + 4, 48), (5, 20, 3)]


@pytest.mark.parametrize("case", WIDE_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}" for c in WIDE_CASES])
def test_wide_bulk_form_matches_cp_async_form(case):
    """The wide-N FFMA kernel's bulk-copy form (B rows and N 16-byte aligned:
    one loader warp, a 6-slab ring) against the oracle, and bit for bit the
    same as its cp.async form, which a B start 4 bytes off a 16-byte
    boundary selects (same arithmetic, same order); N tails that are and
    are not whole 512-column blocks, K tails."""
    M, N, K = case
    p = random_problem(M, N, K, alpha=-0.75, beta=0.5, seed=M + N + K, pad_value=0.0)
    p.C[:, :N] = uniform(np.random.default_rng(N), M * N).reshape(M, N)
    plan = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_FFMA, num_sms=0)
    assert plan["wide"] == 1
    bulk, st = run_sgemm(p, pkg.SGEMM_ALGO_FFMA)
    assert st == 0
    check_against_oracle(p, bulk, what=f"{case} bulk-copy wide form")
    cp, st = run_sgemm(p, pkg.SGEMM_ALGO_FFMA, offsets=(0, 1, 0))
    assert st == 0
    assert np.array_equal(bulk.view(np.uint32), cp.view(np.uint32)), f"{case}: bulk and cp.async forms differ"


C_PAD_CASES = [(17, 15, 33, 20), (200, 301, 77, 304), (130, 1021, 64, 1024), (65, 255, 129, 260), (300, 14161, 40, 14164)]


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
@pytest.mark.parametrize("case", C_PAD_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-ldc{c[3]}" for c in C_PAD_CASES])
def test_c_rows_aligned_but_n_ragged(algo, case):
    """C rows 16-byte aligned (ldc % 4 == 0) while N is not a multiple of 4:
    the padding floats right after each row's last column must stay as they
    were (a TMA store would write the whole last 16-byte unit of a row)."""
    M, N, K, ldc = case
    for beta in (0.0, 0.5):
        p = _with_c(random_problem(M, N, K, alpha=1.25, beta=beta, seed=M + N + ldc, ldc=ldc))
        C, st = run_sgemm(p, algo)
        assert st == 0
        check_against_oracle(p, C, what=f"{case} beta={beta}")


@pytest.mark.parametrize("rows", [64, 256])
def test_tma_and_load_paths_agree_bitwise(rows):
    """Operands copied by TMA keep their raw fp32 words as the hi part (the
    tensor core reads only the top 19 bits of a tf32 operand); operands the
    producers load themselves get hi with the low 13 bits cleared.  Both must
    give the same bits: aligned and misaligned copies of the same problem
    take the two paths with the same schedule and summation order (single
    CTAs: a CTA pair copies both operands by TMA)."""
    M, N, K = 300, 392, 700  # lda and ldb multiples of 4: offset 0 is 16-byte aligned
    p = _with_c(random_problem(M, N, K, alpha=1.0, beta=0.5, seed=rows, pad_value=0.0))
    flags = pkg.SGEMM_FLAG_TILE_ROWS(rows) | pkg.SGEMM_FLAG_WHOLE_TILES | pkg.SGEMM_FLAG_NO_PAIRS
    outs = {}
    # NO_A_COPY: a misaligned A is loaded by the producers, not staged
    for off in [(0, 0, 0), (1, 0, 0), (0, 1, 0), (1, 1, 0)]:
        C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, offsets=off, flags=flags | pkg.SGEMM_FLAG_NO_A_COPY)
        assert st == 0
        outs[off] = C.view(np.uint32)
    check_against_oracle(p, outs[(0, 0, 0)].view(np.float32), what=f"rows={rows} aligned")
    for off, c in outs.items():
        assert np.array_equal(c, outs[(0, 0, 0)]), f"offsets {off} differ from the TMA path"


B4_CASES = [  # (M, N, K, ldb - N, tile rows): B rows not 16-byte aligned, several K tails
    (300, 1021, 700, 0, 128), (384, 1413, 1152, 0, 192), (130, 517, 37, 0, 256), (65, 263, 5, 2, 64),
    (200, 333, 4, 2, 32), (97, 130, 129, 0, 16), (257, 901, 300, 2, 256), (33, 14161, 64, 0, 64)]


@pytest.mark.parametrize("case", B4_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}+{c[3]}-tm{c[4]}" for c in B4_CASES])
def test_unaligned_b_rows_by_tma(case):
    """A B whose rows are not 16-byte aligned comes by TMA as four residue
    classes of rows (k % 4), each class's rows read from a few floats into
    the copied box.  Against the oracle, and bit for bit the same as the
    producers loading B themselves (SGEMM_FLAG_B_ROWS_LOADED), on whole-tile
    and split-K schedules."""
    M, N, K, pad, rows = case
    p = _with_c(random_problem(M, N, K, alpha=1.25, beta=0.5, seed=M + 7 * N + K, ldb=N + pad, pad_value=np.nan))
    assert p.ldb % 4 != 0
    for sched in (pkg.SGEMM_FLAG_WHOLE_TILES, 0):
        # single CTAs on both sides (residue classes on CTA pairs: test_cta_pairs)
        flags = pkg.SGEMM_FLAG_TILE_ROWS(rows) | sched | pkg.SGEMM_FLAG_NO_PAIRS
        splits = 0 if sched else 3
        tma, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=splits, flags=flags)
        assert st == 0
        check_against_oracle(p, tma, what=f"{case} residue-class TMA, splits {splits}")
        loaded, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=splits, flags=flags | pkg.SGEMM_FLAG_B_ROWS_LOADED)
        assert st == 0
        assert np.array_equal(tma.view(np.uint32), loaded.view(np.uint32)), f"{case}: TMA and loaded B differ"


# CTA pairs (SGEMM_FLAG_PAIRS): (M, N, K, ldb padding, tile rows).  Ragged
# edges where one CTA of a pair has no rows of A (M below TM / 2 in the last
# tile row) or no columns of B (N % 256 <= 128), residue-class B, a plan with
# more tiles than pairs (whole waves plus a split tail).
PAIR_CASES = [(256, 256, 64, 0, 256), (300, 700, 200, 0, 256), (257, 129, 33, 0, 256), (100, 120, 48, 0, 256),
              (512, 1000, 1000, 3, 256), (400, 900, 301, 0, 192), (192, 300, 129, 1, 192), (90, 383, 70, 0, 192),
              (1280, 4352, 256, 0, 256)]


@pytest.mark.parametrize("case", PAIR_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}p{c[3]}t{c[4]}" for c in PAIR_CASES])
def test_cta_pairs(case):
    """Tiles on CTA pairs (one cta_group::2 MMA per pair, half of the A tile
    in each CTA) against the oracle on whole tiles, the planner's split tail
    and a forced split-K; whole tiles bit for bit the same as the single-CTA
    kernel with the same tile height."""
    M, N, K, pad, tm = case
    lda = (K + 3) // 4 * 4 + 4  # the pair form copies A by TMA: 16-byte rows
    p = _with_c(random_problem(M, N, K, alpha=0.75, beta=-0.5, seed=3 * M + N + K, lda=lda, ldb=N + pad,
                               pad_value=np.nan))
    base = pkg.SGEMM_FLAG_TILE_ROWS(tm) | pkg.SGEMM_FLAG_PAIRS
    # whole tiles (splits = 1: no split-K either), the planner's schedule
    # (split tail when there are more tiles than pairs), forced split-K
    for sched, splits in ((pkg.SGEMM_FLAG_WHOLE_TILES, 1), (pkg.SGEMM_FLAG_SPLIT_TAIL, 0), (0, 3)):
        flags = base | sched
        plan = pkg.sgemm_plan_info(M, N, K, A=0, B=0, C=0, lda=p.lda, ldb=p.ldb, algo=pkg.SGEMM_ALGO_TF32X3,
                                   splits=splits, flags=flags, beta=p.beta)
        assert plan["pairs"] == 1 and plan["tile_n"] == 256, plan
        got, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=splits, flags=flags)
        assert st == 0
        check_against_oracle(p, got, what=f"{case} pairs, flags {flags:#x} splits {splits}")
        if sched == pkg.SGEMM_FLAG_WHOLE_TILES:
            single, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=1, flags=flags & ~pkg.SGEMM_FLAG_PAIRS)
            assert st == 0
            diff = got.view(np.uint32) != single.view(np.uint32)
            assert not diff.any(), (f"{case}: pair and single differ in {int(diff.sum())} elements, max "
                                    f"{float(np.nanmax(np.abs(got - single)))}, first at "
                                    f"{np.argwhere(diff)[:4].tolist()}")


def test_cta_pairs_with_staged_a():
    """An A whose rows are not 16-byte aligned but that is far smaller than
    B is copied to aligned rows before the kernel; the planner counts it as
    copied by TMA, so 256-row tiles can still run on CTA pairs."""
    M, N, K = 256, 9000, 147
    p = _with_c(random_problem(M, N, K, alpha=1.0, beta=0.5, seed=4242, pad_value=np.nan))
    assert p.lda % 4 != 0
    flags = pkg.SGEMM_FLAG_TILE_ROWS(256) | pkg.SGEMM_FLAG_PAIRS
    plan = pkg.sgemm_plan_info(M, N, K, A=0, B=0, C=0, lda=p.lda, ldb=p.ldb, algo=pkg.SGEMM_ALGO_TF32X3,
                               flags=flags, beta=p.beta)
    assert plan["pairs"] == 1 and plan["vec_a"] == 0, plan
    got, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, flags=flags)
    assert st == 0
    check_against_oracle(p, got, what="pairs with a staged A")
    single, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=1,
                           flags=pkg.SGEMM_FLAG_TILE_ROWS(256) | pkg.SGEMM_FLAG_NO_PAIRS | pkg.SGEMM_FLAG_WHOLE_TILES)
    assert st == 0
    whole, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=1, flags=flags | pkg.SGEMM_FLAG_WHOLE_TILES)
    assert st == 0
    assert np.array_equal(whole.view(np.uint32), single.view(np.uint32))


def test_cta_pairs_repeatable():
    """The pair form under load, run after run: whole 256 x 256 tiles over
    more tiles than pairs (several per pair), eight launches back to back,
    each bit for bit the single-CTA result; then the planner's schedule
    (split tail) twice, identical to itself and within the oracle's bound on
    sampled rows."""
    import torch
    M, N, K = 2304, 4608, 1536
    p = _with_c(random_problem(M, N, K, alpha=1.0, beta=0.5, seed=1234, pad_value=0.0))
    A, B = torch.from_numpy(p.A).cuda(), torch.from_numpy(p.B).cuda()
    C0 = torch.from_numpy(p.C).cuda()
    st = torch.cuda.current_stream()

    def call(flags, splits):
        C = C0.clone()
        assert pkg.sgemm_ex(M, N, K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, st,
                            pkg.SGEMM_ALGO_TF32X3, splits, flags) == 0
        return C

    whole = pkg.SGEMM_FLAG_TILE_ROWS(256) | pkg.SGEMM_FLAG_WHOLE_TILES
    single = call(whole | pkg.SGEMM_FLAG_NO_PAIRS, 1)
    outs = [call(whole | pkg.SGEMM_FLAG_PAIRS, 1) for _ in range(8)]
    assert pkg.sgemm_check_status(st) == 0
    for i, o in enumerate(outs):
        assert torch.equal(o, single), f"launch {i}: pair result differs from the single-CTA result"
    plan = pkg.sgemm_plan_info(M, N, K, A=A.data_ptr(), B=B.data_ptr(), C=C0.data_ptr(), algo=pkg.SGEMM_ALGO_TF32X3,
                               beta=p.beta)
    assert plan["pairs"] == 1
    a, b = call(0, 0), call(0, 0)
    assert pkg.sgemm_check_status(st) == 0
    assert torch.equal(a, b)
    rows = sample_rows(M, 24, seed=5)
    check_against_oracle(p, a.cpu().numpy(), rows=rows, what="pairs, planner schedule")


def test_unaligned_b_rows_batched_and_misaligned_start():
    """The residue-class maps with a batch dimension (a B stride that is a
    multiple of 4 floats), and a B whose start is not 16-byte aligned (the
    producers load it): both against the oracle."""
    import torch
    M, N, K, batch = 150, 389, 203, 3
    ps = [_with_c(random_problem(M, N, K, alpha=0.5, beta=0.25, seed=60 + b, pad_value=0.0), seed=70 + b)
          for b in range(batch)]
    for p in ps[1:]:
        p.A = ps[0].A
    sB = (K * N + 3) // 4 * 4 + 8
    sC = M * N + 5
    hB = np.full(sB * batch, np.nan, np.float32)
    hC = np.zeros(sC * batch, np.float32)
    for b, p in enumerate(ps):
        hB[b * sB:b * sB + K * N] = p.B.reshape(-1)
        hC[b * sC:b * sC + M * N] = p.C.reshape(-1)
    dA = torch.from_numpy(ps[0].A).cuda()
    dB, dC = torch.from_numpy(hB).cuda(), torch.from_numpy(hC).cuda()
    st = torch.cuda.current_stream()
    rc = pkg.sgemm_strided_batched(0, 0, M, N, K, 0.5, dA, K, 0, dB, N, sB, 0.25, dC, N, sC, batch, st,
                                   pkg.SGEMM_ALGO_TF32X3)
    assert rc == 0 and pkg.sgemm_check_status(st) == 0
    out = dC.cpu().numpy()
    for b, p in enumerate(ps):
        check_against_oracle(p, out[b * sC:b * sC + M * N].reshape(M, N), what=f"batched residue classes, {b}")
    p = _with_c(random_problem(M, N, K, alpha=1.0, beta=0.5, seed=5, pad_value=np.nan))
    C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, offsets=(0, 1, 0))
    assert st == 0
    check_against_oracle(p, C, what="B start not 16-byte aligned")


@pytest.mark.parametrize("shape", [(40, 2000, 147), (64, 4096, 27), (17, 3000, 333)],
                         ids=["40x2000x147", "64x4096x27", "17x3000x333"])
def test_unaligned_a_is_staged(shape):
    """An A with unaligned rows that is far smaller than B is copied to
    aligned rows and comes by TMA: against the oracle, and bit for bit the
    same as the producers loading it themselves (SGEMM_FLAG_NO_A_COPY)."""
    M, N, K = shape
    p = _with_c(random_problem(M, N, K, alpha=0.75, beta=0.5, seed=M + N, lda=K + (2 if (K + 1) % 4 == 0 else 1),
                               pad_value=np.nan))
    assert p.lda % 4 != 0
    staged, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3)
    assert st == 0
    check_against_oracle(p, staged, what=f"{shape} staged A")
    loaded, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, flags=pkg.SGEMM_FLAG_NO_A_COPY)
    assert st == 0
    assert np.array_equal(staged.view(np.uint32), loaded.view(np.uint32)), "staged and loaded A differ"


TILE_ROWS = [16, 32, 64, 128, 192, 256]


@pytest.mark.parametrize("rows", TILE_ROWS)
@pytest.mark.parametrize("shape", [(300, 270, 200), (37, 1000, 45), (513, 129, 1100)],
                         ids=["300x270x200", "37x1000x45", "513x129x1100"])
def test_every_tile_height(rows, shape):
    """Each tensor-core kernel instantiation (C rows per tile) on ragged shapes
    spanning several tiles and pipeline wraps, with and without split-K."""
    M, N, K = shape
    p = _with_c(random_problem(M, N, K, alpha=1.25, beta=-0.5, seed=rows + M))
    for splits in (1, 3):
        C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=splits, flags=pkg.SGEMM_FLAG_TILE_ROWS(rows))
        assert st == 0
        check_against_oracle(p, C, what=f"{shape} rows={rows} splits={splits}")


TAIL_SHAPES = [(2560, 16384, 640), (8192, 8192, 256), (7000, 4700, 333)]


@pytest.mark.parametrize("shape", TAIL_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in TAIL_SHAPES])
def test_split_tail(shape):
    """Shapes whose leftover tiles after the whole waves are split along K,
    checked on sampled rows against the oracle and the whole-tile schedule."""
    M, N, K = shape
    p = _with_c(random_problem(M, N, K, alpha=1.0, beta=-0.75, seed=M ^ N ^ K, pad_value=0.0))
    tail = pkg.SGEMM_FLAG_SPLIT_TAIL
    info = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_TF32X3, flags=tail, num_sms=0)
    assert info["tail_tiles"] > 0
    rows = sample_rows(M, 40, seed=7)
    C_sk, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, flags=tail)
    assert st == 0
    check_against_oracle(p, C_sk, rows=rows, what=f"{shape} split tail")
    C_dp, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, flags=pkg.SGEMM_FLAG_WHOLE_TILES)
    assert st == 0
    check_against_oracle(p, C_dp, rows=rows, what=f"{shape} whole tiles")
    C_sk2, _ = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, flags=tail)
    assert np.array_equal(C_sk.view(np.uint32), C_sk2.view(np.uint32)), "split tail is not deterministic"


@pytest.mark.parametrize("K", [2048, 2047])
def test_many_split_units_per_sm(K):
    """Forced split counts that give more shared tiles than one CTA may
    finish: the planner then runs more CTAs than SMs, and every tile's
    partial sums still meet in one deferred sum."""
    import torch

    M, N = 1000, 2000
    p = _with_c(random_problem(M, N, K, alpha=0.5, beta=2.0, seed=K, pad_value=0.0))
    flags = pkg.SGEMM_FLAG_TILE_ROWS(64)
    info = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_TF32X3, splits=8, flags=flags, num_sms=0)
    assert info["splits"] == 8 and info["units"] == 16 * 16 * 8
    assert info["grid"] * 8 >= info["units"] and info["grid"] > torch.cuda.get_device_properties(0).multi_processor_count
    C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=8, flags=flags)
    assert st == 0
    check_against_oracle(p, C, rows=sample_rows(M, 40, seed=K), what=f"K={K} splits=8 rows=64")


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_forced_split_k(algo, splits):
    p = _with_c(random_problem(129, 257, 1000, alpha=1.0, beta=0.5, seed=5))
    C, st = run_sgemm(p, algo, splits=splits)
    assert st == 0
    check_against_oracle(p, C, what=f"splits={splits} algo={algo}")


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
@pytest.mark.parametrize("name", ["square256", "square1024", "ragged1023x1021x1025"])
def test_small_configs_full(algo, name):
    p = make_problem(name, pad_value=0.0)
    C, st = run_sgemm(p, algo)
    assert st == 0
    check_against_oracle(p, C, what=f"{name} algo={algo}")


@pytest.mark.parametrize("algo", [pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA], ids=["auto", "ffma"])
def test_square5120_sampled(algo):
    p = make_problem("square5120", pad_value=0.0)
    C, st = run_sgemm(p, algo)
    assert st == 0
    check_against_oracle(p, C, rows=sample_rows(p.M, 48, seed=1), what=f"square5120 algo={algo}")


@pytest.mark.parametrize("algo", [pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA], ids=["auto", "ffma"])
@pytest.mark.parametrize("shape", SKINNY_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in SKINNY_SHAPES])
def test_skinny_shapes_sampled(algo, shape):
    M, N, K = shape
    p = make_problem(f"skinny{M}x{N}x{K}", pad_value=0.0)
    C, st = run_sgemm(p, algo)
    assert st == 0
    check_against_oracle(p, C, rows=sample_rows(M, 24, seed=2), what=f"{shape} algo={algo}")


@pytest.mark.parametrize("size", SWEEP_SIZES)
def test_sweep_sampled(size):
    p = make_problem(f"sweep{size}", pad_value=0.0)
    for algo in (pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA):
        C, st = run_sgemm(p, algo)
        assert st == 0
        check_against_oracle(p, C, rows=sample_rows(p.M, 12, seed=3), what=f"sweep{size} algo={algo}")


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
def test_deterministic_bits(algo):
    p = make_problem("square1024", pad_value=0.0)
    C1, _ = run_sgemm(p, algo)
    C2, _ = run_sgemm(p, algo)
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_small_integers_exact(algo, beta):
    rng = np.random.default_rng(31)
    M, N, K = 130, 260, 300
    p = random_problem(M, N, K, alpha=1.0, beta=beta, seed=1, pad_value=0.0)
    Ai = rng.integers(-8, 9, size=(M, K))
    Bi = rng.integers(-8, 9, size=(K, N))
    Ci = rng.integers(-8, 9, size=(M, N))
    p.A[:] = Ai
    p.B[:] = Bi
    p.C[:] = Ci
    C, st = run_sgemm(p, algo)
    assert st == 0
    want = Ai @ Bi + (Ci if beta else 0)
    assert np.array_equal(C, want.astype(np.float32))


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
def test_beta_zero_ignores_nan_c(algo):
    p = random_problem(150, 140, 50, alpha=2.0, beta=0.0, seed=3, pad_value=0.0)
    p.C[:] = np.nan
    C, st = run_sgemm(p, algo)
    assert st == 0 and np.all(np.isfinite(C))
    check_against_oracle(p, C, what="beta=0, C=NaN")


@pytest.mark.parametrize("alpha,K", [(0.0, 40), (1.0, 0)])
@pytest.mark.parametrize("beta", [0.0, 1.0, -2.5])
def test_alpha_or_k_zero(alpha, K, beta):
    M, N = 70, 90
    p = random_problem(M, N, max(K, 1), alpha=alpha, beta=beta, seed=4, pad_value=np.nan)
    p.K = K
    p.A[:] = np.nan
    p.B[:] = np.nan
    p.C[:, :N] = uniform(np.random.default_rng(5), M * N).reshape(M, N)
    C, st = run_sgemm(p)
    assert st == 0
    want = (beta * p.C[:, :N]) if beta != 0 else np.zeros((M, N), np.float32)
    assert np.array_equal(C[:, :N], want.astype(np.float32))


@pytest.mark.parametrize("algo", ALGOS, ids=ALGO_IDS)
def test_special_values(algo):
    M, N, K = 40, 48, 37
    p = random_problem(M, N, K, alpha=1.0, beta=0.5, seed=6, pad_value=0.0)
    p.C[:, :N] = uniform(np.random.default_rng(7), M * N).reshape(M, N)
    # partners that are exact tf32 values (their lo part is zero)
    p.B[3, :] = 0.5
    p.A[:, 9] = -2.0
    p.A[0, 3] = np.inf            # row 0: +-Inf wherever B[3, n] != 0
    p.A[1, 5] = np.nan            # row 1: NaN
    p.B[9, 7] = -np.inf           # column 7: -Inf * -2 = +Inf except rows 0 (Inf*0.5 + Inf)
    p.A[2, 0] = np.float32(3.0e37)
    p.A[4, :] = 0.0
    p.A[4, 2] = -0.0
    p.A[5, 1] = np.float32(1e-40)  # subnormal among normal terms
    p.B[1, 11] = np.float32(1e-39)
    p.C[6, 13] = np.nan            # beta * NaN = NaN
    C, st = run_sgemm(p, algo)
    assert st == 0
    check_against_oracle(p, C, what=f"special values algo={algo}")


def test_timeout_is_reported_and_recoverable():
    """A withheld pipeline arrive makes the bounded wait run out: the call
    reports SGEMM_ERR_DEVICE_TIMEOUT and the next call works normally."""
    p = random_problem(256, 256, 256, alpha=1.0, beta=0.0, seed=8, pad_value=0.0)
    _, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, flags=pkg.SGEMM_FLAG_DEBUG_WITHHOLD_ARRIVE)
    assert st == pkg.SGEMM_ERR_DEVICE_TIMEOUT
    C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3)
    assert st == 0
    check_against_oracle(p, C, what="after timeout")
    C, st = run_sgemm(p, pkg.SGEMM_ALGO_TF32X3, splits=4)
    assert st == 0
    check_against_oracle(p, C, what="split-K after timeout")


@pytest.mark.parametrize("algo", [pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA], ids=["auto", "ffma"])
def test_host_entry_point(algo):
    import torch
    p = _with_c(random_problem(300, 200, 150, alpha=1.5, beta=0.5, seed=9, pad_value=0.0))
    A = torch.from_numpy(p.A).pin_memory()
    B = torch.from_numpy(p.B).pin_memory()
    C = torch.from_numpy(p.C.copy()).pin_memory()
    rc = pkg.sgemm_host(p.M, p.N, p.K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta,
                        C.data_ptr(), p.ldc, algo)
    assert rc == 0
    check_against_oracle(p, C.numpy(), what=f"sgemm_host algo={algo}")
    # pageable numpy buffers work too
    Cn = p.C.copy()
    assert pkg.sgemm_host(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, Cn, p.ldc, algo) == 0
    check_against_oracle(p, Cn, what="sgemm_host pageable")


@pytest.mark.parametrize("algo", [pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA], ids=["auto", "ffma"])
def test_host_entry_point_pipelined(algo):
    """A call over 64 MB runs as row blocks whose copies overlap the GEMMs
    (padded leading dimensions; the blocks sgemm_host_blocks reports): rows
    on both sides of every block boundary against the oracle, pinned and
    pageable host buffers."""
    import torch
    M, N, K = 2000, 3000, 2500
    p = _with_c(random_problem(M, N, K, alpha=0.5, beta=-0.75, seed=19, lda=K + 4, ldb=N + 8, ldc=N + 4,
                               pad_value=0.0))
    axis, sizes = pkg.sgemm_host_blocks(M, N, K, p.lda, p.ldb, p.ldc, p.alpha, p.beta, algo)
    assert axis == 0 and len(sizes) > 1 and sum(sizes) == M
    edges = np.cumsum(sizes)[:-1]
    rows = sorted(set(sample_rows(M, 48, seed=3)) | {int(e) + d for e in edges for d in (-1, 0)} | {M - 1})
    A = torch.from_numpy(p.A).pin_memory()
    B = torch.from_numpy(p.B).pin_memory()
    C = torch.from_numpy(p.C.copy()).pin_memory()
    assert pkg.sgemm_host(M, N, K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(),
                          p.ldc, algo) == 0
    check_against_oracle(p, C.numpy(), rows=rows, what=f"pipelined sgemm_host algo={algo}")
    assert np.array_equal(C.numpy()[:, N:].view(np.uint32), p.C[:, N:].view(np.uint32)), "ldc padding written"
    Cn = p.C.copy()
    assert pkg.sgemm_host(M, N, K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta, Cn, p.ldc, algo) == 0
    assert np.array_equal(Cn.view(np.uint32), C.numpy().view(np.uint32)), "pageable and pinned calls differ"


def test_host_entry_point_column_blocks():
    """A short, wide call over 64 MB runs as column blocks with pitched
    copies (M = 200, N = 40000, padded ldb / ldc): columns on both sides of
    the block boundaries against the oracle, padding untouched."""
    import torch
    M, N, K = 200, 40000, 700
    p = _with_c(random_problem(M, N, K, alpha=1.25, beta=0.5, seed=23, ldb=N + 8, ldc=N + 12, pad_value=0.0))
    A = torch.from_numpy(p.A).pin_memory()
    B = torch.from_numpy(p.B).pin_memory()
    C = torch.from_numpy(p.C.copy()).pin_memory()
    assert pkg.sgemm_host(M, N, K, p.alpha, A.data_ptr(), p.lda, B.data_ptr(), p.ldb, p.beta, C.data_ptr(),
                          p.ldc, pkg.SGEMM_ALGO_AUTO) == 0
    check_against_oracle(p, C.numpy(), rows=sample_rows(M, 40, seed=5), what="column-block sgemm_host")
    assert np.array_equal(C.numpy()[:, N:].view(np.uint32), p.C[:, N:].view(np.uint32)), "ldc padding written"


def test_torch_matmul_and_streams():
    import torch
    a = torch.rand(513, 257, device="cuda") - 0.5
    b = torch.rand(257, 1025, device="cuda") - 0.5
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        c = pkg.matmul(a, b)
    s.synchronize()
    ref, scale = oracle.sgemm_ref(513, 1025, 257, 1.0, a.cpu().numpy(), 257, b.cpu().numpy(), 1025,
                                  0.0, None, 1025)
    assert not oracle.first_failures(c.cpu().numpy(), ref, scale)
    # column slices (ld > cols) through the tensor API
    big = torch.rand(300, 700, device="cuda")
    sub = big[:, 50:307]                      # 300 x 257, lda = 700
    bsub = b[:, 100:164]                      # 257 x 64, ldb = 1025
    cs = pkg.matmul(sub, bsub)
    ref, scale = oracle.sgemm_ref(300, 64, 257, 1.0, big.cpu().numpy()[:, 50:307].copy(), 257,
                                  bsub.cpu().numpy().copy(), 64, 0.0, None, 64)
    assert not oracle.first_failures(cs.cpu().numpy(), ref, scale)


def test_concurrent_calls_from_host_threads():
    """Four host threads call the library at the same time, each on its own
    stream, with plans that need the split-K workspace (forced slices, a
    split tail) or the aligned copy of an unaligned A.  Those buffers belong
    to a (device, stream) pair, so every thread's result must equal, bit for
    bit, the same call made alone, which in turn matches the oracle."""
    import threading
    import torch

    cases = [  # M, N, K, alpha, beta, algo, forced K slices
        (300, 700, 2048, 1.0, 0.5, pkg.SGEMM_ALGO_TF32X3, 4),
        (129, 513, 4096, 1.5, 0.0, pkg.SGEMM_ALGO_TF32X3, 8),
        (1023, 1021, 1025, 1.0, 1.0, pkg.SGEMM_ALGO_AUTO, 0),
        (64, 20000, 147, 1.0, 0.0, pkg.SGEMM_ALGO_AUTO, 0),
        (200, 300, 1000, 2.0, 0.5, pkg.SGEMM_ALGO_FFMA, 3),
    ]
    dev = []
    for i, (M, N, K, alpha, beta, algo, splits) in enumerate(cases):
        p = random_problem(M, N, K, alpha=alpha, beta=beta, seed=70 + i, pad_value=0.0)
        A = torch.from_numpy(p.A).cuda()
        B = torch.from_numpy(p.B).cuda()
        C0 = torch.from_numpy(p.C).cuda()
        dev.append((p, A, B, C0, algo, splits))

    def call(i, C, stream):
        p, A, B, _, algo, splits = dev[i]
        return pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, stream, algo,
                            splits, 0)

    solo = []
    for i, (p, _, _, C0, _, _) in enumerate(dev):
        C = C0.clone()
        st = torch.cuda.current_stream()
        assert call(i, C, st) == 0
        assert pkg.sgemm_check_status(st) == 0
        solo.append(C.cpu().numpy())
        check_against_oracle(p, solo[-1], what=f"solo {i}")

    reps, errors, outs = 6, [], {}

    def worker(t):
        try:
            s = torch.cuda.Stream()
            mine = []
            for r in range(reps):
                i = (t + r) % len(dev)
                C = dev[i][3].clone()  # the clone is ordered on the current stream, not s
                s.wait_stream(torch.cuda.current_stream())
                rc = call(i, C, s)
                if rc != 0:
                    errors.append((t, r, rc))
                    return
                mine.append((i, C))
            st = pkg.sgemm_check_status(s)
            if st != 0:
                errors.append((t, "status", st))
            s.synchronize()
            outs[t] = [(i, C.cpu().numpy()) for i, C in mine]
        except Exception as e:  # surfaced below
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert sorted(outs) == [0, 1, 2, 3]
    for t, res in outs.items():
        for i, C in res:
            assert np.array_equal(C.view(np.uint32), solo[i].view(np.uint32)), f"thread {t}, case {i}"


@pytest.mark.parametrize("n,splits", [(256, 4), (512, 0), (1024, 2)])
def test_back_to_back_dependent_calls(n, splits):
    """A chain of calls enqueued on one stream with no host synchronisation,
    each reading the previous call's output as its A: Y_{i+1} = Y_i W.  The
    tensor-core kernels may start while the kernel ahead of them finishes
    (programmatic dependent launch) and share the stream's split-K
    workspace, so any access before the predecessor completed would read a
    stale Y_i or a busy workspace.  An FFMA call in the middle of the chain
    puts a kernel without that launch mode between two with it.  Every link
    is checked against the oracle applied to the previous link's result."""
    import torch

    rng = np.random.default_rng(n + splits)
    W = (uniform(rng, n * n).reshape(n, n) / np.sqrt(n)).astype(np.float32)
    X = uniform(rng, n * n).reshape(n, n).astype(np.float32)
    dW = torch.from_numpy(W).cuda()
    ys = [torch.from_numpy(X).cuda()] + [torch.empty(n, n, device="cuda") for _ in range(8)]
    st = torch.cuda.current_stream()
    torch.cuda.synchronize()
    for i in range(8):
        algo = pkg.SGEMM_ALGO_FFMA if i == 4 else pkg.SGEMM_ALGO_TF32X3
        rc = pkg.sgemm_ex(n, n, n, 1.0, ys[i], n, dW, n, 0.0, ys[i + 1], n, st, algo,
                          splits if algo == pkg.SGEMM_ALGO_TF32X3 else 0, 0)
        assert rc == 0
    assert pkg.sgemm_check_status(st) == 0
    host = [y.cpu().numpy() for y in ys]
    for i in range(8):
        ref, scale = oracle.sgemm_ref(n, n, n, 1.0, host[i], n, W, n, 0.0, None, n)
        msg = oracle.first_failures(host[i + 1], ref, scale)
        assert not msg, f"link {i}: {msg}"


def test_plan_info_on_device_matches_sm_count():
    import torch
    props = torch.cuda.get_device_properties(0)
    info = pkg.sgemm_plan_info(5120, 5120, 5120, num_sms=0)
    assert info["grid"] == min(info["units"], props.multi_processor_count)


def test_tf32_mma_rate_is_plausible():
    """The tensor-core rate probe finishes with a plausible rate, narrower
    MMAs are not faster, and the 3xTF32 GEMM (three MMAs per product) at
    4096^3 does not beat a third of the probed rate by more than noise."""
    import time
    import torch

    rate = pkg.sgemm_tf32_mma_rate(256, 4000)
    assert 200.0 < rate < 5000.0, rate
    small = pkg.sgemm_tf32_mma_rate(64, 4000)
    assert 0.0 < small <= rate * 1.05
    M = N = K = 4096
    g = torch.Generator(device="cpu").manual_seed(0)
    A = (torch.rand(M, K, generator=g) * 2 - 1).cuda()
    B = (torch.rand(K, N, generator=g) * 2 - 1).cuda()
    C = torch.empty(M, N, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(2):
        assert pkg.sgemm(M, N, K, 1.0, A, K, B, N, 0.0, C, N, st) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(5):
        assert pkg.sgemm(M, N, K, 1.0, A, K, B, N, 0.0, C, N, st) == 0
    torch.cuda.synchronize()
    gemm = 2.0 * M * N * K * 5 / (time.perf_counter() - t0) / 1e12
    assert gemm < rate / 3.0 * 1.1, (gemm, rate)


WIDE_SHAPES = [(1, 1, 1), (3, 513, 1), (32, 1537, 27), (17, 5000, 64), (32, 70001, 16), (7, 130, 33)]


@pytest.mark.parametrize("layout", ["packed", "odd_ld", "misaligned_ptrs"])
@pytest.mark.parametrize("shape", WIDE_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in WIDE_SHAPES])
def test_wide_kernel(shape, layout):
    """The FFMA path's wide-N kernel (M <= 32, K <= 64): every element against
    the oracle, with 16-byte and 4-byte B copies, pair and single C stores,
    and beta 0 over a NaN-filled C as well as beta != 0."""
    M, N, K = shape
    L = LAYOUTS[layout]
    info = pkg.sgemm_plan_info(M, N, K, algo=pkg.SGEMM_ALGO_FFMA, num_sms=0)
    assert info["wide"] == 1
    for beta in (0.0, -0.5):
        p = _with_c(random_problem(M, N, K, alpha=-1.5, beta=beta, seed=M * N + K,
                                   lda=K + L["ld"][0], ldb=N + L["ld"][1], ldc=N + L["ld"][2]))
        if beta == 0.0:
            p.C[...] = np.nan
        C, st = run_sgemm(p, pkg.SGEMM_ALGO_FFMA, offsets=L["off"])
        assert st == 0
        check_against_oracle(p, C, what=f"{shape} {layout} beta={beta}")


def _stored(X, trans, ld_pad):
    """Row-major storage of X, or of X^T when trans, with ld_pad NaN columns."""
    S = X.T if trans else X
    rows, cols = S.shape
    out = np.full((rows, cols + ld_pad), np.nan, np.float32)
    out[:, :cols] = S
    return out, cols + ld_pad


TRANS_SHAPES = [(130, 260, 129), (257, 130, 160), (31, 500, 20), (64, 1000, 27)]


@pytest.mark.parametrize("algo", [pkg.SGEMM_ALGO_AUTO, pkg.SGEMM_ALGO_FFMA, pkg.SGEMM_ALGO_TF32X3],
                         ids=["auto", "ffma", "tf32x3"])
@pytest.mark.parametrize("trans", [(0, 1), (1, 0), (1, 1), (0, 0)], ids=["NT", "TN", "TT", "NN"])
@pytest.mark.parametrize("shape", TRANS_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in TRANS_SHAPES])
def test_transposed_operands(shape, trans, algo):
    """sgemm_t: A stored K x M and/or B stored N x K (padded leading
    dimensions full of NaN), every element against the oracle."""
    import torch

    M, N, K = shape
    ta, tb = trans
    p = _with_c(random_problem(M, N, K, alpha=0.75, beta=-1.25, seed=M + N + K + 2 * ta + tb))
    As, lda = _stored(p.A[:, :K], ta, 3)
    Bs, ldb = _stored(p.B[:, :N], tb, 5)
    dA, dB = torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda()
    dC = torch.from_numpy(p.C.copy()).cuda()
    st = torch.cuda.current_stream()
    assert pkg.sgemm_t(ta, tb, M, N, K, p.alpha, dA, lda, dB, ldb, p.beta, dC, p.ldc, st, algo) == 0
    assert pkg.sgemm_check_status(st) == 0
    check_against_oracle(p, dC.cpu().numpy(), what=f"{shape} trans={trans} algo={algo}")


FUSED_TB_SHAPES = [(130, 260, 129), (257, 130, 160), (300, 1000, 64), (64, 2000, 147), (1024, 1024, 1024),
                   (17, 333, 21)]


@pytest.mark.parametrize("ta", [0, 1], ids=["NT", "TT"])
@pytest.mark.parametrize("shape", FUSED_TB_SHAPES, ids=[f"{m}x{n}x{k}" for m, n, k in FUSED_TB_SHAPES])
def test_transposed_b_read_in_place(shape, ta):
    """A transposed B with 16-byte rows is read in place by the tensor
    kernel's transposed-B form (no transpose pass): every element against
    the oracle, ragged K and N included, and bit for bit the same as the
    row-major kernel on an explicitly transposed copy of B."""
    import torch

    M, N, K = shape
    p = _with_c(random_problem(M, N, K, alpha=1.25, beta=0.5, seed=M * 7 + N + K + ta))
    pad_a = 4 - (M if ta else K) % 4
    pad_b = 4 - K % 4  # ldb = K + pad_b: a multiple of 4
    As, lda = _stored(p.A[:, :K], ta, pad_a)
    Bs, ldb = _stored(p.B[:, :N], 1, pad_b)
    assert ldb % 4 == 0
    dA, dB = torch.from_numpy(As).cuda(), torch.from_numpy(Bs).cuda()
    dC = torch.from_numpy(p.C.copy()).cuda()
    st = torch.cuda.current_stream()
    assert pkg.sgemm_t(ta, 1, M, N, K, p.alpha, dA, lda, dB, ldb, p.beta, dC, p.ldc, st, pkg.SGEMM_ALGO_TF32X3) == 0
    assert pkg.sgemm_check_status(st) == 0
    got = dC.cpu().numpy()
    check_against_oracle(p, got, what=f"{shape} ta={ta} transposed B in place")
    # the same product with B materialised row-major (K x N, ldb a multiple of 4)
    Bn, ldn = _stored(p.B[:, :N], 0, 4 - N % 4)
    dC2 = torch.from_numpy(p.C.copy()).cuda()
    assert pkg.sgemm_t(ta, 0, M, N, K, p.alpha, dA, lda, torch.from_numpy(Bn).cuda(), ldn, p.beta, dC2, p.ldc, st,
                       pkg.SGEMM_ALGO_TF32X3) == 0
    torch.cuda.synchronize()
    assert np.array_equal(got.view(np.uint32), dC2.cpu().numpy().view(np.uint32)), "transposed-B form differs in bits"


@pytest.mark.parametrize("tb", [0, 1], ids=["B", "Bt"])
def test_strided_batched(tb):
    """A batch of 3 sharing one A (stride 0), with B and C strided past
    padding; each matrix of the batch against the oracle."""
    import torch

    M, N, K, batch = 100, 130, 64, 3
    ps = [_with_c(random_problem(M, N, K, alpha=1.5, beta=0.5, seed=40 + b), seed=70 + b) for b in range(batch)]
    for p in ps[1:]:
        p.A = ps[0].A
    lda = ps[0].lda
    stored = [_stored(p.B[:, :N], tb, 2) for p in ps]
    ldb = stored[0][1]
    sB = stored[0][0].size + 17
    sC = ps[0].C.size + 9
    hB = np.full(sB * batch, np.nan, np.float32)
    hC = np.full(sC * batch, np.nan, np.float32)
    for b in range(batch):
        hB[b * sB:b * sB + stored[b][0].size] = stored[b][0].reshape(-1)
        hC[b * sC:b * sC + ps[b].C.size] = ps[b].C.reshape(-1)
    dA = torch.from_numpy(np.ascontiguousarray(ps[0].A)).cuda()
    dB, dC = torch.from_numpy(hB).cuda(), torch.from_numpy(hC).cuda()
    st = torch.cuda.current_stream()
    rc = pkg.sgemm_strided_batched(0, tb, M, N, K, ps[0].alpha, dA, lda, 0, dB, ldb, sB, ps[0].beta, dC,
                                   ps[0].ldc, sC, batch, st)
    assert rc == 0 and pkg.sgemm_check_status(st) == 0
    out = dC.cpu().numpy()
    for b, p in enumerate(ps):
        C = out[b * sC:b * sC + p.C.size].reshape(p.C.shape)
        check_against_oracle(p, C, what=f"batch {b} tb={tb}")


# (M, N, K, batch, transa, transb, shared A, stride padding in floats, beta)
BATCH_CASES = [
    (200, 300, 96, 5, 0, 0, False, 0, 0.5),     # 16-byte strides: tensor-map copies of every matrix
    (200, 300, 96, 5, 0, 0, False, 3, 0.5),     # odd strides: element loads
    (256, 256, 2048, 2, 0, 0, False, 0, 0.0),   # few tiles, deep K: K slices of every matrix
    (512, 512, 1024, 10, 0, 0, True, 0, 1.0),   # 160 tiles: whole waves, then a split tail
    (130, 260, 129, 4, 1, 1, False, 1, 0.5),    # both operands transposed
    (130, 260, 129, 4, 1, 0, True, 0, 0.5),     # one transposed A shared by the batch
    (24, 3000, 27, 3, 0, 0, False, 0, 0.5),     # FFMA wide-N shape: matrix by matrix
    (130, 260, 128, 4, 0, 1, False, 0, 0.5),    # transposed B read in place over the batch
    (130, 260, 129, 3, 1, 1, True, 0, -1.0),    # transposed shared A copied, transposed B in place
]


@pytest.mark.parametrize("case", BATCH_CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}b{c[3]}t{c[4]}{c[5]}"
                                                   f"{'s' if c[6] else ''}p{c[7]}" for c in BATCH_CASES])
def test_strided_batched_one_launch(case):
    """Strided batches on the paths that run them in one launch; every
    matrix against the oracle, with the gaps between the C matrices checked
    untouched."""
    import torch

    M, N, K, batch, ta, tb, shared_a, pad, beta = case
    aligned = pad % 4 == 0  # leading dimensions and strides in whole 16-byte words

    def ld_pad(cols, odd):
        return 4 - cols % 4 if aligned else odd

    ps = [_with_c(random_problem(M, N, K, alpha=0.75, beta=beta, seed=300 + b,
                                 ldc=N + ld_pad(N, 3)), seed=400 + b) for b in range(batch)]
    if shared_a:
        for p in ps[1:]:
            p.A = ps[0].A
    sa = [_stored(p.A[:, :K], ta, ld_pad(M if ta else K, 1)) for p in ps]
    sb = [_stored(p.B[:, :N], tb, ld_pad(K if tb else N, 2)) for p in ps]
    lda, ldb, ldc = sa[0][1], sb[0][1], ps[0].ldc
    sA = 0 if shared_a else sa[0][0].size + pad
    sB = sb[0][0].size + pad
    sC = ps[0].C.size + pad + 4
    nA = 1 if shared_a else batch
    hA = np.full(max(sA, sa[0][0].size) * nA, np.nan, np.float32)
    hB = np.full(sB * batch, np.nan, np.float32)
    hC = np.full(sC * batch, np.float32(-7.5), np.float32)
    for b in range(batch):
        if b < nA:
            hA[b * sA:b * sA + sa[b][0].size] = sa[b][0].reshape(-1)
        hB[b * sB:b * sB + sb[b][0].size] = sb[b][0].reshape(-1)
        hC[b * sC:b * sC + ps[b].C.size] = ps[b].C.reshape(-1)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (hA, hB, hC))
    st = torch.cuda.current_stream()
    rc = pkg.sgemm_strided_batched(ta, tb, M, N, K, ps[0].alpha, dA, lda, sA, dB, ldb, sB, beta, dC, ldc, sC,
                                   batch, st)
    assert rc == 0 and pkg.sgemm_check_status(st) == 0
    out = dC.cpu().numpy()
    rows = sample_rows(M, 96, seed=M) if M * N * batch > 1 << 20 else None
    for b, p in enumerate(ps):
        C = out[b * sC:b * sC + p.C.size].reshape(p.C.shape)
        check_against_oracle(p, C, rows=rows, what=f"batch {b}")
        gap = out[b * sC + p.C.size:(b + 1) * sC]
        assert np.all(gap == np.float32(-7.5)), f"write between C matrices after batch {b}"


@pytest.mark.parametrize("shape,algo", [((1024, 1024, 1024), pkg.SGEMM_ALGO_AUTO),
                                        ((300, 5000, 200), pkg.SGEMM_ALGO_TF32X3),
                                        ((24, 3000, 27), pkg.SGEMM_ALGO_AUTO),
                                        ((257, 130, 160), pkg.SGEMM_ALGO_FFMA),
                                        ((40, 2000, 147), pkg.SGEMM_ALGO_TF32X3)],
                         ids=["1024-auto", "300x5000x200-tf32x3", "24x3000x27-wide", "257x130x160-ffma",
                              "40x2000x147-staged-A"])
def test_cuda_graph_capture_and_replay(shape, algo):
    """After one call has sized the library's buffers, calls can be captured
    into a CUDA graph on a side stream and replayed (beta = 0, so replays are
    idempotent); the result matches the oracle."""
    import torch

    M, N, K = shape
    p = random_problem(M, N, K, alpha=1.25, beta=0.0, seed=M + K, pad_value=0.0)
    A = torch.from_numpy(p.A).cuda()
    B = torch.from_numpy(p.B).cuda()
    C = torch.full(p.C.shape, float("nan"), device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert pkg.sgemm_ex(M, N, K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, side, algo, 0, 0) == 0
    side.synchronize()
    C.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(3):
            rc = pkg.sgemm_ex(M, N, K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, side, algo, 0, 0)
            assert rc == 0
    for _ in range(4):
        graph.replay()
    torch.cuda.synchronize()
    assert pkg.sgemm_check_status(side) == 0
    check_against_oracle(p, C.cpu().numpy(), what=f"graph {shape} algo={algo}")


@pytest.mark.parametrize("layer", [(2, 3, 20, 22, 16, 3, 3, 1), (1, 32, 12, 12, 48, 3, 3, 0),
                                   (2, 3, 17, 19, 64, 7, 7, 3)],
                         ids=["wide-ffma-padded", "channels-order", "tap-table-padded"])
def test_cuda_graph_capture_conv(layer):
    """sgemm_conv2d calls (filter staging and zero-bordered copies included)
    captured into a CUDA graph after one sizing call, then replayed."""
    import torch

    nb, C, H, W, F, KH, KW, pad = layer
    rng = np.random.default_rng(F + KH)
    X = (rng.random((nb, C, H, W), dtype=np.float32) * 2 - 1)
    Wt = (rng.random((F, C, KH, KW), dtype=np.float32) * 2 - 1)
    OH, OW = oracle.conv2d_out_size(H, W, KH, KW, (1, 1), (pad, pad))
    dX, dW = torch.from_numpy(X).cuda(), torch.from_numpy(Wt).cuda()
    Y = torch.full((nb, F, OH, OW), float("nan"), device="cuda")
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        assert pkg.sgemm_conv2d(dX, dW, Y, pad=(pad, pad), stream=side) == 0
    side.synchronize()
    Y.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(2):
            assert pkg.sgemm_conv2d(dX, dW, Y, pad=(pad, pad), stream=side) == 0
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert pkg.sgemm_check_status(side) == 0
    ref, scale = oracle.conv2d_ref(1.0, X, Wt, pad=(pad, pad))
    msg = oracle.first_failures(Y.cpu().numpy(), ref, scale)
    assert not msg, msg

