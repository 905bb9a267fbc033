"""SGEMM benchmark: TFLOP/s (2MNK / time) and fraction of the per-shape roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--algo auto|ffma|tf32x3] [--shapes-out FILE]

--workload conv...: one implicit-GEMM convolution layer per step
(sgemm_conv2d; the layers whose im2col GEMMs are the skinny workloads).

One step is one C = alpha*A*B + beta*C call on the workload (default
square5120: M=N=K=5120, alpha=1, beta=0.5, the size of the overview table of
"NVIDIA_SGEMM_PRACTICE"), inputs resident in HBM.  Inputs (315 MB) exceed the
129 MB L2, so no flush is needed between steps.  Rank 0 prints one JSON line.

  value     device time of K back-to-back steps, CUDA events on the launch
            stream, max over ranks; whole-job TFLOP/s = N * 2MNK * K / time.
            Workloads under twice the L2 (256^3 ... 2048^3, 384x14161x1152)
            flush it before every step instead (512 MB written, untimed) and
            sum per-step event pairs
  e2e       the same metric through sgemm_host() (host buffers, pinned): per
            step host->device copies of A, B, C, the GEMM, device->host C
  roofline  the GEMM kernel's 2MNK per launch / mean launch time (timed
            region over its steps) against the path's peak
  cpu_baseline  the float64 oracle on a bounded row sample, host cores
  per_shape every benchmark workload on both paths and every convolution
            layer, measured after the headline (value, roofline fraction,
            L2 mode, clocks); on by default for the square5120 run on one
            GPU, --no-per-shape leaves it out
--impl reference times the oracle alone (the pages publish no GPU code to
run here), same workload and metric.
Multi-GPU (torchrun): independent replicas, one per GPU ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import signal
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SGEMM TFLOP/s (2MNK/time) and % of per-shape roofline, 1×GB300"
UNIT = "TFLOP/s"
# The pages' own number for this metric and size: "NVIDIA_SGEMM_PRACTICE"
# overview table, kernel_7 (double-buffered prefetch), 5120^3, RTX 3090.
PAGES_5120_TFLOPS = 13.63498
# nominal dense tensor rates (per GPU): tf32 1.1 PFLOP/s, bf16 2.25 PFLOP/s
TF32_OVER_BF16 = 1.1 / 2.25
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "sm_max_mhz": 2070.0}
# The sources each kernel family's code comes from: a committed ncu summary
# records the hash of its family's sources, so work on one family does not
# retire the others' summaries.
_COMMON_SOURCES = ["dense_fp32_matrix_05_gb300/csrc/common.cuh", "dense_fp32_matrix_05_gb300/csrc/ptx.cuh"]
KERNEL_SOURCES = {
    "tf32x3": ["dense_fp32_matrix_05_gb300/csrc/tf32x3_gemm.cuh", "dense_fp32_matrix_05_gb300/csrc/tf32x3_gemm.cu",
               "dense_fp32_matrix_05_gb300/csrc/gemm_tb.cu", "dense_fp32_matrix_05_gb300/csrc/conv_gemm.cu"]
              + _COMMON_SOURCES,
    "ffma": ["dense_fp32_matrix_05_gb300/csrc/ffma_gemm.cuh", "dense_fp32_matrix_05_gb300/csrc/ffma_gemm.cu"]
            + _COMMON_SOURCES,
    "ffma_wide": ["dense_fp32_matrix_05_gb300/csrc/ffma_wide.cu"] + _COMMON_SOURCES,
}
L2_FLUSH_BYTES = 512 << 20  # written between timed steps of workloads that fit in the 129 MB L2


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_family(path_name: str) -> str:
    """The kernel family of a summary name (tf32x3, tf32x3_NT, ffma_wide ...)."""
    return "ffma_wide" if path_name.startswith("ffma_wide") else ("ffma" if path_name.startswith("ffma") else "tf32x3")


def kernel_source_hash(family: str = "tf32x3") -> str:
    """Hash of one kernel family's source code: comments and blank lines are
    left out, so editing a comment does not retire a recorded ncu summary."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, rel)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            code = re.sub(r"//.*", "", line).rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profile_name(path_name: str, trans: str = "NN") -> str:
    """Name of the ncu summary for a path: a transposed form (sgemm_t with
    NT, TN or TT) runs another kernel instantiation and has its own."""
    return path_name if trans == "NN" else f"{path_name}_{trans}"


def recorded_traffic(workload: str, path_name: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (the summary records their hash)."""
    fn = os.path.join(ROOT, "profiles", f"{path_name}_{workload}.md")
    if not os.path.exists(fn):
        return None
    text = open(fn).read()
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash(kernel_family(path_name)):
        return None
    return float(m_bytes.group(1))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL, start_new_session=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            try:
                os.killpg(self.proc.pid, signal.SIGTERM)
            except Exception:
                self.proc.terminate()
            self.proc.wait(timeout=10)

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, flags in rows for i, v in enumerate(flags)
                          if v.lower() == "active"})
        return {"sm_mhz": float(np.median([r[0] for r in rows])), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


_MMA_RATE = {}
_FFMA_RATE = {}


def ffma_rate(pkg):
    """fp32 TFLOP/s of packed fma.rn.f32x2 on this GPU (measured once)."""
    if "v" not in _FFMA_RATE:
        try:
            _FFMA_RATE["v"] = pkg.sgemm_ffma_rate(True, 20000)
        except Exception as exc:  # reported, not fatal: the formula peak stands
            log(f"FFMA rate probe failed: {exc}")
            _FFMA_RATE["v"] = None
    return _FFMA_RATE["v"]


def tf32_mma_rate(pkg) -> float:
    """Raw tf32 TFLOP/s of the kernel's MMA form on this GPU (measured once)."""
    if "v" not in _MMA_RATE:
        try:
            _MMA_RATE["v"] = pkg.sgemm_tf32_mma_rate(256, 20000)
        except Exception as exc:  # reported, not fatal: the contract's peak stands
            log(f"tf32 MMA rate probe failed: {exc}")
            _MMA_RATE["v"] = None
    return _MMA_RATE["v"]


# launch-bound sizes: also timed as back-to-back launches replayed from a CUDA graph
GRAPH_WORKLOADS = ("square256", "square1024", "ragged1023x1021x1025")


def graph_rate(pkg, p, A, B, C, algo: int, flops: float, per_graph: int = 20, replays: int = 10) -> dict:
    """TFLOP/s of `per_graph` GEMMs captured into one CUDA graph (after the
    timed region has sized every library buffer), replayed `replays` times
    between CUDA events."""
    import torch

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    # one plain call on the capture stream sizes its buffers (no allocation may happen while capturing)
    rc = pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, side, algo, 0, 0)
    if rc != 0:
        raise pkg.SgemmError("sgemm_ex (graph warm-up)", rc)
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(per_graph):
            rc = pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, side, algo, 0, 0)
            if rc != 0:
                raise pkg.SgemmError("sgemm_ex (graph capture)", rc)
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (replays * per_graph)
    st = pkg.sgemm_check_status(side)
    if st != 0:
        raise pkg.SgemmError("graph replay", st)
    return {"value": round(flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT, "ms_per_gemm": round(ms, 5),
            "gemms_per_graph": per_graph, "replays": replays,
            "note": "context: repeated GEMMs on the same operands, which stay L2-resident"}


def copy_bound(hA, hB, hC, A, B, C, read_c: bool, stream, reps: int = 3, rounds: int = 4) -> dict:
    """The host-link floor of one end-to-end step: the same bytes sgemm_host
    moves (A, B and, when beta != 0, C up; C down), as plain pinned copies
    timed with CUDA events, best of `rounds` rounds of `reps` copies.  Up
    and down are timed alone and together on two streams; the floor is the
    slower direction alone (the step's copies can at best overlap each other
    and the GEMM), and the concurrent pair is reported beside it."""
    import torch
    down = torch.cuda.Stream()

    def up_copies():
        A.copy_(hA, non_blocking=True)
        B.copy_(hB, non_blocking=True)
        if read_c:
            C.copy_(hC, non_blocking=True)

    def timed(fn):
        best = float("inf")
        for _ in range(rounds):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1) / reps)
        return best

    def down_copy():
        hC.copy_(C, non_blocking=True)

    def both():
        down.wait_stream(stream)
        with torch.cuda.stream(down):
            hC.copy_(C, non_blocking=True)
        up_copies()
        stream.wait_stream(down)

    with torch.cuda.stream(stream):
        up_ms = timed(up_copies)
        down_ms = timed(down_copy)
        both_ms = timed(both)
    up_b = 4 * (hA.numel() + hB.numel() + (hC.numel() if read_c else 0))
    down_b = 4 * hC.numel()
    return {"h2d_ms": round(up_ms, 4), "d2h_ms": round(down_ms, 4), "both_ms": round(both_ms, 4),
            "h2d_gbs": round(up_b / (up_ms * 1e-3) / 1e9, 1), "d2h_gbs": round(down_b / (down_ms * 1e-3) / 1e9, 1),
            "copy_bound_ms": round(max(up_ms, down_ms), 4),
            "note": "pinned cudaMemcpyAsync of the step's bytes, best of rounds; floor = slower direction "
                    "alone; both_ms = up and down at once on two streams"}


def max_over_ranks(local_ms: float, device=None) -> float:
    """The job's time: the largest of the ranks' timed regions (every rank
    calls this; device None means a single process).  The tensor lives on
    `device`: the GPU under NCCL, the CPU under gloo."""
    if device is None:
        return local_ms
    import torch
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_step: float, steps: int, job_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs `steps` GEMMs of `flops_per_step`
    (replicas, weak scaling) within the job's time."""
    return world * flops_per_step * steps / (job_ms * 1e-3) / 1e12


def pipeline_bound(copy: dict, prefix_bytes: float, gemm_ms: float, step_ms: float) -> dict:
    """Floor of one pipelined host-buffer call: the smaller of A and B goes
    up whole before the first block's GEMM can start (sgemm_host's row
    blocks send B first, its column blocks A), after which the other copies
    can overlap the GEMMs; and never less than the copy floor."""
    prefix_ms = prefix_bytes / (copy["h2d_gbs"] * 1e9) * 1e3
    bound = max(copy["copy_bound_ms"], prefix_ms + gemm_ms)
    return {"pipeline_bound_ms": round(bound, 4), "frac_of_pipeline_bound": round(bound / step_ms, 4),
            "pipeline_note": "max(copy floor, upload of the smaller of A and B + the GEMM's device time)"}


def roofline_peak(path: int, peaks: dict, source: str, sms: int):
    """(bound, peak TFLOP/s, basis text) for a path."""
    import dense_fp32_matrix_05_gb300 as pkg
    if path == pkg.SGEMM_ALGO_TF32X3:
        tf32 = peaks["bf16_tflops"] * TF32_OVER_BF16
        return ("tensor", tf32 / 3.0,
                f"3xTF32 fp32-accurate tensor peak = {source} bf16 burst {peaks['bf16_tflops']} TF/s "
                f"x (tf32 1.1 / bf16 2.25 nominal) / 3 MMAs per fp32 product "
                f"(raw tf32 peak {tf32:.1f} TF/s)")
    mhz = peaks.get("sm_max_mhz", 2070.0)
    formula = sms * 128 * 2 * mhz * 1e6 / 1e12
    measured = ffma_rate(pkg)
    if measured:
        return ("alu", measured,
                f"FFMA peak measured by sgemm_ffma_rate (packed fma.rn.f32x2, 2048 threads x 16 chains per SM): "
                f"{measured:.1f} TF/s; formula {sms} SMs x 128 fp32 lanes x 2 flop x {mhz} MHz = {formula:.1f}")
    return ("alu", formula, f"FFMA peak = {sms} SMs x 128 fp32 lanes x 2 flop x {mhz} MHz ({source} max clock)")


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch

    import dense_fp32_matrix_05_gb300 as pkg
    from dense_fp32_matrix_05_gb300.workloads import WORKLOADS, make_problem

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from dense_fp32_matrix_05_gb300 import _build_ext
    _build_ext.build()
    pkg.library()
    w = WORKLOADS[args.workload]
    algo = {"auto": 0, "ffma": 1, "tf32x3": 2}[args.algo]
    p = make_problem(w, pad_value=0.0)
    A = torch.from_numpy(p.A).to(dev)
    B = torch.from_numpy(p.B).to(dev)
    C = torch.from_numpy(p.C).to(dev)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    plan = pkg.sgemm_plan_info(p.M, p.N, p.K, A.data_ptr(), p.lda, B.data_ptr(), p.ldb,
                               C.data_ptr(), p.ldc, algo=algo, num_sms=props.multi_processor_count)
    flops = 2.0 * p.M * p.N * p.K

    ta, tb = (args.trans[0] == "T"), (args.trans[1] == "T")
    if ta or tb:
        # transposed storage: A as K x M, B as N x K (sgemm_t copies them back)
        At = A[:, :p.K].t().contiguous() if ta else A
        Bt = B[:, :p.N].t().contiguous() if tb else B
        lda_t = p.M if ta else p.lda
        ldb_t = p.K if tb else p.ldb

    def step():
        if ta or tb:
            rc = pkg.sgemm_t(int(ta), int(tb), p.M, p.N, p.K, p.alpha, At, lda_t, Bt, ldb_t, p.beta, C, p.ldc,
                             stream, algo)
        else:
            rc = pkg.sgemm_ex(p.M, p.N, p.K, p.alpha, A, p.lda, B, p.ldb, p.beta, C, p.ldc, stream, algo, 0, 0)
        if rc != 0:
            raise pkg.SgemmError("sgemm_t" if (ta or tb) else "sgemm_ex", rc)

    for _ in range(args.warmup):
        step()
    st = pkg.sgemm_check_status(stream)
    if st != 0:
        raise pkg.SgemmError("warmup", st)

    dist = world > 1
    # Workloads whose compulsory bytes are under twice the 129 MB L2 get the
    # L2 flushed before every step (a 512 MB write, outside the timed region),
    # so that each launch reads its operands from HBM; each step then has its
    # own pair of events and the value is the sum of the step times.  Larger
    # workloads run their K steps back to back on the stream between two
    # events, as a caller issues them: no event between launches, which would
    # keep programmatic dependent launch from overlapping a launch's set-up
    # with the previous kernel's tail.  A step is one kernel launch (plus the
    # transposes of a transposed A, or of B off the tensor path).
    flush = w.compulsory_bytes < 2 * 129e6
    back_to_back = None
    if flush:
        # context only: the same launches back to back on L2-resident operands
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for _ in range(args.steps):
            step()
        b1.record(stream)
        torch.cuda.synchronize()
        back_to_back = b0.elapsed_time(b1) / args.steps
        fbuf = torch.empty(L2_FLUSH_BYTES // 4, device=dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        if flush:
            for i in range(args.steps):
                fbuf.zero_()
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
        else:
            t0.record(stream)
            for _ in range(args.steps):
                step()
            t1.record(stream)
        torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    total_ms = float(np.sum([a.elapsed_time(b) for a, b in ev])) if flush else t0.elapsed_time(t1)
    launch_ms = total_ms / args.steps
    st = pkg.sgemm_check_status(stream)
    if st != 0:
        raise pkg.SgemmError("timed region", st)
    total_ms = max_over_ranks(total_ms, dev if dist else None)
    clocks = clk.summary()

    # ---------------------------------------------------------- e2e
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    hA = torch.from_numpy(p.A).pin_memory()
    hB = torch.from_numpy(p.B).pin_memory()
    hC = torch.from_numpy(p.C.copy()).pin_memory()

    def host_step():
        rc = pkg.sgemm_host(p.M, p.N, p.K, p.alpha, hA.data_ptr(), p.lda, hB.data_ptr(), p.ldb,
                            p.beta, hC.data_ptr(), p.ldc, algo)
        if rc != 0:
            raise pkg.SgemmError("sgemm_host", rc)

    for _ in range(min(3, args.warmup)):
        host_step()
    torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    step_s = []
    h0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_step()
        step_s.append(time.perf_counter())
    e2e_s = step_s[-1] - h0
    step_s = np.diff([h0] + step_s)
    if dist:
        t = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())
    h2d = 4 * (p.A.size + p.B.size + (p.C.size if p.beta != 0 else 0))
    d2h = 4 * p.C.size
    copy = copy_bound(hA, hB, hC, A, B, C, p.beta != 0, stream)

    # ---------------------------------------------------------- context: cuBLAS SGEMM
    cublas = None
    if args.cublas and rank == 0:
        torch.backends.cuda.matmul.allow_tf32 = False
        a2 = A[:, :p.K]
        b2 = B[:, :p.N]
        out = torch.empty((p.M, p.N), device=dev)
        for _ in range(3):
            torch.matmul(a2, b2, out=out)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = max(3, min(args.steps, 50))
        c0.record()
        for _ in range(n):
            torch.matmul(a2, b2, out=out)
        c1.record()
        torch.cuda.synchronize()
        cublas = flops * n / (c0.elapsed_time(c1) * 1e-3) / 1e12

    peaks, peak_src = load_peaks()
    bound, peak, basis = roofline_peak(plan["path"], peaks, peak_src, props.multi_processor_count)
    # per-shape roofline: the slower of the path's compute peak and moving the
    # compulsory bytes at the measured HBM bandwidth
    t_compute = flops / (peak * 1e12)
    t_memory = w.compulsory_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_memory > t_compute:
        bound, peak, unit_r = "hbm", peaks["hbm_gbs"], "GB/s"
        achieved = w.compulsory_bytes / (launch_ms * 1e-3) / 1e9
        basis = f"{peak_src} HBM copy bandwidth {peaks['hbm_gbs']} GB/s (compulsory bytes / launch time)"
    else:
        unit_r = "TFLOP/s"
        achieved = flops / (launch_ms * 1e-3) / 1e12
    path_name = {1: "ffma", 2: "tf32x3"}[plan["path"]]
    kernel_name = "ffma_wide_kernel" if plan.get("wide") else f"{path_name}_gemm_kernel"
    if plan.get("wide"):
        path_name = "ffma_wide"
    traffic = recorded_traffic(args.workload, profile_name(path_name, args.trans))
    value = job_throughput(world, flops, args.steps, total_ms)

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": round(value / PAGES_5120_TFLOPS, 3) if args.workload == "square5120" else None,
        "vs_baseline_ref": "NVIDIA_SGEMM_PRACTICE overview table, kernel_7, 5120^3, RTX 3090, 13634.98 GFLOPS",
        "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": f"{w.name}: M={p.M} N={p.N} K={p.K} fp32 row-major, {w.note}",
            "algo": f"{args.algo} -> {path_name}",
            "tile": f"{plan['tile_m']}x{plan['tile_n']}", "splits": plan["splits"],
            "split_tail_tiles": plan.get("tail_tiles", 0),
            "grid": plan["grid"], "stages": plan["stages"],
            "l2": (f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB written, untimed; "
                   f"compulsory bytes {w.compulsory_bytes / 1e6:.0f} MB vs 129 MB L2)" if flush else
                   f"no flush: inputs larger than L2 ({w.compulsory_bytes / 1e6:.0f} MB vs 129 MB)"),
            "parallelism": f"replicas x{world}",
            "trans": args.trans,
        },
        "roofline": {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 3),
                     "unit": unit_r, "frac": round(achieved / peak, 4), "traffic": traffic,
                     "peak_basis": basis, "kernel": kernel_name,
                     "launch_ms": round(launch_ms, 5),
                     "launch_note": ("sum of per-step event pairs over the steps, L2 flushed before each step"
                                     if flush else
                                     "timed region over its steps: one launch per step, launches back to back"),
                     "compulsory_bytes": w.compulsory_bytes,
                     "hbm_frac_of_measured": round(w.compulsory_bytes / (launch_ms * 1e-3) /
                                                   (peaks["hbm_gbs"] * 1e9), 4)},
        "e2e": {"value": round(world * flops * e2e_steps / e2e_s / 1e12, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "api": "sgemm_host (pinned host buffers)",
                "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 4),
                "ms_per_step_median": round(float(np.median(step_s)) * 1e3, 4),
                "ms_per_step_max": round(float(np.max(step_s)) * 1e3, 4),
                "copy_bound_ms": copy["copy_bound_ms"],
                "frac_of_copy_bound": round(copy["copy_bound_ms"] / (e2e_s * 1e3 / e2e_steps), 4),
                "frac_of_concurrent_copies": round(copy["both_ms"] / (e2e_s * 1e3 / e2e_steps), 4),
                **pipeline_bound(copy, 4 * min(p.A.size, p.B.size), launch_ms, e2e_s * 1e3 / e2e_steps),
                "copies": copy},
        "gpu_launches": args.steps * (1 + int(ta) + int(tb)),
        "clocks": clocks,
    }
    if cublas is not None:
        result["context_cublas_sgemm_tflops"] = round(cublas, 3)
    if back_to_back is not None:
        # not the value: the operands stay in L2 from one launch to the next
        result["context_back_to_back_l2_resident"] = {
            "value": round(flops / (back_to_back * 1e-3) / 1e12, 3), "unit": UNIT,
            "launch_ms": round(back_to_back, 5),
            "note": "the same launches back to back on the same operands, no flush (operands L2-resident)"}
    if w.name in GRAPH_WORKLOADS and not (ta or tb):
        result["graph"] = graph_rate(pkg, p, A, B, C, algo, flops)
    if bound == "tensor":
        rate = tf32_mma_rate(pkg)
        if rate:
            # second denominator: the tf32 rate measured on the kernel's own MMA form
            result["roofline"]["tf32_mma_rate_tflops"] = round(rate, 1)
            result["roofline"]["frac_of_mma_rate"] = round(achieved / (rate / 3.0), 4)
    return result, p


def conv_path(layer, algo: str) -> str:
    """Kernel sgemm_conv2d runs for a layer: the wide FFMA form for at most 32
    filters of at most 48 taps under AUTO (64 when FFMA is asked for)."""
    m, _, k = layer.gemm_mnk
    if algo == "ffma" or (algo == "auto" and m <= 32 and k <= 48):
        return "ffma_wide"
    return "tf32x3"


def run_conv_ours(args, rank: int, world: int, local_rank: int):
    """One step = one sgemm_conv2d call over the whole layer (implicit GEMM)."""
    import torch

    import dense_fp32_matrix_05_gb300 as pkg
    from dense_fp32_matrix_05_gb300.workloads import CONV_LAYERS, make_conv_inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    from dense_fp32_matrix_05_gb300 import _build_ext
    _build_ext.build()
    pkg.library()
    layer = CONV_LAYERS[args.workload]
    algo = {"auto": 0, "ffma": 1, "tf32x3": 2}[args.algo]
    Xh, Wh = make_conv_inputs(layer)
    X = torch.from_numpy(Xh).to(dev)
    Wt = torch.from_numpy(Wh).to(dev)
    oh, ow = layer.out_hw
    Y = torch.zeros((layer.nb, layer.F, oh, ow), device=dev)
    stream = torch.cuda.current_stream(dev)
    M, N, K = layer.gemm_mnk
    flops = layer.flops
    st_pad = (layer.stride, layer.stride), (layer.pad, layer.pad)
    path_name = conv_path(layer, args.algo)
    # kernels per call: the conv kernel, plus the zero-bordered input copy
    # (padded layers whose channels are not a multiple of 16) or the OHWI
    # filter reorder (channels a multiple of 16, tensor path)
    launches = 1 + int(layer.pad > 0 and layer.C % 16 != 0) + int(path_name == "tf32x3" and layer.C % 16 == 0)

    def step():
        rc = pkg.sgemm_conv2d(X, Wt, Y, stride=st_pad[0], pad=st_pad[1], stream=stream, algo=algo)
        if rc != 0:
            raise pkg.SgemmError("sgemm_conv2d", rc)

    for _ in range(args.warmup):
        step()
    st = pkg.sgemm_check_status(stream)
    if st != 0:
        raise pkg.SgemmError("warmup", st)
    flush = layer.compulsory_bytes < 2 * 129e6
    fbuf = torch.empty(L2_FLUSH_BYTES // 4, device=dev) if flush else None
    dist = world > 1
    if dist:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk:
        for i in range(args.steps):
            if flush:
                fbuf.zero_()
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    if dist:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(float(np.sum(step_ms)), dev if dist else None)
    launch_ms = float(np.mean(step_ms))
    st = pkg.sgemm_check_status(stream)
    if st != 0:
        raise pkg.SgemmError("timed region", st)
    clocks = clk.summary()

    # e2e: pinned host input and filter in, the layer, the output back, every step
    e2e_steps = max(1, min(args.steps, args.e2e_steps))
    hX = torch.from_numpy(Xh).pin_memory()
    hW = torch.from_numpy(Wh).pin_memory()
    hY = torch.empty(tuple(Y.shape), dtype=torch.float32).pin_memory()

    def host_step():
        X.copy_(hX, non_blocking=True)
        Wt.copy_(hW, non_blocking=True)
        step()
        hY.copy_(Y, non_blocking=True)
        torch.cuda.synchronize()

    for _ in range(min(3, args.warmup)):
        host_step()
    if dist:
        torch.distributed.barrier()
    step_s = []
    h0 = time.perf_counter()
    for _ in range(e2e_steps):
        host_step()
        step_s.append(time.perf_counter())
    e2e_s = step_s[-1] - h0
    step_s = np.diff([h0] + step_s)
    if dist:
        t = torch.tensor([e2e_s], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_s = float(t.item())

    props = torch.cuda.get_device_properties(dev)
    peaks, peak_src = load_peaks()
    bound, peak, basis = roofline_peak(1 if path_name == "ffma_wide" else 2, peaks, peak_src,
                                       props.multi_processor_count)
    t_compute = flops / (peak * 1e12)
    t_memory = layer.compulsory_bytes / (peaks["hbm_gbs"] * 1e9)
    if t_memory > t_compute:
        bound, peak, unit_r = "hbm", peaks["hbm_gbs"], "GB/s"
        achieved = layer.compulsory_bytes / (launch_ms * 1e-3) / 1e9
        basis = f"{peak_src} HBM copy bandwidth {peaks['hbm_gbs']} GB/s (compulsory bytes / call time)"
    else:
        unit_r = "TFLOP/s"
        achieved = flops / (launch_ms * 1e-3) / 1e12
    value = job_throughput(world, flops, args.steps, total_ms)
    kernel_name = "ffma_wide_kernel<conv>" if path_name == "ffma_wide" else "tf32x3_gemm_kernel<conv>"
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {
            "workload": f"{layer.name}: {layer.note()}",
            "algo": f"{args.algo} -> {path_name} (implicit GEMM, sgemm_conv2d)",
            "l2": (f"flushed between steps ({L2_FLUSH_BYTES >> 20} MB written, untimed)" if flush else
                   f"no flush: compulsory bytes {layer.compulsory_bytes / 1e6:.0f} MB vs 129 MB L2"),
            "parallelism": f"replicas x{world}",
        },
        "roofline": {"bound": bound, "achieved": round(achieved, 3), "peak": round(peak, 3), "unit": unit_r,
                     "frac": round(achieved / peak, 4), "traffic": recorded_traffic(args.workload, path_name),
                     "peak_basis": basis, "kernel": kernel_name, "launch_ms": round(launch_ms, 5),
                     "launch_note": "whole sgemm_conv2d call: conv kernel plus any input/filter staging kernel",
                     "compulsory_bytes": layer.compulsory_bytes,
                     "hbm_frac_of_measured": round(layer.compulsory_bytes / (launch_ms * 1e-3) /
                                                   (peaks["hbm_gbs"] * 1e9), 4)},
        "e2e": {"value": round(world * flops * e2e_steps / e2e_s / 1e12, 3), "unit": UNIT,
                "h2d_bytes_per_step": int(Xh.nbytes + Wh.nbytes), "d2h_bytes_per_step": int(4 * Y.numel()),
                "steps": e2e_steps, "api": "sgemm_conv2d with pinned host copies in and out",
                "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 4),
                "ms_per_step_median": round(float(np.median(step_s)) * 1e3, 4),
                "ms_per_step_max": round(float(np.max(step_s)) * 1e3, 4)},
        "gpu_launches": args.steps * launches,
        "clocks": clocks,
    }
    return result, layer


def conv_oracle_sample(layer, target_s: float, threads: int = 0):
    """Time the conv oracle on the first image and the first f filters,
    growing f until the call takes target_s; returns (TFLOP/s, f, seconds)."""
    import oracle

    from dense_fp32_matrix_05_gb300.workloads import make_conv_inputs
    oracle.build()
    X, Wt = make_conv_inputs(layer)
    x0 = np.ascontiguousarray(X[:1])
    oh, ow = layer.out_hw
    f = 1
    while True:
        t = time.perf_counter()
        oracle.conv2d_ref(1.0, x0, np.ascontiguousarray(Wt[:f]), stride=(layer.stride,) * 2,
                          pad=(layer.pad,) * 2, threads=threads)
        dt = time.perf_counter() - t
        if dt >= target_s or f >= layer.F:
            return 2.0 * f * oh * ow * layer.C * layer.KH * layer.KW / dt / 1e12, f, dt
        f = min(layer.F, max(f + 1, int(f * min(8.0, 1.3 * target_s / max(dt, 1e-3)))))


def conv_cpu_baseline(layer, target_s: float):
    import oracle
    v, f, dt = conv_oracle_sample(layer, target_s)
    return {"value": v, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"image 0 of {layer.nb}, filters 0..{f - 1} of {layer.F}, all output pixels, "
                      f"float64 direct convolution (oracle as committed), {dt:.1f} s"}


def run_conv_reference(args, world: int):
    """The reference arm for a convolution layer: the float64 direct
    convolution oracle on a bounded sample (first image, first f filters)."""
    import oracle

    from dense_fp32_matrix_05_gb300.workloads import CONV_LAYERS, make_conv_inputs
    layer = CONV_LAYERS[args.workload]
    per_step = max(0.02, args.reference_budget_s / max(1, args.warmup + args.steps))
    _, f, _ = conv_oracle_sample(layer, per_step)
    X, Wt = make_conv_inputs(layer)
    x0, w0 = np.ascontiguousarray(X[:1]), np.ascontiguousarray(Wt[:f])
    oh, ow = layer.out_hw

    def step():
        oracle.conv2d_ref(1.0, x0, w0, stride=(layer.stride,) * 2, pad=(layer.pad,) * 2)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    value = 2.0 * f * oh * ow * layer.C * layer.KH * layer.KW * args.steps / dt / 1e12
    sample = f"image 0 of {layer.nb}, filters 0..{f - 1} of {layer.F} per step, float64 direct convolution"
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{layer.name}: {layer.note()}",
                   "algo": "float64 CPU oracle (the pages publish no GPU code to run here)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def oracle_sample_rate(p, target_s: float, threads: int = 0):
    """Time the oracle on a bounded row sample; returns (TFLOP/s, rows, seconds)."""
    import oracle
    oracle.build()
    rows = 1
    while True:
        sel = np.linspace(0, p.M - 1, rows).astype(np.int64).tolist()
        t = time.perf_counter()
        oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta,
                         p.C if p.beta != 0 else None, p.ldc, rows=sel, threads=threads)
        dt = time.perf_counter() - t
        if dt >= target_s or rows >= p.M:
            return 2.0 * rows * p.N * p.K / dt / 1e12, rows, dt
        rows = min(p.M, max(rows + 1, int(rows * min(8.0, 1.3 * target_s / max(dt, 1e-3)))))


def cpu_baseline(p, target_s: float):
    import oracle
    v, rows, dt = oracle_sample_rate(p, target_s)
    return {"value": v, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{rows} of {p.M} output rows x all {p.N} columns, K={p.K}, float64 "
                      f"(oracle as committed), {dt:.1f} s"}


def run_reference(args, world: int):
    """The reference arm: the float64 oracle on the host cores."""
    import oracle

    from dense_fp32_matrix_05_gb300.workloads import WORKLOADS, make_problem
    w = WORKLOADS[args.workload]
    p = make_problem(w, pad_value=0.0)
    oracle.build()
    # size one step so that warmup + steps fit the time budget
    per_step = max(0.02, args.reference_budget_s / max(1, args.warmup + args.steps))
    _, rows, _ = oracle_sample_rate(p, per_step)
    sel = np.linspace(0, p.M - 1, rows).astype(np.int64).tolist()

    def step():
        oracle.sgemm_ref(p.M, p.N, p.K, p.alpha, p.A, p.lda, p.B, p.ldb, p.beta,
                         p.C if p.beta != 0 else None, p.ldc, rows=sel)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    flops_step = 2.0 * rows * p.N * p.K
    value = flops_step * args.steps / dt / 1e12
    sample = f"{rows} of {p.M} output rows x all {p.N} columns per step, K={p.K}, float64"
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: M={p.M} N={p.N} K={p.K} fp32 row-major, {w.note}",
                   "algo": "float64 CPU oracle (the pages publish no GPU code to run here)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="square5120")
    ap.add_argument("--algo", choices=["auto", "ffma", "tf32x3"], default="auto")
    ap.add_argument("--trans", choices=["NN", "NT", "TN", "TT"], default="NN",
                    help="op(A) op(B) storage through sgemm_t (timed with its transposes)")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-baseline-s", type=float, default=10.0)
    ap.add_argument("--reference-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cublas", dest="cublas", action="store_false")
    ap.add_argument("--shapes-out", default=None,
                    help="also measure every benchmark workload and write JSON lines here")
    ap.add_argument("--per-shape", dest="per_shape", action="store_true", default=None,
                    help="add a per_shape summary of every workload to the line (default: on for the "
                         "default square5120 run on one GPU)")
    ap.add_argument("--no-per-shape", dest="per_shape", action="store_false")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if "WORLD_SIZE" not in os.environ:
        world = 1

    from dense_fp32_matrix_05_gb300.workloads import CONV_LAYERS
    conv = args.workload in CONV_LAYERS
    if conv and args.trans != "NN":
        ap.error("--trans applies to GEMM workloads")
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_conv_reference(args, world) if conv else run_reference(args, world)), flush=True)
        return 0

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result, p = (run_conv_ours if conv else run_ours)(args, rank, world, local_rank)
    if rank == 0 and world == 1:
        result["cpu_baseline"] = (conv_cpu_baseline if conv else cpu_baseline)(p, args.cpu_baseline_s)
    elif rank == 0:
        result["cpu_baseline"] = None
    per_shape = args.per_shape
    if per_shape is None:
        per_shape = args.workload == "square5120" and args.trans == "NN" and args.algo == "auto"
    if rank == 0 and world == 1 and (per_shape or args.shapes_out):
        lines = measure_all(args, local_rank)
        if per_shape:
            result["per_shape"] = [shape_summary(r) for r in lines]
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


def shape_summary(r: dict) -> dict:
    """The figures of one per-shape line that the per_shape list carries."""
    if "error" in r:
        return r
    rf = r["roofline"]
    s = {"workload": r["config"]["workload"].split(":")[0], "algo": r["config"]["algo"],
         "value": r["value"], "unit": r["unit"], "bound": rf["bound"], "frac": rf["frac"],
         "launch_ms": rf["launch_ms"], "steps": r["steps"],
         "l2": "flushed" if r["config"]["l2"].startswith("flushed") else "larger than L2",
         "sm_mhz": (r.get("clocks") or {}).get("sm_mhz"), "reasons": (r.get("clocks") or {}).get("reasons")}
    if "frac_of_mma_rate" in rf:
        s["frac_of_mma_rate"] = rf["frac_of_mma_rate"]
    if "context_cublas_sgemm_tflops" in r:
        s["context_cublas_sgemm_tflops"] = r["context_cublas_sgemm_tflops"]
    if "context_back_to_back_l2_resident" in r:
        s["context_back_to_back_l2_resident"] = r["context_back_to_back_l2_resident"]["value"]
    e = r.get("e2e") or {}
    if "value" in e:
        s["e2e"] = e["value"]
        for k in ("frac_of_copy_bound", "frac_of_pipeline_bound"):
            if e.get(k) is not None:
                s["e2e_" + k] = e[k]
    return s


def measure_all(args, local_rank) -> list:
    """Every benchmark workload on both paths and every convolution layer, one
    result each; written as JSON lines to --shapes-out when given."""
    from dense_fp32_matrix_05_gb300.workloads import WORKLOADS
    out = open(args.shapes_out, "w") if args.shapes_out else None
    lines = []
    names = ["square256", "square1024", "ragged1023x1021x1025", "square5120"] + \
        [n for n in WORKLOADS if n.startswith("skinny")] + [n for n in WORKLOADS if n.startswith("sweep")]
    for name in names:
        for algo in ("auto", "ffma"):
            a = argparse.Namespace(**vars(args))
            a.workload, a.algo = name, algo
            w = WORKLOADS[name]
            a.steps = max(5, min(200, int(2e12 / max(w.flops, 1.0))))
            a.warmup = 3
            a.e2e_steps = 10
            a.cublas = True
            try:
                r, _ = run_ours(a, 0, 1, local_rank)
            except Exception as e:  # keep measuring the rest
                r = {"workload": name, "algo": algo, "error": str(e)}
            lines.append(r)
            if out:
                out.write(json.dumps(r) + "\n")
                out.flush()
            log(f"{name} {algo}: {r.get('value')} TFLOP/s, roofline {r.get('roofline', {}).get('frac')}")
    from dense_fp32_matrix_05_gb300.workloads import CONV_LAYERS
    for name, layer in CONV_LAYERS.items():
        a = argparse.Namespace(**vars(args))
        a.workload, a.algo = name, "auto"
        a.steps = max(5, min(200, int(2e12 / layer.flops)))
        a.warmup, a.e2e_steps = 3, 10
        try:
            r, _ = run_conv_ours(a, 0, 1, local_rank)
        except Exception as e:  # keep measuring the rest
            r = {"workload": name, "algo": "auto", "error": str(e)}
        lines.append(r)
        if out:
            out.write(json.dumps(r) + "\n")
            out.flush()
        log(f"{name}: {r.get('value')} TFLOP/s, roofline {r.get('roofline', {}).get('frac')}")
    if out:
        out.close()
    return lines


if __name__ == "__main__":
    sys.exit(main())
