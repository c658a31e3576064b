#!/usr/bin/env python3
"""Benchmark: causal GQA attention forward + delta + backward on GB300.

One step = attn_fwd -> attn_bwd_delta -> attn_bwd (dK/dV kernel, then dQ
kernel) over one batch of the workload, inputs resident in HBM.  The metric
is credited TFLOP/s: 3.5 x the forward FLOPs (4*B*Hq*Lq*Lk*D, halved for
causal) over the summed device time of the step's kernels.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--block-mask none|window:W|random:P] [--kv-capacity N] [--decode]
                    [--lce [--lce-workload NAME]]

Prints one JSON line (rank 0).  Under torchrun each rank runs its own replica
of the workload on its own GPU (weak scaling); the value is all ranks' work
over the slowest rank's time.  `--impl reference` times the fp64 CPU oracle on
the host cores instead, on a bounded sample of the same workload.

With `--block-mask` the step runs the block-sparse entry points
(attn_fwd_masked, attn_bwd_delta, attn_bwd_masked) and the metric credits
3.5 x 4*D FLOPs per (query, key) pair the mask and the causal rule leave
visible.  With `--kv-capacity N` k and v are the first Lk rows of each head
of an N-row cache whose other rows hold large stale values, and the step runs
attn_fwd_ex / attn_bwd_ex.  With `--decode` (short query lengths) the step
runs attn_fwd_decode, attn_bwd_delta and attn_bwd_decode, and the roofline
is HBM bytes (the key/value range read and the gradients written).  With
`--lce` the step is the fused linear cross-entropy (lce_fwd + lce_bwd) of a
Qwen3-8B output layer, credited 2 N V Dm FLOPs forward and 3 x that backward.
"""

from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from bwd_flashattention_fwd_gb300 import flops as F  # noqa: E402
from bwd_flashattention_fwd_gb300 import replicas  # noqa: E402
from bwd_flashattention_fwd_gb300.inputs import (  # noqa: E402
    LCE_WORKLOADS,
    WORKLOADS,
    LceWorkload,
    Workload,
    block_mask,
    make_inputs,
    make_lce_inputs,
)

METRIC = "fwd+bwd attention TFLOP/s, causal GQA L=8192 D=128 bf16; % of BF16 TC peak"
METRIC_MASKED = "block-sparse fwd+bwd attention TFLOP/s (3.5 x 4*D FLOPs per visible pair)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "qwen3_8b_gqa_l8192_d128"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_per_launch.txt")
TENSOR_PIPE_FILE = os.path.join(ROOT, "profiles", "tensor_pipe_per_launch.txt")
# dense 16-bit tensor-core work one SM completes per clock (kind::f16 MMAs with
# fp32 accumulation: an M=128, N=256, K=16 MMA is 1 Mi FLOP in 128 clocks)
TENSOR_FLOP_PER_CLK_SM = 8192
LONG_RUN_STEPS = 100


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


KERNEL_FILES = {
    "fwd": "fwd2_kernel.cuh",
    "delta": "delta_kernel.cuh",
    "bwd_dkv": "bwd_dkv2_kernel.cuh",
    "bwd_dq": "bwd_dq3_kernel.cuh",
}
# head dimension 256 runs other kernels for the same phases
KERNEL_FILES_D256 = dict(KERNEL_FILES, fwd="fwd_kernel.cuh", bwd_dkv="bwd_dkv_kernel.cuh", bwd_dq="bwd_dq_kernel.cuh")


def _code_only(text: bytes) -> bytes:
    """Source text without // and /* */ comments, trailing spaces and blank
    lines, so that an edit touching only comments keeps a kernel's hash."""
    t = re.sub(rb"/\*.*?\*/", b"", text, flags=re.S)
    t = re.sub(rb"//[^\n]*", b"", t)
    return b"\n".join(line.rstrip() for line in t.split(b"\n") if line.strip())


def kernel_source_hash(kernel: str | None = None, D: int = 128) -> str:
    """Hash of the code (comments excluded) that defines a phase's kernel at
    head dimension D (its own file, the shared device headers and the launch
    code), or of all sources."""
    csrc = os.path.join(ROOT, "bwd_flashattention_fwd_gb300", "csrc")
    if kernel is None:
        files = sorted(glob.glob(os.path.join(csrc, "*")))
    else:
        own = (KERNEL_FILES_D256 if D == 256 else KERNEL_FILES)[kernel]
        files = [os.path.join(csrc, n) for n in (own, "kernel_common.cuh", "ptx.cuh", "inst.cu")]
    h = hashlib.sha256()
    for p in files:
        with open(p, "rb") as f:
            h.update(os.path.basename(p).encode() + _code_only(f.read()))
    return h.hexdigest()[:16]


def recorded_figure(path: str, kernel: str, workload: str, D: int = 128):
    """A per-launch figure from a committed ncu summary, if it was taken on
    the current kernel sources (else None).  Line format:
    `<kernel> <workload> <value> <source_hash>`."""
    if kernel not in KERNEL_FILES or not os.path.exists(path):
        return None
    cur = kernel_source_hash(kernel, D)
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 4 and not line.startswith("#") and parts[0] == kernel and parts[1] == workload:
                return float(parts[2]) if parts[3] == cur else None
    return None


def recorded_traffic(kernel: str, workload: str, D: int = 128):
    """DRAM bytes (read + write) per launch, from the committed ncu summary."""
    return recorded_figure(TRAFFIC_FILE, kernel, workload, D)


def recorded_tensor_pipe(kernel: str, workload: str, D: int = 128):
    """ncu's sm__pipe_tensor_cycles_active (% of peak, active SMs) per launch."""
    return recorded_figure(TENSOR_PIPE_FILE, kernel, workload, D)


class ClockSampler:
    """nvidia-smi sampled every 50 ms, each sample carrying the tool's own
    timestamp (a pipe delivers its lines in bursts, so arrival times say
    nothing).  Start it before the warm-up (the tool takes a while to begin),
    bracket each timed region with begin() / end() (wall-clock times of this
    host), and window() keeps the samples taken inside it."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_S = 0.05

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.thread = None
        self.samples = []  # (arrival time, fields)
        self.t_begin = self.t_end = None

    def start(self):
        import atexit
        import threading

        atexit.register(self.stop)  # no sampler outlives the bench, whatever ends it
        import shutil

        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms",
               str(int(self.PERIOD_S * 1000)), "-i", str(self.gpu_index)]
        if shutil.which("stdbuf"):
            cmd = ["stdbuf", "-oL"] + cmd  # one line per sample through the pipe
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def read():
            from datetime import datetime

            for line in self.proc.stdout:
                p = [x.strip() for x in line.split(",")]
                try:
                    t = datetime.strptime(p[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                except (ValueError, IndexError):
                    continue
                self.samples.append((t, p))

        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()

    def wait_first(self, timeout_s: float = 3.0):
        """Give the tool time to start sampling before a timed region."""
        t0 = time.time()
        while self.proc is not None and not self.samples and time.time() - t0 < timeout_s:
            time.sleep(0.01)

    def begin(self):
        self.t_begin = time.time()

    def end(self):
        self.t_end = time.time()

    def stop(self):
        if self.proc is not None and self.proc.poll() is None:
            import signal

            self.proc.send_signal(signal.SIGINT)  # ends the sampling loop the way Ctrl-C does
            try:
                self.proc.wait(timeout=3)
            except subprocess.TimeoutExpired:
                self.proc.terminate()
                try:
                    self.proc.wait(timeout=3)
                except subprocess.TimeoutExpired:
                    self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=5)

    def window(self, t_begin=None, t_end=None) -> dict:
        """Statistics of the samples that arrived between t_begin and t_end
        (default: the last begin() / end()), plus one sampling period after
        the end for a region shorter than the period."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        t0 = self.t_begin if t_begin is None else t_begin
        t1 = (self.t_end if t_end is None else t_end) + self.PERIOD_S
        sm, smax, power, reasons = [], [], [], set()
        for t, p in list(self.samples):
            if not (t0 <= t <= t1) or len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
                power.append(float(p[3]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, p[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm),
                "window_s": round(t1 - t0, 4)}


def gemm_canary(dev, n: int = 8192, reps: int = 3) -> float:
    """TFLOP/s of a bf16 n x n x n library GEMM (torch.matmul), timed with
    CUDA events: run before and after the timed steps, it shows whether the
    clocks moved between them.  A measurement aid, not part of the step."""
    a = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
    b = torch.randn((n, n), device=dev, dtype=torch.bfloat16)
    torch.matmul(a, b)  # warm
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        torch.matmul(a, b)
    e1.record()
    torch.cuda.synchronize(dev)
    return 2.0 * n ** 3 * reps / (e0.elapsed_time(e1) * 1e-3) / 1e12


def physical_gpu_index(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if local_rank < len(ids) and ids[local_rank].isdigit():
        return int(ids[local_rank])
    return local_rank


def workload_config(w: Workload, extra: dict) -> dict:
    cfg = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Lq": w.Lq, "Lk": w.Lk, "D": w.D,
           "causal": w.causal, "dtype": w.dtype, "input_std": w.std, "seed": w.seed}
    cfg.update(extra)
    return cfg


# ---------------------------------------------------------------------------
# CPU oracle timing (the reported baseline and the reference arm)
# ---------------------------------------------------------------------------


def oracle_sample_problem(w: Workload, rows: int):
    """The last `rows` query rows of head (b=0, hq=0) with the keys they can
    see: with bottom-right causal alignment that row block is itself a causal
    problem (Lq' = rows, Lk' = visible keys), so the oracle runs on it as is."""
    q, k, v, do = make_inputs(w, "cpu")
    from bwd_flashattention_fwd_gb300.inputs import to_f64

    r0 = w.Lq - rows
    qs = to_f64(q[:1, :1, r0:])
    dos = to_f64(do[:1, :1, r0:])
    ks = to_f64(k[:1, :1])  # the last query row sees every key
    vs = to_f64(v[:1, :1])
    # credit 3.5 x 4*D FLOPs per visible (query, key) pair of the sample; over a
    # whole causal problem that is the half-rectangle count of the metric
    credited = 3.5 * 4.0 * w.D * F.visible_pairs(rows, w.Lk, w.causal)
    return (qs, ks, vs, dos), credited


def run_oracle_sample(arrays, w: Workload):
    import oracle.attention as A

    qs, ks, vs, dos = arrays
    o, lse2, _ = A.forward(qs, ks, vs, w.scale, w.causal)
    A.delta(o, dos)
    A.backward(qs, ks, vs, o, dos, w.scale, w.causal)


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w: Workload, rows: int) -> dict:
    arrays, credited = oracle_sample_problem(w, rows)
    run_oracle_sample(arrays, w)  # warm
    t0 = time.perf_counter()
    n = 0
    while True:
        run_oracle_sample(arrays, w)
        n += 1
        if time.perf_counter() - t0 > 5.0:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": credited / dt / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 oracle fwd+delta+bwd on the last {rows} query rows of head (b=0,hq=0) and the "
                      f"keys they see ({credited:.3g} credited FLOP per run, {n} runs, {dt:.3f} s each)"}


ORACLE_TABLE = ("llama_gqa_l2048_d128", "qwen3_8b_gqa_l8192_d128", "gqa_l8192_d256", "ragged_mha_q4064_k4112_d96")


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def blas_threads():
    try:
        from threadpoolctl import threadpool_info

        return [{"api": d.get("internal_api"), "threads": d.get("num_threads")} for d in threadpool_info()]
    except ImportError:
        return {k: os.environ[k] for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS") if k in os.environ} or \
            "library default (one thread per core)"


def run_oracle_table(args):
    """The fp64 oracle on each full workload, timed on the host cores.  Each
    (batch, KV head) group is an independent problem the oracle loops over,
    so one group (its G query heads with their K/V head) is timed and the
    whole workload's time is that x B x Hkv."""
    import oracle.attention as A
    from bwd_flashattention_fwd_gb300.inputs import to_f64

    rows = []
    for name in ORACLE_TABLE:
        w = WORKLOADS[name]
        G = w.Hq // w.Hkv
        q, k, v, do = make_inputs(w, "cpu")
        qs, dos = to_f64(q[:1, :G]), to_f64(do[:1, :G])
        ks, vs = to_f64(k[:1, :1]), to_f64(v[:1, :1])
        t0 = time.perf_counter()
        o, _, _ = A.forward(qs, ks, vs, w.scale, w.causal)
        A.delta(o, dos)
        A.backward(qs, ks, vs, o, dos, w.scale, w.causal)
        dt = time.perf_counter() - t0
        groups = w.B * w.Hkv
        full_s = dt * groups
        credited = F.credited_fwd_bwd(w.B, w.Hq, w.Lq, w.Lk, w.D, w.causal)
        rows.append({"workload": name, "group_s": dt, "groups": groups, "full_s": full_s,
                     "tflops_credited": credited / full_s / 1e12})
        print(json.dumps(rows[-1]), flush=True)
    print(json.dumps({"oracle_table": rows, "cores": cpu_cores(), "cpu_model": cpu_model(),
                      "blas_threads": blas_threads(),
                      "method": "fp64 oracle fwd + delta + bwd on one (batch, KV head) group, x B x Hkv"}),
          flush=True)
    return 0


def run_reference(args):
    rank, local_rank, ws = replicas.world()
    if rank != 0:
        return 0
    w = WORKLOADS[args.workload]
    rows = args.ref_rows
    arrays, credited = oracle_sample_problem(w, rows)
    for _ in range(args.warmup):
        run_oracle_sample(arrays, w)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_sample(arrays, w)
    dt = time.perf_counter() - t0
    value = credited * args.steps / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, {"sample_rows": rows, "parallelism": "host cores"}),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"each step: fp64 oracle fwd+delta+bwd on the last {rows} query rows of "
                                   f"head (b=0,hq=0) and the keys they see"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------


def run_ours(args):
    from bwd_flashattention_fwd_gb300 import build, gbattn

    rank, local_rank, ws = replicas.world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    replicas.init("nccl")
    build.build()
    gbattn.load_library()

    w = WORKLOADS[args.workload]
    q, k, v, do = make_inputs(w, dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Lq), dtype=torch.float32, device=dev)
    dlt = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    sc, causal = w.scale, w.causal
    bm_np = block_mask(args.block_mask, w.Lq, w.Lk, seed=w.seed)
    bm = None if bm_np is None else torch.from_numpy(bm_np).to(dev)
    kv_cap = args.kv_capacity
    # the end-to-end run's pinned host buffers, allocated and copied through
    # once now: in a fresh process, fresh pinned memory showed one-off copy
    # stalls of ~15 ms for a while after its allocation
    e2e_host = None
    if not args.no_e2e and not kv_cap and not args.decode:
        e2e_host = e2e_host_buffers(w, dev)
    if kv_cap:
        if kv_cap < w.Lk:
            raise SystemExit(f"--kv-capacity {kv_cap} is below Lk = {w.Lk}")
        caches = []
        for t in (k, v):
            c = torch.full((w.B, w.Hkv, kv_cap, w.D), 3.0e4, dtype=t.dtype, device=dev)
            c[:, :, :w.Lk].copy_(t)
            caches.append(c)
        k, v = caches[0][:, :, :w.Lk], caches[1][:, :, :w.Lk]

    if args.decode:
        if bm is not None or kv_cap:
            raise SystemExit("--decode takes neither --block-mask nor --kv-capacity")
        split_names, split_calls = None, None
        ws_dec = gbattn.decode_workspace(q, k)
        phase_names = ("fwd", "delta", "bwd")
        calls = (
            lambda: gbattn.attn_fwd_decode(q, k, v, o, lse, ws_dec, sc, causal, stream),
            lambda: gbattn.attn_bwd_delta(o, do, dlt, stream),
            lambda: gbattn.attn_bwd_decode(q, k, v, o, do, lse, dlt, dq, dk, dv, ws_dec, sc, causal, stream),
        )
    elif bm is None and not kv_cap:
        # the step: attn_fwd, attn_bwd_delta, attn_bwd (its dQ kernel fills
        # the SMs the dK/dV kernel's last wave frees); the kernels are timed
        # one by one in a second pass, through attn_bwd_dkv and attn_bwd_dq
        phase_names = ("fwd", "delta", "bwd")
        calls = (
            lambda: gbattn.attn_fwd(q, k, v, o, lse, sc, causal, stream),
            lambda: gbattn.attn_bwd_delta(o, do, dlt, stream),
            lambda: gbattn.attn_bwd(q, k, v, o, do, lse, dlt, dq, dk, dv, sc, causal, stream),
        )
        split_names = ("fwd", "delta", "bwd_dkv", "bwd_dq")
        split_calls = (
            calls[0], calls[1],
            lambda: gbattn.attn_bwd_dkv(q, k, v, do, lse, dlt, dk, dv, sc, causal, stream),
            lambda: gbattn.attn_bwd_dq(q, k, v, do, lse, dlt, dq, sc, causal, stream),
        )
    else:
        # attn_bwd_ex launches the dK/dV kernel, then the dQ kernel
        split_names, split_calls = None, None
        phase_names = ("fwd", "delta", "bwd")
        calls = (
            lambda: gbattn.attn_fwd_ex(q, k, v, o, lse, sc, causal, block_mask=bm, stream=stream),
            lambda: gbattn.attn_bwd_delta(o, do, dlt, stream),
            lambda: gbattn.attn_bwd_ex(q, k, v, o, do, lse, dlt, dq, dk, dv, sc, causal, block_mask=bm,
                                       stream=stream),
        )
    n_ev = len(calls) + 1

    def step(ev=None):
        for j, c in enumerate(calls):
            if ev is not None:
                ev[j].record(stream)
            c()
        if ev is not None:
            ev[-1].record(stream)

    clocks = ClockSampler(physical_gpu_index(local_rank))
    clocks.start()
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize(dev)
    if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
        raise RuntimeError("device-side wait timed out during warm-up")
    clocks.wait_first()
    canary_before = None if args.no_canary else gemm_canary(dev)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    replicas.barrier(dev)
    torch.cuda.synchronize(dev)
    clocks.begin()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)  # L2 flush between steps, outside the step's events
        step(events[i])
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    clocks.end()
    replicas.barrier(dev)
    if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
        raise RuntimeError("device-side wait timed out during the timed steps")

    # the same steps over a longer region (power and clocks settle), reported
    # beside the K-step value, never in place of it
    long_run = None
    if args.steps < LONG_RUN_STEPS and not args.no_long_run:
        lev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(LONG_RUN_STEPS)]
        torch.cuda.synchronize(dev)
        t_l0 = time.time()
        for i in range(LONG_RUN_STEPS):
            flush.fill_(i & 0xFF)
            lev[i][0].record(stream)
            step()
            lev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t_l1 = time.time()
        if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
            raise RuntimeError("device-side wait timed out during the long run")
        long_run = {"steps": LONG_RUN_STEPS, "ms_per_step": statistics.mean(a.elapsed_time(b) for a, b in lev),
                    "_window": (t_l0, t_l1)}

    per_phase = {n: [] for n in phase_names}
    step_ms = []
    for ev in events:
        for j, n in enumerate(phase_names):
            per_phase[n].append(ev[j].elapsed_time(ev[j + 1]))
        step_ms.append(ev[0].elapsed_time(ev[-1]))
    # the kernels one by one (the same number of steps), for the per-kernel rooflines
    split = None
    if split_calls is not None:
        sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(split_calls) + 1)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            for j, c in enumerate(split_calls):
                sev[i][j].record(stream)
                c()
            sev[i][-1].record(stream)
        torch.cuda.synchronize(dev)
        if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
            raise RuntimeError("device-side wait timed out in the per-kernel pass")
        split = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in sev) for j, n in enumerate(split_names)}
    local_s = sum(step_ms) / 1e3
    if bm is None:
        pairs = F.visible_pairs(w.Lq, w.Lk, w.causal)
        credited = F.credited_fwd_bwd(w.B, w.Hq, w.Lq, w.Lk, w.D, w.causal)
    else:
        pairs = F.visible_pairs_masked(w.Lq, w.Lk, w.causal, bm_np)
        credited = 3.5 * 4.0 * w.D * w.B * w.Hq * pairs
    value_flops, _, max_s = replicas.aggregate_throughput(credited * args.steps, local_s, dev)
    value = value_flops / 1e12
    peaks = load_peaks()
    if long_run is not None:
        long_run["value"] = credited / (long_run["ms_per_step"] * 1e-3) / 1e12
        long_run["unit"] = UNIT
        long_run["pct_of_bf16_peak"] = 100.0 * long_run["value"] / peaks["bf16_tflops"]
        long_run["pct_of_bf16_peak_sustained"] = 100.0 * long_run["value"] / peaks["bf16_tflops_sustained"]
    avg = {n: statistics.mean(v) for n, v in per_phase.items()}
    kavg = dict(avg, **split) if split else avg  # per-kernel times
    canary_after = None if args.no_canary else gemm_canary(dev)
    clocks.stop()  # the tool exits and flushes its last lines
    clk = clocks.window()
    if long_run is not None:
        long_run["clocks"] = clocks.window(*long_run.pop("_window"))
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # clock-independent ceiling of the tensor pipe at the clock the run held
    pipe_tflops = (TENSOR_FLOP_PER_CLK_SM * n_sms * clk["sm_mhz"] * 1e6 / 1e12) if clk.get("sm_mhz") else None

    # roofline per kernel (algorithmic work / average launch time)
    kernels = {}
    mm_phases = [n for n in (split_names or phase_names) if n != "delta"]
    for n in mm_phases:
        if args.decode:  # bound by the key/value range read
            by = F.decode_bytes(n, w.B, w.Hq, w.Hkv, w.Lq, w.Lk, w.D)
            ach = by / (kavg[n] * 1e-3) / 1e9
            kernels[n] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": ach / peaks["hbm_gbs"], "avg_ms": kavg[n], "algorithmic": by, "traffic": None}
            continue
        fl = F.kernel_flops_pairs(n, w.B, w.Hq, w.D, pairs)
        ach = fl / (kavg[n] * 1e-3) / 1e12
        plain = bm is None and not kv_cap
        kernels[n] = {"bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                      "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                      "frac_sustained": ach / peaks["bf16_tflops_sustained"],
                      "avg_ms": kavg[n], "algorithmic": fl,
                      "traffic": recorded_traffic(n, w.name, w.D) if plain else None,
                      "ncu_tensor_pipe_pct": recorded_tensor_pipe(n, w.name, w.D) if plain else None}
        if pipe_tflops:
            kernels[n]["frac_of_clock_ceiling"] = ach / pipe_tflops
    db = F.delta_bytes(w.B, w.Hq, w.Lq, w.D)
    ach = db / (kavg["delta"] * 1e-3) / 1e9
    kernels["delta"] = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": ach / peaks["hbm_gbs"], "avg_ms": kavg["delta"], "algorithmic": db,
                        "traffic": recorded_traffic("delta", w.name, w.D)}
    dominant = max(mm_phases, key=lambda n: kavg[n])
    roof = {k2: kernels[dominant][k2] for k2 in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = dominant
    if kernels[dominant]["bound"] == "tensor":
        roof["peak_kind"] = f"bf16 dense, burst ({peaks['source']}; the timed region is tens of milliseconds)"
        roof["peak_sustained"] = peaks["bf16_tflops_sustained"]
        roof["frac_sustained"] = kernels[dominant]["frac_sustained"]
        roof["ncu_tensor_pipe_pct"] = kernels[dominant]["ncu_tensor_pipe_pct"]
        if pipe_tflops:
            roof["clock_ceiling"] = {"tflops": pipe_tflops, "frac": kernels[dominant]["frac_of_clock_ceiling"],
                                     "basis": f"{TENSOR_FLOP_PER_CLK_SM} FLOP/clk/SM x {n_sms} SMs x median "
                                              f"sampled SM clock {clk['sm_mhz']} MHz"}
    else:
        roof["peak_kind"] = f"HBM copy bandwidth ({peaks['source']})"

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and not kv_cap and not args.decode:
        e2e = run_e2e(args, w, dev, stream, gbattn, credited, e2e_host, bm)

    n_dkv = 1  # one dK/dV launch (at D = 256 it holds both halves)
    extra = {}
    if bm is not None:
        extra = {"block_mask": args.block_mask, "mask_blocks_kept": int(bm_np.sum()),
                 "mask_blocks": int(bm_np.size)}
    if kv_cap:
        extra["kv_capacity"] = kv_cap
    if args.decode:
        extra["path"] = "decode (packed GQA rows, split key range)"
    extra["visible_pairs_per_head"] = pairs
    line = {
        "metric": METRIC if bm is None else METRIC_MASKED, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": max_s * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, {
            "l2": "flushed between steps (256 MiB write outside the step events); inputs 384 MiB",
            "parallelism": "replicas" if ws > 1 else "single GPU",
            "timing": "CUDA events on the launching stream, sum over steps",
            **extra,
        }),
        "pct_of_bf16_peak": 100.0 * value / ws / peaks["bf16_tflops"],
        # the same time with 3.5 x 4*D FLOPs credited per visible (query, key)
        # pair instead of the half-rectangle convention (differs for Lq != Lk)
        "tflops_visible_pairs": 3.5 * 4.0 * w.D * w.B * w.Hq * pairs * ws * args.steps / max_s / 1e12,
        "pct_of_bf16_peak_sustained": 100.0 * value / ws / peaks["bf16_tflops_sustained"],
        "peaks": peaks,
        "phase_ms": avg,
        "kernel_ms": split,  # each kernel timed on its own (None: the phases are the kernels)
        "roofline": roof,
        "kernels": kernels,
        "long_run": long_run,
        "e2e": e2e,
        # fwd, delta, dK/dV, dQ; the decode path adds
        # the combine and the dQ reduction
        "gpu_launches": args.steps * (1 + 1 + n_dkv + 1 + (2 if args.decode else 0)),
        "clocks": clk,
        # a bf16 8192^3 cuBLAS GEMM just before and just after the timed steps
        "gemm_canary_tflops": {"before": canary_before, "after": canary_after},
        "wall_s_timed_region": t_wall,
        "kernel_source_hash": kernel_source_hash(),
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_rows)
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    replicas.shutdown()
    return 0


def e2e_host_buffers(w, dev):
    """Pinned host inputs (q, k, v, dO) and one set of pinned host outputs (o,
    lse, dq, dk, dv) for run_e2e, each copied to and from the device once."""
    ins_h = tuple(t.pin_memory() for t in make_inputs(w, "cpu"))
    shapes = [(ins_h[0].shape, ins_h[0].dtype), ((w.B, w.Hq, w.Lq), torch.float32), (ins_h[0].shape, ins_h[0].dtype),
              (ins_h[1].shape, ins_h[1].dtype), (ins_h[2].shape, ins_h[2].dtype)]
    outs_h = [torch.empty(sh, dtype=dt).pin_memory() for sh, dt in shapes]
    for t in (*ins_h, *outs_h):
        d = t.to(dev, non_blocking=True)
        t.copy_(d, non_blocking=True)
    torch.cuda.synchronize(dev)
    return ins_h, outs_h


def run_e2e(args, w, dev, stream, gbattn, credited, host, bm=None):
    """Same metric through attn_fwd / attn_bwd_delta / attn_bwd with pinned
    host buffers: every step copies q, k, v, dO in and o, lse, dq, dk, dv out.
    Steps are pipelined over three sets of device buffers and three streams
    (copies in, compute, copies out), so step i's results travel to the host
    while step i+1 computes and step i+2's inputs arrive (a third set keeps
    one slow copy from stalling the compute stream); the timed region spans
    the first input copy to the last output copy."""
    ins_h, outs_h = host
    h2d = sum(t.numel() * t.element_size() for t in ins_h)

    def device_set():
        q, k, v, do = (torch.empty_like(t, device=dev) for t in ins_h)
        o, dq = torch.empty_like(q), torch.empty_like(q)
        dk, dv = torch.empty_like(k), torch.empty_like(v)
        lse = torch.empty((w.B, w.Hq, w.Lq), dtype=torch.float32, device=dev)
        return {"in": (q, k, v, do), "o": o, "lse": lse, "dlt": torch.empty_like(lse), "dq": dq, "dk": dk, "dv": dv}

    NSET = 3
    sets = [device_set() for _ in range(NSET)]
    # one host output set: the output copies run in order on one stream
    d2h = sum(t.numel() * t.element_size() for t in outs_h)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # at least 200 steps (~0.3 s): the pipeline's fill and drain (the first
    # input copy and the last output copy, ~1 ms each) would weigh ~6% in 20,
    # and host copies on this shared machine stall now and then for ~15 ms at
    # a time, which a 50-step window (~80 ms) cannot absorb
    n = max(200, min(args.steps, 400))
    # an untimed pass of the same length first: in a fresh process the first
    # few dozen pipelined steps showed one-off stalls of ~15 ms in the host
    # copies (later passes ran clean at the compute rate)
    warm = NSET + n
    total = warm + n
    ev_in = [torch.cuda.Event() for _ in range(total)]
    ev_comp = [torch.cuda.Event() for _ in range(total)]
    ev_out = [torch.cuda.Event() for _ in range(total)]

    def e2e_step(i):
        b = i % NSET
        s_ = sets[b]
        with torch.cuda.stream(s_in):
            if i >= NSET:
                s_in.wait_event(ev_comp[i - NSET])  # buffer set b's inputs are free again
            for dst, src in zip(s_["in"], ins_h):
                dst.copy_(src, non_blocking=True)
            ev_in[i].record(s_in)
        stream.wait_event(ev_in[i])
        if i >= NSET:
            stream.wait_event(ev_out[i - NSET])  # buffer set b's outputs reached the host
        q, k, v, do = s_["in"]
        if bm is None:
            gbattn.attn_fwd(q, k, v, s_["o"], s_["lse"], w.scale, w.causal, stream)
            gbattn.attn_bwd_delta(s_["o"], do, s_["dlt"], stream)
            gbattn.attn_bwd(q, k, v, s_["o"], do, s_["lse"], s_["dlt"], s_["dq"], s_["dk"], s_["dv"], w.scale,
                            w.causal, stream)
        else:
            gbattn.attn_fwd_masked(q, k, v, s_["o"], s_["lse"], bm, w.scale, w.causal, stream)
            gbattn.attn_bwd_delta(s_["o"], do, s_["dlt"], stream)
            gbattn.attn_bwd_masked(q, k, v, s_["o"], do, s_["lse"], s_["dlt"], bm, s_["dq"], s_["dk"], s_["dv"],
                                   w.scale, w.causal, stream)
        ev_comp[i].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[i])
            for dst, src in zip(outs_h, (s_["o"], s_["lse"], s_["dq"], s_["dk"], s_["dv"])):
                dst.copy_(src, non_blocking=True)
            ev_out[i].record(s_out)

    for i in range(warm):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    replicas.barrier(dev)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(warm, total):
        e2e_step(i)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    local_s = e0.elapsed_time(e1) / 1e3
    if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
        raise RuntimeError("device-side wait timed out during the end-to-end steps")
    value, _, _ = replicas.aggregate_throughput(credited * n, local_s, dev)
    return {"value": value / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "ms_per_step": local_s * 1e3 / n,
            "pipelining": "three device buffer sets; input copies, compute and output copies on separate streams"}


# ---------------------------------------------------------------------------
# Fused linear cross-entropy
# ---------------------------------------------------------------------------

METRIC_LCE = "fused linear cross-entropy fwd+bwd TFLOP/s, Qwen3-8B output layer (N=8192, hidden 4096, vocab 151936) bf16"


def lce_cpu_baseline(w: LceWorkload, rows: int = 4) -> dict:
    """The fp64 oracle's loss and dH for a few rows (all of V and Dm)."""
    import oracle.linear_ce as L
    from bwd_flashattention_fwd_gb300.inputs import to_f64

    h, wt, t, dloss = make_lce_inputs(w, "cpu")
    sel = list(range(rows))
    hd, tn, dn = to_f64(h[sel]), t[sel].numpy().astype("int64"), dloss[sel].numpy().astype("float64")
    chunk = lambda v0, v1: to_f64(wt[v0:v1])  # noqa: E731  (decoded per chunk: 0.5 GB at a time)
    t0 = time.perf_counter()
    L.forward_rows(hd, tn, chunk, w.V)
    L.dhidden_rows(hd, tn, dn, chunk, w.V)
    dt = time.perf_counter() - t0
    # forward_rows twice (once inside dhidden_rows) plus g W: four products of 2 V Dm per row
    credited = rows * 4 * 2.0 * w.V * w.Dm
    return {"value": credited / dt / 1e12, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 oracle loss and dH for {rows} rows at full vocabulary and hidden size "
                      f"({credited:.3g} FLOP, {dt:.2f} s)"}


def run_lce(args):
    from bwd_flashattention_fwd_gb300 import build, gbattn

    rank, local_rank, ws_n = replicas.world()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    replicas.init("nccl")
    build.build()
    gbattn.load_library()
    w = LCE_WORKLOADS[args.lce_workload]
    h, wt, t, dloss = make_lce_inputs(w, dev)
    loss = torch.empty(w.N, dtype=torch.float32, device=dev)
    lse = torch.empty_like(loss)
    dh, dw = torch.empty_like(h), torch.empty_like(wt)
    wsb = gbattn.lce_workspace(h, wt)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        gbattn.lce_fwd(h, wt, t, loss, lse, wsb, stream)
        if ev is not None:
            ev[1].record(stream)
        gbattn.lce_bwd(h, wt, t, lse, dloss, dh, dw, wsb, stream)
        if ev is not None:
            ev[2].record(stream)

    clocks = ClockSampler(physical_gpu_index(local_rank))
    clocks.start()
    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        step()
    torch.cuda.synchronize(dev)
    if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
        raise RuntimeError("device-side wait timed out during warm-up")
    clocks.wait_first()
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    replicas.barrier(dev)
    torch.cuda.synchronize(dev)
    clocks.begin()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(events[i])
    torch.cuda.synchronize(dev)
    clocks.end()
    replicas.barrier(dev)
    clocks.stop()
    clk = clocks.window()
    if gbattn.attn_last_device_status(stream) != gbattn.ATTN_OK:
        raise RuntimeError("device-side wait timed out during the timed steps")
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in events)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in events)
    local_s = sum(e[0].elapsed_time(e[2]) for e in events) / 1e3
    f_fwd = 2.0 * w.N * w.V * w.Dm
    f_bwd = 3.0 * f_fwd
    value_flops, _, max_s = replicas.aggregate_throughput((f_fwd + f_bwd) * args.steps, local_s, dev)
    peaks = load_peaks()
    pk = peaks["bf16_tflops_sustained"]
    kernels = {}
    for n, fl, ms in (("lce_fwd", f_fwd, fwd_ms), ("lce_bwd", f_bwd, bwd_ms)):
        ach = fl / (ms * 1e-3) / 1e12
        kernels[n] = {"bound": "tensor", "achieved": ach, "peak": pk, "unit": "TFLOP/s", "frac": ach / pk,
                      "frac_burst": ach / peaks["bf16_tflops"], "avg_ms": ms, "algorithmic": fl, "traffic": None}
    dominant = max(kernels, key=lambda n: kernels[n]["avg_ms"])
    roof = {k2: kernels[dominant][k2] for k2 in ("bound", "achieved", "peak", "unit", "frac", "traffic")}
    roof["kernel"] = {"lce_fwd": "lce_fwd (fused logits tiles + online LSE, then the row merge)",
                      "lce_bwd": "lce_bwd (per vocabulary chunk: gradient tiles, dH and dW products; all "
                                 "tcgen05 kernels of this library)"}[dominant]
    roof["peak_kind"] = (f"bf16 dense, sustained ({peaks['source']}; each step runs ~25 ms of back-to-back "
                         "products under the power cap)")
    roof["frac_burst"] = kernels[dominant]["frac_burst"]

    e2e = None
    if not args.no_e2e:
        # per step: hidden, targets and dloss in from pinned host memory; loss and
        # dH back; the weight and its gradient stay on the device (parameters)
        hh, th, dh_host = h.cpu().pin_memory(), t.cpu().pin_memory(), dloss.cpu().pin_memory()
        loss_h = torch.empty_like(loss, device="cpu").pin_memory()
        dhid_h = torch.empty_like(dh, device="cpu").pin_memory()
        n = max(3, min(args.steps, 10))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(n):
            h.copy_(hh, non_blocking=True)
            t.copy_(th, non_blocking=True)
            dloss.copy_(dh_host, non_blocking=True)
            step()
            loss_h.copy_(loss, non_blocking=True)
            dhid_h.copy_(dh, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        es = e0.elapsed_time(e1) / 1e3
        ev, _, _ = replicas.aggregate_throughput((f_fwd + f_bwd) * n, es, dev)
        e2e = {"value": ev / 1e12, "unit": UNIT, "steps": n, "ms_per_step": es * 1e3 / n,
               "h2d_bytes_per_step": sum(x.numel() * x.element_size() for x in (hh, th, dh_host)),
               "d2h_bytes_per_step": sum(x.numel() * x.element_size() for x in (loss_h, dhid_h))}
    n_chunks = -(-w.V // 16384)
    line = {
        "metric": METRIC_LCE, "value": value_flops / 1e12, "unit": UNIT, "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": max_s * 1e3 / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "N": w.N, "hidden": w.Dm, "vocab": w.V, "h_std": w.h_std, "w_std": w.w_std,
                   "seed": w.seed, "l2": "256 MiB written between steps; the weight (1.2 GB) exceeds L2",
                   "parallelism": "replicas" if ws_n > 1 else "single GPU",
                   "flops": "forward 2 N V Dm; backward 3 x that (recomputed logits, g W, g^T H)",
                   "timing": "CUDA events on the launching stream, sum over steps"},
        "pct_of_bf16_peak": 100.0 * value_flops / 1e12 / ws_n / peaks["bf16_tflops"],
        "peaks": peaks, "phase_ms": {"lce_fwd": fwd_ms, "lce_bwd": bwd_ms}, "roofline": roof, "kernels": kernels,
        "e2e": e2e,
        # ours: logits kernel + combine (forward); per chunk the gradient tiles and the dH and dW products
        "gpu_launches": args.steps * (2 + 3 * n_chunks),
        "library_launches_per_step": {},
        "clocks": clk, "kernel_source_hash": kernel_source_hash(),
    }
    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = lce_cpu_baseline(w)
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    replicas.shutdown()
    return 0


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--block-mask", default="none",
                    help="block-sparse pattern: none, window:W (W key blocks of 128), random:P")
    ap.add_argument("--kv-capacity", type=int, default=0,
                    help="k/v as the first Lk rows of an N-row cache per head (0: contiguous)")
    ap.add_argument("--decode", action="store_true", help="short-query path (attn_fwd_decode / attn_bwd_decode)")
    ap.add_argument("--lce", action="store_true", help="fused linear cross-entropy step instead of attention")
    ap.add_argument("--lce-workload", default="lce_qwen3_8b_n8192", choices=sorted(LCE_WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-long-run", action="store_true",
                    help=f"skip the extra {LONG_RUN_STEPS}-step run reported beside a shorter timed region")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-canary", action="store_true",
                    help="skip the library GEMM run before and after the timed steps (for kernel launch lists)")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the fp64 oracle on every full workload (host cores; no GPU)")
    ap.add_argument("--cpu-rows", type=int, default=1024, help="query rows in the CPU-baseline sample")
    ap.add_argument("--ref-rows", type=int, default=128, help="query rows per reference-arm step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.oracle_table:
        return run_oracle_table(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.lce:
        return run_lce(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
