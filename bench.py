#!/usr/bin/env python
"""Throughput of the tensor-parallel MLP (column-parallel linear + GeLU -> row-parallel linear,
forward + backward, all shards on one GB300) through the library's C ABI.

One step = tp_mlp_forward + tp_mlp_backward over one batch of the workload (every kernel of the
path: column GEMM with the bias + GeLU epilogue, row GEMM with the fused shard sum, the dY GEMM
with the GeLU' epilogue, both weight-gradient GEMMs, the input-gradient GEMM with the fused
shard sum, and the bias-gradient column sums). Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W]
                  [--workload gpt3|mlp2|p3|attn|p3col|ln|sweep:T:n]
                  [--reduce fused|partials] [--impl native|reference]

--impl reference times the fp64 CPU oracle on the host cores instead (a bounded sample of the
same workload per step). With N > 1 (torchrun) every rank runs an independent replica of the
workload on its own GPU: there is no exchange between the replicas (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "TP-sharded MLP fwd+bwd TFLOP/s (bf16) on 1 GB300 and % of tensor-core peak"
UNIT = "TFLOP/s"
KERNEL_SOURCES = ["tc_gemm.cuh", "tc2_gemm.cuh", "tc_launch.cu", "tc_gemm_kmn.cu", "tc_gemm_kk.cu",
                  "tc_gemm_mnmn.cu", "tc_gemm_dual.cu", "device_common.cuh"]
# fp32 FFMA peak: 152 SMs x 128 lanes x 2 flops per FFMA x 2.07 GHz (maximum SM clock).
FFMA_F32_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
TRACE_PER_STEP = 24  # trace slots per step (launches per step are at most 16)
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gemm_tc_gpt3_mlp_T2048_tp8.md")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="gpt3")
    ap.add_argument("--reduce", choices=["fused", "partials", "auto", "partials_bf16", "overlap"],
                    default="auto")
    ap.add_argument("--sp", action="store_true",
                    help="sequence-parallel step: token-sharded X, dZ in and Z, dX out")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--oracle-full", action="store_true",
                    help="time the fp64 oracle on whole workloads (comma-separated --workload "
                         "names, attn included) on the host cores; no GPU")
    return ap.parse_args()


def workload(name: str) -> wl.MlpWorkload:
    if name == "gpt3":
        return wl.GPT3_MLP_T2048_TP8
    if name == "mlp2":
        return wl.MLP_T4096_H1024_F4096_TP2
    if name == "p3":
        return wl.P3_FP32_FWD
    if name.startswith("sweep:"):
        _, T, n = name.split(":")
        return wl.SWEEP_H8192_F28672.with_shape(tokens=int(T), tp_degree=int(n))
    if name.startswith("mlp:"):
        # a smaller case with the GPT-3-shaped slice's distributions (for profiler captures
        # that must stay small): mlp:T:H:F:n
        _, T, H, F, n = name.split(":")
        w = wl.GPT3_MLP_T2048_TP8.with_shape(tokens=int(T), hidden=int(H), ffn=int(F),
                                             tp_degree=int(n))
        return wl.dataclasses.replace(w, name=f"mlp_bf16_T{T}_H{H}_F{F}_tp{n}")
    raise SystemExit(f"unknown workload {name}")


# ----------------------------------------------------------------------------- distributed
def dist_setup(gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != gpus and world > 1:
        raise SystemExit(f"--gpus {gpus} but WORLD_SIZE {world}")
    return world, rank, local


def dist_init(world: int, local: int):
    import torch
    import torch.distributed as dist

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return torch.device("cuda", local)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (the slowest replica's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(work_per_step: float, steps: int, ms_local: float, world: int):
    """Whole-job throughput of `world` independent replicas: all replicas' work divided by the
    slowest replica's time. Returns (max ms, TFLOP/s)."""
    ms = max_over_ranks(ms_local, world)
    return ms, work_per_step * steps * world / (ms / 1e3) / 1e12


# ----------------------------------------------------------------------------- clocks
CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
CLOCK_INTERVAL_MS = 50


def enforced_power_limit(device_index: int):
    """The board's enforced power limit in W (read only; None if nvidia-smi cannot say)."""
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=enforced.power.limit",
                              "--format=csv,noheader,nounits", "-i", str(device_index)],
                             capture_output=True, text=True, timeout=10)
        return float(out.stdout.strip().splitlines()[0]) if out.returncode == 0 else None
    except (OSError, ValueError, IndexError, subprocess.TimeoutExpired):
        return None


def parse_clock_lines(text: str, window=None) -> dict:
    """Clock samples (nvidia-smi CSV lines of CLOCK_QUERY) -> the summary put on the JSON line.
    With window = (t0, t1) (host wall-clock seconds of the timed region), only samples stamped
    inside it count for the median SM clock and the reasons; the samples before and after it
    (an idle GPU at its highest clock) would otherwise pull the median up."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    rows = []
    for line in text.strip().splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 10:
            continue
        try:
            ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            ts += float("0." + f[0].split(".")[1]) if "." in f[0] else 0.0
            rows.append((ts, float(f[2]), float(f[3]), float(f[4]),
                         {nm for nm, v in zip(names, f[6:10]) if v.lower() == "active"}))
        except (ValueError, IndexError):
            continue
    inside = [r for r in rows if window is None or window[0] <= r[0] <= window[1]]
    basis = "samples inside the timed region"
    if window is not None and not inside:
        # a region shorter than the sampling interval: the first samples after it started
        inside = [r for r in rows if r[0] >= window[0]][:2]
        basis = "first samples after the timed region started (region shorter than the interval)"
    sm = [r[1] for r in inside]
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(r[2] for r in rows) if rows else None,
            "power_w_median": statistics.median([r[3] for r in inside]) if inside else None,
            "samples": len(inside), "samples_total": len(rows),
            "interval_ms": CLOCK_INTERVAL_MS, "basis": basis,
            "reasons": sorted(set().union(*[r[4] for r in inside])) if inside else []}


class ClockSampler:
    def __init__(self, device_index: int):
        self.proc = None
        self.device_index = device_index
        self.window = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                 "-i", str(device_index), "-lms", str(CLOCK_INTERVAL_MS)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def mark(self, t0: float, t1: float) -> None:
        """Host wall-clock bounds of the timed region."""
        self.window = (t0, t1)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        res = parse_clock_lines(out, self.window)
        res["power_limit_w"] = enforced_power_limit(self.device_index)
        if self.window is not None:
            res["timed_region_s"] = self.window[1] - self.window[0]
        return res


# ----------------------------------------------------------------------------- peaks / profile
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"bf16_sustained": p["bf16_tflops_sustained"], "bf16_burst": p["bf16_tflops"],
                "hbm_gbs": p["hbm_gbs"], "source": "measured", "ffma_f32": FFMA_F32_TFLOPS,
                "sm_max_mhz": p.get("sm_max_mhz", 2070.0)}
    return {"bf16_sustained": 1700.0, "bf16_burst": 1900.0, "hbm_gbs": 6800.0,
            "source": "fallback", "ffma_f32": FFMA_F32_TFLOPS, "sm_max_mhz": 2070.0}


def code_lines(text: str):
    """The lines of a C++ source with // comments and blank lines removed (a comment edit does
    not change the kernel the counters were taken on)."""
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            yield code


def kernel_source_hash(read=None) -> str:
    """Hash of the code of the tensor-core GEMM's sources; `read(name)` supplies a file's text
    (default: the working tree)."""
    if read is None:
        def read(f):
            return open(os.path.join(ROOT, "tensor_sharded_linear_bias_gb300", "csrc", f)).read()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        for line in code_lines(read(f)):
            h.update(line.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch of the tensor-core GEMM from the committed ncu summary, if that
    summary was taken on the current kernel source and this workload; else None."""
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    fields = {}
    for line in open(PROFILE_SUMMARY):
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    if fields.get("kernel_source_sha") != kernel_source_hash():
        return None
    if fields.get("workload") != workload_name:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- the step
class MlpBench:
    def __init__(self, w: wl.MlpWorkload, reduce: int, device, keep_host: bool, sp: bool = False):
        import numpy as np
        import torch

        import tensor_sharded_linear_bias_gb300 as tp

        self.tp, self.w, self.device = tp, w, device
        bf16 = w.dtype == "bf16"
        cdt = torch.bfloat16 if bf16 else torch.float32
        n, T, H, F = w.tp_degree, w.tokens, w.hidden, w.ffn
        Fs = F // n
        raw = wl.mlp_tensors(w)
        host = {}
        dev = {}
        for k, v in raw.items():
            if bf16:
                t, f = wl.to_bf16(v)
            else:
                t, f = torch.from_numpy(np.ascontiguousarray(v)), v
            dev[k] = t
            if keep_host:
                host[k] = f
        del raw
        self.host = host
        self.X = dev["X"].to(device)
        self.dZ = dev["dZ"].to(device)
        self.X_pinned = dev["X"].pin_memory()
        self.dZ_pinned = dev["dZ"].pin_memory()
        self.A = [dev["A"][:, i * Fs:(i + 1) * Fs].contiguous().to(device) for i in range(n)]
        self.a = [dev["a"][i * Fs:(i + 1) * Fs].contiguous().to(device) for i in range(n)]
        self.B = [dev["B"][i * Fs:(i + 1) * Fs, :].contiguous().to(device) for i in range(n)]
        self.b = dev["b"].to(device)
        del dev
        self.desc = tp.MlpDesc(tokens=T, hidden=H, ffn=F, tp_degree=n,
                               dtype=tp.TP_BF16 if bf16 else tp.TP_F32,
                               act=tp.TP_ACT_GELU_ERF, reduce=reduce)
        self.sp = sp
        self.ws = tp.new_workspace(tp.tp_mlp_sp_workspace_size(self.desc) if sp else
                                   tp.tp_mlp_workspace_size(self.desc), device)
        if sp:
            Ts = T // n
            self.Xs = [self.X[j * Ts:(j + 1) * Ts].contiguous() for j in range(n)]
            self.dZs = [self.dZ[j * Ts:(j + 1) * Ts].contiguous() for j in range(n)]
            self.Zs = [torch.empty(Ts, H, dtype=torch.float32, device=device) for _ in range(n)]
            self.dXs = [torch.empty(Ts, H, dtype=torch.float32, device=device) for _ in range(n)]
        f32 = dict(dtype=torch.float32, device=device)
        self.Z = torch.empty(T, H, **f32)
        self.Hs = [torch.empty(T, Fs, dtype=cdt, device=device) for _ in range(n)]
        self.Ys = [torch.empty(T, Fs, dtype=cdt, device=device) for _ in range(n)]
        self.dX = torch.empty(T, H, **f32)
        self.dA = [torch.empty(H, Fs, **f32) for _ in range(n)]
        self.dB = [torch.empty(Fs, H, **f32) for _ in range(n)]
        self.da = [torch.empty(Fs, **f32) for _ in range(n)]
        self.db = torch.empty(H, **f32)
        self.h2d_stream = torch.cuda.Stream(device=device)
        self.d2h_stream = torch.cuda.Stream(device=device)
        self.X2 = [self.X, torch.empty_like(self.X)]
        self.dZ2 = [self.dZ, torch.empty_like(self.dZ)]
        self.Z2 = [self.Z, torch.empty_like(self.Z)]
        self.dX2 = [self.dX, torch.empty_like(self.dX)]
        self.Z_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
        self.dX_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
        self.backward = w.backward
        e = 2 if bf16 else 4
        self.operand_bytes = e * (T * H * 2 + 2 * H * F) + e * 2 * T * F

    def step(self):
        tp = self.tp
        if self.sp:
            tp.tp_mlp_forward_sp(self.desc, self.Xs, self.A, self.a, self.B, self.b, self.Zs,
                                 self.Hs, self.Ys, self.ws)
            if self.backward:
                tp.tp_mlp_backward_sp(self.desc, self.Xs, self.A, self.B, self.Hs, self.Ys,
                                      self.dZs, self.dXs, self.dA, self.da, self.dB, self.db,
                                      self.ws)
            return
        tp.tp_mlp_forward(self.desc, self.X, self.A, self.a, self.B, self.b, self.Z, self.Hs,
                          self.Ys, self.ws)
        if self.backward:
            tp.tp_mlp_backward(self.desc, self.X, self.A, self.B, self.Hs, self.Ys, self.dZ,
                               self.dX, self.dA, self.da, self.dB, self.db, self.ws)

    def run_e2e(self, steps: int) -> None:
        """`steps` steps end to end: every step uploads its inputs (X, dZ) from pinned host
        memory and downloads its results (Z, dX) to pinned host memory. Two device slots per
        input and output let the copies of neighbouring steps overlap compute, as a training
        loop's input prefetch does: step i+1's uploads run during step i, Z's download during
        the backward, dX's download during the next step's forward. All copies are issued on
        two copy streams (host->device, device->host) ordered by events; the caller's stream
        runs the compute and, at the end, waits for both copy streams."""
        import torch

        tp = self.tp
        cur = torch.cuda.current_stream()
        h2d, d2h = self.h2d_stream, self.d2h_stream
        h2d.wait_stream(cur)
        d2h.wait_stream(cur)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        bwd_done, zdown, dxdown = {}, {}, {}
        for i in range(steps):
            s = i % 2
            X, dZ, Z, dX = self.X2[s], self.dZ2[s], self.Z2[s], self.dX2[s]
            x_ready, dz_ready, fwd_done = ev(), ev(), ev()
            with torch.cuda.stream(h2d):
                if i - 2 in bwd_done:
                    h2d.wait_event(bwd_done[i - 2])   # slot s is no longer read
                X.copy_(self.X_pinned, non_blocking=True)
                x_ready.record(h2d)
                if self.backward:
                    dZ.copy_(self.dZ_pinned, non_blocking=True)
                    dz_ready.record(h2d)
            cur.wait_event(x_ready)
            if i - 2 in zdown:
                cur.wait_event(zdown[i - 2])          # Z slot downloaded
            tp.tp_mlp_forward(self.desc, X, self.A, self.a, self.B, self.b, Z, self.Hs,
                              self.Ys, self.ws)
            fwd_done.record(cur)
            if self.backward:
                cur.wait_event(dz_ready)
                if i - 2 in dxdown:
                    cur.wait_event(dxdown[i - 2])     # dX slot downloaded
                tp.tp_mlp_backward(self.desc, X, self.A, self.B, self.Hs, self.Ys, dZ, dX,
                                   self.dA, self.da, self.dB, self.db, self.ws)
                bwd_done[i] = ev()
                bwd_done[i].record(cur)
            with torch.cuda.stream(d2h):
                d2h.wait_event(fwd_done)
                self.Z_host.copy_(Z, non_blocking=True)
                zdown[i] = ev()
                zdown[i].record(d2h)
                if self.backward:
                    d2h.wait_event(bwd_done[i])
                    self.dX_host.copy_(dX, non_blocking=True)
                    dxdown[i] = ev()
                    dxdown[i].record(d2h)
        cur.wait_stream(h2d)
        cur.wait_stream(d2h)

    def e2e_step(self):
        """One step end to end, serially on the current stream: upload X (and dZ) from pinned
        host memory, forward (and backward), download Z (and dX) to pinned host memory."""
        tp = self.tp
        self.X.copy_(self.X_pinned, non_blocking=True)
        if self.backward:
            self.dZ.copy_(self.dZ_pinned, non_blocking=True)
        tp.tp_mlp_forward(self.desc, self.X, self.A, self.a, self.B, self.b, self.Z, self.Hs,
                          self.Ys, self.ws)
        self.Z_host.copy_(self.Z, non_blocking=True)
        if self.backward:
            tp.tp_mlp_backward(self.desc, self.X, self.A, self.B, self.Hs, self.Ys, self.dZ,
                               self.dX, self.dA, self.da, self.dB, self.db, self.ws)
            self.dX_host.copy_(self.dX, non_blocking=True)

    @property
    def flops(self) -> int:
        return self.w.flops_fwd_bwd if self.backward else self.w.flops_fwd

    @property
    def h2d_bytes(self) -> int:
        return self.X.numel() * self.X.element_size() * (2 if self.backward else 1)

    @property
    def d2h_bytes(self) -> int:
        return self.Z.numel() * 4 * (2 if self.backward else 1)


L2_FLUSH_FACTOR = 4  # flush between steps unless a step reads this many L2 sizes of operands


class L2Flush:
    """Before a timed step, outside the step's events: writes a buffer of twice the L2 size (a
    different value each time), then reads a second one of the same size. The write evicts the
    previous step's data; the read evicts the written lines again, so that their write-back to
    HBM is not charged to the timed step. The step then starts with a cold, clean L2."""

    def __init__(self, device):
        import torch

        props = torch.cuda.get_device_properties(device)
        self.l2 = int(getattr(props, "L2_cache_size", 0) or (126 << 20))
        self.buf = torch.empty(2 * self.l2 // 4, dtype=torch.float32, device=device)
        self.clean = torch.ones(2 * self.l2 // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)
        self.k = 0

    def __call__(self):
        import torch

        self.k += 1
        self.buf.fill_(float(self.k))
        torch.sum(self.clean, dim=0, out=self.sink)

    def describe(self) -> str:
        return (f"flushed: {self.buf.numel() * 4 / 1e6:.0f} MB written, then another "
                f"{self.clean.numel() * 4 / 1e6:.0f} MB read, before every timed step, outside "
                f"the step's events (L2 {self.l2 / 1e6:.0f} MB)")


def make_flush(device, operand_bytes: int):
    """An L2 flush when the step's operands are fewer than L2_FLUSH_FACTOR L2 sizes, else None."""
    f = L2Flush(device)
    if operand_bytes >= L2_FLUSH_FACTOR * f.l2:
        return None, (f"no flush: {operand_bytes / 1e9:.2f} GB of operands per step vs "
                      f"{f.l2 / 1e6:.0f} MB of L2")
    return f, f.describe()


def time_steps(fn, steps: int, world: int, flush=None, host_ahead: bool = False):
    """Device time of `steps` calls of fn (ms), barrier + synchronize on both sides. Without a
    flush: one event pair around all steps. With one: flush, then an event pair around each
    step; the sum of the steps' times. host_ahead (no flush): a sleep kernel runs on the stream
    before the start event while the host enqueues every step, so that a step whose host-side
    enqueue takes longer than its device time (a few-token step) is timed on the device, not
    on the host."""
    import torch

    barrier(world)
    torch.cuda.synchronize()
    if flush is None:
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        if host_ahead and hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(2e6 * (1.0 + 0.2 * steps)))  # ~1 ms + 0.2 ms per step at 2 GHz
        start.record()
        for _ in range(steps):
            fn()
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(end)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for a, b in evs:
        flush()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    barrier(world)
    return sum(a.elapsed_time(b) for a, b in evs)


def timed_then_traced(tp, fn, steps: int, world: int, flush, trace_capacity: int, sampler):
    """Times `steps` steps with tracing off (the reported throughput), then the same number of
    steps with the library's per-launch trace on (per-kernel times for the roofline).
    Returns (ms of the untraced steps, trace records, clocks sampled during the untraced
    steps)."""
    t0 = time.time()
    ms = time_steps(fn, steps, world, flush)
    if sampler:
        sampler.mark(t0, time.time())
    clocks = sampler.stop() if sampler else None
    tp.tp_trace_start(trace_capacity)
    time_steps(fn, steps, world, flush)
    recs = tp.tp_trace_stop(trace_capacity)
    return ms, recs, clocks


# Dense bf16 tensor-core rate per SM and clock: 8192 flop (a 128 x 256 x 16 MMA per 128 cycles).
# Consistent with ncu on GB300: cuBLAS's kernel for a 2048 x 8192 x 28672 GEMM ran 2030 TFLOP/s
# with its tensor pipe 96 % busy at ~1.65-1.7 GHz (2030e12 / (0.96 * 152 * 8192) = 1.70 GHz).
TENSOR_FLOP_PER_CLK_SM = 8192
NUM_SMS = 152
BURST_REGION_S = 2.0     # longer timed regions run into the power cap: the sustained peak
BURST_CLOCK_FRAC = 0.97  # median SM clock within 3 % of its maximum: a burst


def tensor_peak(pk, clocks):
    """The measured bf16 peak that matches the timed region's regime. MEASURED_PEAKS.json holds
    a burst figure (cuBLAS timed alone, best of 10, at the maximum clock) and a sustained one
    (cuBLAS back to back for seconds under the power cap). A short region is a burst and is
    divided by the burst peak; only a region long enough for the power cap to pull the clock
    down (over BURST_REGION_S, with the median clock below the maximum) is divided by the
    sustained peak. Returns (peak, regime, note)."""
    mhz = (clocks or {}).get("sm_mhz")
    mx = (clocks or {}).get("sm_max_mhz") or pk.get("sm_max_mhz") or 2070.0
    region = (clocks or {}).get("timed_region_s")
    long_region = region is not None and region > BURST_REGION_S
    capped = mhz is not None and mhz < BURST_CLOCK_FRAC * mx
    if not (long_region and capped):
        return pk["bf16_burst"], "burst", (f"MEASURED_PEAKS.json bf16_tflops (of {pk['source']}): "
                                          f"median SM clock {mhz} of {mx} MHz over a "
                                          f"{region if region is None else round(region, 3)} s region")
    return pk["bf16_sustained"], "sustained", (f"MEASURED_PEAKS.json bf16_tflops_sustained (of "
                                              f"{pk['source']}): median SM clock {mhz} of {mx} "
                                              f"MHz over a {region if region is None else round(region, 3)} s region")


def tensor_fractions(achieved, pk, clocks):
    """The same achieved rate against every denominator: both measured peaks, the burst peak
    scaled to the region's median clock (the burst ran at the maximum clock), and the tensor
    pipe's own rate at that clock."""
    mhz = (clocks or {}).get("sm_mhz")
    mx = pk.get("sm_max_mhz") or 2070.0
    out = {"frac_vs_burst": achieved / pk["bf16_burst"],
           "frac_vs_sustained": achieved / pk["bf16_sustained"]}
    if mhz:
        scaled = pk["bf16_burst"] * mhz / mx
        pipe = TENSOR_FLOP_PER_CLK_SM * NUM_SMS * mhz * 1e6 / 1e12
        out["clock_normalised"] = {"peak": scaled, "frac": achieved / scaled, "sm_mhz": mhz,
                                   "note": f"bf16_tflops x {mhz} / {mx} MHz (the burst peak "
                                           f"taken at the maximum clock)"}
        out["tensor_pipe_at_clock"] = {"peak": pipe, "frac": achieved / pipe,
                                       "note": f"{TENSOR_FLOP_PER_CLK_SM} flop/clock/SM x "
                                               f"{NUM_SMS} SMs x {mhz} MHz"}
    return out


def roofline_from_trace(recs, pk, workload_name=None, clocks=None):
    """The dominant kernel (largest total traced device time) against its roofline, and the
    per-(kernel, tag) breakdown."""
    by_kernel, by_tag = {}, {}
    for r in recs:
        k = by_kernel.setdefault(r["kernel"], {"ms": 0.0, "flops": 0.0, "bytes": 0.0, "n": 0})
        k["ms"] += r["ms"]
        k["flops"] += r["flops"]
        k["bytes"] += r["bytes"]
        k["n"] += 1
        t = by_tag.setdefault(f'{r["kernel"]}:{r["tag"]}', {"ms": 0.0, "flops": 0.0, "n": 0})
        t["ms"] += r["ms"]
        t["flops"] += r["flops"]
        t["n"] += 1
    dom = max(by_kernel, key=lambda k: by_kernel[k]["ms"])
    d = by_kernel[dom]
    total_ms = sum(v["ms"] for v in by_kernel.values())
    if dom == "gemm_tc":
        achieved = d["flops"] / (d["ms"] / 1e3) / 1e12
        peak, regime, note = tensor_peak(pk, clocks)
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "regime": regime,
                "peak_source": note, **tensor_fractions(achieved, pk, clocks)}
    elif dom == "gemm_ffma":
        achieved = d["flops"] / (d["ms"] / 1e3) / 1e12
        peak = pk["ffma_f32"]
        roof = {"bound": "alu", "kernel": dom, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2.07 GHz"}
    else:
        achieved = d["bytes"] / (d["ms"] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / pk["hbm_gbs"],
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs (of {pk['source']})"}
    if roof["unit"] != "GB/s":
        # the same launches as algorithmic bytes per second, against HBM
        gbs = d["bytes"] / (d["ms"] / 1e3) / 1e9
        roof["hbm_view"] = {"achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                            "frac": gbs / pk["hbm_gbs"]}
    roof["launches"] = d["n"]
    roof["avg_launch_ms"] = d["ms"] / d["n"]
    roof["share_of_kernel_time"] = d["ms"] / total_ms
    traffic = profiled_traffic(workload_name) if workload_name else None
    roof["traffic"] = traffic
    roof["traffic_note"] = ("dram__bytes_read.sum + dram__bytes_write.sum per launch from the "
                            "committed ncu summary" if traffic is not None else
                            "null: no ncu capture of the current kernel source for this workload")
    kernels = {k: {"launches": v["n"], "avg_ms": v["ms"] / v["n"],
                   "tflops": (v["flops"] / (v["ms"] / 1e3) / 1e12) if v["flops"] else None,
                   "share": v["ms"] / total_ms} for k, v in sorted(by_tag.items())}
    return roof, kernels


# ----------------------------------------------------------------------------- the oracle
def oracle_sample(w: wl.MlpWorkload, host: dict, rows: int, cols_per_shard: int):
    """A bounded sample of the workload for the CPU oracle: `rows` token rows and the first
    `cols_per_shard` ffn columns of every shard (the MLP restricted to those rows and ffn
    columns, still split into tp_degree shards). Returns (callable, flops per call, text)."""
    import numpy as np

    import oracle

    n, Fs = w.tp_degree, w.ffn // w.tp_degree
    c = min(cols_per_shard, Fs)
    r = min(rows, w.tokens)
    cols = np.concatenate([np.arange(i * Fs, i * Fs + c) for i in range(n)])
    X, dZ = host["X"][:r], host["dZ"][:r]
    A, a, B, b = host["A"][:, cols], host["a"][cols], host["B"][cols, :], host["b"]

    def run():
        fwd = oracle.mlp_forward(X, A, a, B, b, n)
        if w.backward:
            oracle.mlp_backward(X, A, a, B, b, dZ, n, fwd)

    per = (12 if w.backward else 4) * r * w.hidden * (c * n)
    text = (f"{r} token rows x {c} ffn columns per shard ({c * n} of {w.ffn}) of the workload, "
            f"{'fwd+bwd' if w.backward else 'fwd'}, fp64 numpy")
    return run, per, text


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(w, host, seconds: float):
    run, per, text = oracle_sample(w, host, rows=256, cols_per_shard=64)
    run()  # warm caches / BLAS threads
    reps, t0 = 0, time.perf_counter()
    while True:
        run()
        reps += 1
        el = time.perf_counter() - t0
        if (el >= seconds and reps >= 3) or reps >= 1000:
            break
    value = per * reps / el / 1e12
    return {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
            "sample": f"{text}; {reps} repetitions in {el:.1f} s"}


def mem_available_bytes():
    """MemAvailable of the host (Linux), or None."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except OSError:
        pass
    return None


def timed_cpu(fn):
    """Wall-clock seconds of fn() and the host threads it kept busy on average (process CPU
    time / wall time)."""
    c0, t0 = os.times(), time.perf_counter()
    fn()
    el = time.perf_counter() - t0
    c1 = os.times()
    busy = ((c1.user - c0.user) + (c1.system - c0.system)) / el if el > 0 else 0.0
    return el, busy


def oracle_full_line(name: str) -> dict:
    """The fp64 oracle as it stands, on the whole workload (every output of fwd + bwd), timed
    on the host cores. Workloads whose oracle would not fit the host's free memory (about 3x
    the fp64 inputs and outputs) or whose full run is long (T >= 8192 in the sweep) are timed
    on their first 1024 token rows (every ffn column; the MLP restricted to those rows) and
    extrapolated by flops, labelled as such."""
    import numpy as np  # noqa: F401

    import oracle

    if name == "attn":
        w = wl.ATTN_T4096_H5120_TP8
        t = {k: wl.to_bf16(v)[1] for k, v in wl.attn_tensors(w).items()}

        def run():
            oracle.attn_forward(t["X"], t["Wqkv"], t["C"], t["Wo"], w.heads, w.head_dim,
                                w.tp_degree)
            oracle.attn_backward(t["X"], t["Wqkv"], t["C"], t["Wo"], t["dQKV"], t["dO"],
                                 w.heads, w.head_dim, w.tp_degree)

        flops, kind, text = w.flops_fwd_bwd, "full", "whole workload, fwd+bwd, fp64 numpy"
    else:
        w = workload(name)
        host = {k: (wl.to_bf16(v)[1] if w.dtype == "bf16" else v)
                for k, v in wl.mlp_tensors(w).items()}
        T, H, F = w.tokens, w.hidden, w.ffn
        need = 8 * 3 * (2 * T * H + 2 * H * F + 3 * T * F + (2 * H * F if w.backward else 0))
        avail = mem_available_bytes()
        full = (T < 8192) and (avail is None or need < avail)
        if full:
            def run():
                fwd = oracle.mlp_forward(host["X"], host["A"], host["a"], host["B"], host["b"],
                                         w.tp_degree)
                if w.backward:
                    oracle.mlp_backward(host["X"], host["A"], host["a"], host["B"], host["b"],
                                        host["dZ"], w.tp_degree, fwd)

            flops = w.flops_fwd_bwd if w.backward else w.flops_fwd
            kind = "full"
            text = f"whole workload, {'fwd+bwd' if w.backward else 'fwd'}, fp64 numpy"
        else:
            run, flops, text = oracle_sample(w, host, rows=1024, cols_per_shard=w.ffn)
            kind = "extrapolated from the measured sample"
            text += (f"; full run skipped: {'T >= 8192' if T >= 8192 else 'host memory'} "
                     f"(needs ~{need / 1e9:.0f} GB, {0 if avail is None else avail / 1e9:.0f} GB "
                     f"available)")
    el, busy = timed_cpu(run)
    if kind != "full":
        # a sample takes a fraction of a second: repeat it for a few seconds
        reps = max(1, int(3.0 / max(el, 1e-3)))
        el, busy = timed_cpu(lambda: [run() for _ in range(reps)])
        el /= reps
    tflops = flops / el / 1e12
    total = (w.flops_fwd_bwd if getattr(w, "backward", True) else w.flops_fwd) \
        if name != "attn" else w.flops_fwd_bwd
    shape = ({"tokens": w.tokens, "hidden": w.hidden, "heads": w.heads, "tp_degree": w.tp_degree}
             if name == "attn" else {"tokens": w.tokens, "hidden": w.hidden, "ffn": w.ffn,
                                     "tp_degree": w.tp_degree})
    return {"impl": "oracle", "workload": w.name, **shape, "kind": kind, "value": tflops,
            "unit": UNIT, "seconds": el, "seconds_full_workload": total / (tflops * 1e12),
            "cores": host_cores(), "nproc": os.cpu_count(), "threads_busy": round(busy, 1),
            "sample": text, "dtype": "f64"}


def run_oracle_full(args):
    """One JSON line per workload of --workload (comma-separated): the oracle's wall clock."""
    for name in args.workload.split(","):
        print(json.dumps(oracle_full_line(name.strip())), flush=True)
    return 0


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    import numpy as np  # noqa: F401

    host = {}
    raw = wl.mlp_tensors(w)
    for k, v in raw.items():
        host[k] = wl.to_bf16(v)[1] if w.dtype == "bf16" else v
    del raw
    run, per, text = oracle_sample(w, host, rows=128, cols_per_shard=32)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    el = time.perf_counter() - t0
    value = per * args.steps / el / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden,
                       "ffn": w.ffn, "tp_degree": w.tp_degree, "sample": text},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(),
                             "kind": "oracle", "sample": text},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- attention projections
class AttnBench:
    """The attention-projection workload: the fused QKV projection split by heads (column
    parallel, no bias, no activation) and the output projection split by rows (row parallel),
    forward and backward, through the linear entry points."""

    def __init__(self, w: wl.AttnWorkload, reduce: int, device):
        import torch

        import tensor_sharded_linear_bias_gb300 as tp

        self.tp, self.w = tp, w
        n, T, Hm, hd, heads = w.tp_degree, w.tokens, w.hidden, w.head_dim, w.heads
        hw = heads // n * hd
        t = {k: wl.to_bf16(v)[0].to(device) for k, v in wl.attn_tensors(w).items()}
        blk = lambda M, s: torch.cat([M[:, b * Hm + s * hw: b * Hm + (s + 1) * hw]  # noqa: E731
                                      for b in range(3)], 1).contiguous()
        self.X, self.dO = t["X"], t["dO"]
        self.Wq = [blk(t["Wqkv"], s) for s in range(n)]
        self.dQ = [blk(t["dQKV"], s) for s in range(n)]
        self.Cs = [t["C"][:, s * hw:(s + 1) * hw].contiguous() for s in range(n)]
        self.Wo = [t["Wo"][s * hw:(s + 1) * hw, :].contiguous() for s in range(n)]
        self.col = tp.LinearDesc(tokens=T, in_features=Hm, out_features=3 * Hm, tp_degree=n,
                                 dtype=tp.TP_BF16, act=0, reduce=reduce, gather=0)
        self.row = tp.LinearDesc(tokens=T, in_features=Hm, out_features=Hm, tp_degree=n,
                                 dtype=tp.TP_BF16, act=0, reduce=reduce, gather=0)
        self.ws = tp.new_workspace(max(tp.tp_linear_workspace_size(self.col, tp.TP_COLUMN),
                                       tp.tp_linear_workspace_size(self.row, tp.TP_ROW)), device)
        f32 = dict(dtype=torch.float32, device=device)
        self.QKV = [torch.empty(T, 3 * hw, dtype=torch.bfloat16, device=device) for _ in range(n)]
        self.O = torch.empty(T, Hm, **f32)
        self.dX = torch.empty(T, Hm, **f32)
        self.dWq = [torch.empty(Hm, 3 * hw, **f32) for _ in range(n)]
        self.dC = [torch.empty(T, hw, **f32) for _ in range(n)]
        self.dWo = [torch.empty(hw, Hm, **f32) for _ in range(n)]
        self.flops = w.flops_fwd_bwd
        self.operand_bytes = 2 * (2 * T * Hm + 3 * Hm * Hm + T * 3 * Hm + T * Hm + Hm * Hm)

    def step(self):
        tp = self.tp
        tp.tp_linear_column_forward(self.col, self.X, self.Wq, None, self.QKV, None, self.ws)
        tp.tp_linear_row_forward(self.row, self.Cs, self.Wo, None, self.O, self.ws)
        tp.tp_linear_column_backward(self.col, self.X, self.Wq, None, self.dQ, self.dX, self.dWq,
                                     None, self.ws)
        tp.tp_linear_row_backward(self.row, self.Cs, self.Wo, self.dO, self.dC, self.dWo, None,
                                  self.ws)


def run_attention(args, world, rank, local):
    import torch  # noqa: F401

    import tensor_sharded_linear_bias_gb300 as tp

    device = dist_init(world, local)
    w = wl.ATTN_T4096_H5120_TP8
    reduce = {"fused": tp.TP_REDUCE_FUSED, "partials": tp.TP_REDUCE_PARTIALS,
              "auto": tp.TP_REDUCE_AUTO, "partials_bf16": tp.TP_REDUCE_PARTIALS_BF16,
              "overlap": tp.TP_REDUCE_OVERLAP}[args.reduce]
    ab = AttnBench(w, reduce, device)
    for _ in range(args.warmup):
        ab.step()
    tp.tp_check_status(ab.ws)
    flush, l2_note = make_flush(device, ab.operand_bytes)
    sampler = ClockSampler(device.index or 0) if rank == 0 else None
    ms, recs, clocks = timed_then_traced(tp, ab.step, args.steps, world, flush,
                                         args.steps * TRACE_PER_STEP + 16, sampler)
    tp.tp_check_status(ab.ws)
    ms, value = replica_throughput(ab.flops, args.steps, ms, world)
    if rank == 0:
        pk = peaks()
        roof, kernels = roofline_from_trace(recs, pk, clocks=clocks)
        peak, regime, _ = tensor_peak(pk, clocks)
        print(json.dumps({
            "metric": "attention projections (QKV split by heads + output projection) fwd+bwd "
                      "TFLOP/s (bf16)",
            "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden,
                       "heads": w.heads, "head_dim": w.head_dim, "tp_degree": w.tp_degree,
                       "reduce": args.reduce, "l2": l2_note},
            "pct_of_peak": value / peak * 100.0, "pct_of_peak_basis": regime, "clocks": clocks,
            "gpu_launches": len(recs), "roofline": roof, "kernels": kernels}), flush=True)
    return 0


# ----------------------------------------------------------------------------- hidden-split LayerNorm
def run_layernorm(args, world, rank, local):
    """LayerNorm over a hidden dimension split into tp_degree shards (the statistics combined
    over the shards on the device), forward + backward (dX, dgamma, dbeta), bf16, GPT-3-sized
    rows: T 2048, H 12288, 8 shards. HBM-bound: reported in GB/s of algorithmic traffic."""
    import numpy as np
    import torch

    import tensor_sharded_linear_bias_gb300 as tp

    device = dist_init(world, local)
    T, H, n = 2048, 12288, 8
    Hs = H // n
    g = np.random.Generator(np.random.PCG64(9000))
    mk = lambda *shape, s=1.0, m=0.0: [  # noqa: E731
        torch.from_numpy((g.standard_normal(shape) * s + m).astype(np.float32)).to(device, torch.bfloat16)
        for _ in range(n)]
    X, dY = mk(T, Hs), mk(T, Hs)
    gam, bet = mk(Hs, s=0.5, m=1.0), mk(Hs, s=0.5)
    Y = [torch.empty(T, Hs, dtype=torch.bfloat16, device=device) for _ in range(n)]
    dX = [torch.empty(T, Hs, dtype=torch.bfloat16, device=device) for _ in range(n)]
    f32 = dict(dtype=torch.float32, device=device)
    mean, rstd = torch.empty(T, **f32), torch.empty(T, **f32)
    dg = [torch.empty(Hs, **f32) for _ in range(n)]
    db = [torch.empty(Hs, **f32) for _ in range(n)]
    desc = tp.LayerNormDesc(tokens=T, hidden=H, tp_degree=n, dtype=tp.TP_BF16, eps=1e-5)

    def step():
        tp.tp_layernorm_forward(desc, X, gam, bet, Y, mean, rstd)
        tp.tp_layernorm_backward(desc, X, gam, mean, rstd, dY, dX, dg, db)

    # algorithmic bytes: fwd reads X, writes Y; dX reads X, dY, writes dX; dgamma/dbeta read
    # X, dY (gamma, beta, statistics and parameter gradients are < 0.1 %)
    step_bytes = 7.0 * T * H * 2
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    flush, l2_note = make_flush(device, int(4 * T * H * 2))
    sampler = ClockSampler(device.index or 0) if rank == 0 else None
    ms, recs, clocks = timed_then_traced(tp, step, args.steps, world, flush,
                                         args.steps * TRACE_PER_STEP + 16, sampler)
    ms = max_over_ranks(ms, world)
    if rank == 0:
        pk = peaks()
        roof, kernels = roofline_from_trace(recs, pk, clocks=clocks)
        value = step_bytes * args.steps * world / (ms / 1e3) / 1e9
        print(json.dumps({
            "metric": "hidden-split LayerNorm fwd+bwd (8 shards, statistics combined on the "
                      "device) GB/s of algorithmic traffic (bf16)",
            "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "layernorm_bf16_T2048_H12288_tp8", "tokens": T, "hidden": H,
                       "tp_degree": n, "l2": l2_note},
            "pct_of_hbm": value / pk["hbm_gbs"] * 100.0, "clocks": clocks,
            "gpu_launches": len(recs), "roofline": roof, "kernels": kernels}), flush=True)
    return 0


# ----------------------------------------------------------------------------- pages' example
def run_p3_column_latency(args, world, rank, local):
    """Latency of the pages' column-parallel example: X [32, 768] times W [768, 3072] split
    into 4 column shards, bias per shard, outputs gathered into one [32, 3072] tensor
    (tp_linear_column_forward with gather = 1), fp32 as on the page and bf16."""
    import torch

    from tensor_sharded_linear_bias_gb300.modules import ColumnParallelLinear

    device = dist_init(world, local)
    w = wl.P3_FP32_FWD
    res = {}
    for name, dt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        weight = torch.from_numpy(wl.normal(1000 * w.cid + 1, (w.hidden, w.ffn), 0.01))
        layer = ColumnParallelLinear(w.hidden, w.ffn, w.tp_degree, dtype=dt, device=device,
                                     weight=weight, gather=True)
        x = torch.from_numpy(wl.normal(1000 * w.cid, (w.tokens, w.hidden), 1.0)).to(device, dt)
        for _ in range(max(args.warmup, 10)):
            layer.forward(x)
        layer.check()
        ms = time_steps(lambda: layer.forward(x), args.steps, world, L2Flush(device))
        ms = max_over_ranks(ms, world)
        res[name] = ms / args.steps * 1e3
    if rank == 0:
        print(json.dumps({
            "metric": "column-parallel linear latency, the pages' example (768 -> 3072, batch 32, "
                      "4 shards, gathered output)",
            "value": res["f32"], "unit": "us", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": False, "dtype": "f32",
            "data": "synthetic", "bf16_us": res["bf16"],
            "config": {"workload": "p3_column_linear_T32_K768_N3072_tp4_gather",
                       "calls": "tp_linear_column_forward, one CUDA event pair per call, L2 "
                                "flushed before each call outside its events"},
            "context": "the page expects ~1.5 ms on one GPU and ~1.2 ms with 4-GPU tensor "
                       "parallelism (hardware not stated)"}), flush=True)
    return 0


# ----------------------------------------------------------------------------- main
def main():
    args = parse_args()
    if args.oracle_full:
        return run_oracle_full(args)
    if args.workload == "p3col":
        world, rank, local = dist_setup(args.gpus)
        return run_p3_column_latency(args, world, rank, local)
    if args.workload == "ln":
        if args.impl != "native":
            raise SystemExit("--impl reference times the MLP workloads only")
        world, rank, local = dist_setup(args.gpus)
        return run_layernorm(args, world, rank, local)
    if args.workload == "attn":
        if args.impl != "native":
            raise SystemExit("--impl reference times the MLP workloads only")
        world, rank, local = dist_setup(args.gpus)
        return run_attention(args, world, rank, local)
    w = workload(args.workload)
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import torch

    device = dist_init(world, local)
    import tensor_sharded_linear_bias_gb300 as tp

    reduce = {"fused": tp.TP_REDUCE_FUSED, "partials": tp.TP_REDUCE_PARTIALS,
              "auto": tp.TP_REDUCE_AUTO, "partials_bf16": tp.TP_REDUCE_PARTIALS_BF16,
              "overlap": tp.TP_REDUCE_OVERLAP}[args.reduce]
    keep_host = (rank == 0 and world == 1 and not args.no_cpu_baseline)
    mb = MlpBench(w, reduce, device, keep_host, sp=args.sp)
    if args.sp:
        args.no_e2e = True

    # ---- device-resident throughput (untraced), then the same steps traced for the roofline
    for _ in range(args.warmup):
        mb.step()
    tp.tp_check_status(mb.ws)
    flush, l2_note = make_flush(device, mb.operand_bytes)
    sampler = ClockSampler(device.index if device.index is not None else 0) if rank == 0 else None
    ms, recs, clocks = timed_then_traced(tp, mb.step, args.steps, world, flush,
                                         args.steps * TRACE_PER_STEP + 16, sampler)
    tp.tp_check_status(mb.ws)
    ms, value = replica_throughput(mb.flops, args.steps, ms, world)
    ms_per_step = ms / args.steps

    # ---- the same steps with L2 left warm between them (only where the timed ones flush it)
    warm = None
    if flush is not None:
        ms_w, value_w = replica_throughput(
            mb.flops, args.steps, time_steps(mb.step, args.steps, world, host_ahead=True), world)
        warm = {"value": value_w, "unit": UNIT, "ms_per_step": ms_w / args.steps,
                "l2": "not flushed: operands stay in L2 from step to step; the steps are "
                      "enqueued behind a sleep kernel, so the host's enqueue time is not in it"}

    # ---- end to end: host inputs in, host results out, every step
    e2e = None
    if not args.no_e2e:
        if flush is None:
            mb.run_e2e(args.warmup)
            ms_e = time_steps(lambda: mb.run_e2e(args.steps), 1, world)
        else:
            for _ in range(args.warmup):
                mb.e2e_step()
            ms_e = time_steps(mb.e2e_step, args.steps, world, flush)
        ms_e, value_e = replica_throughput(mb.flops, args.steps, ms_e, world)
        e2e = {"value": value_e, "unit": UNIT,
               "ms_per_step": ms_e / args.steps, "h2d_bytes_per_step": mb.h2d_bytes,
               "d2h_bytes_per_step": mb.d2h_bytes,
               "mode": ("two copy streams, neighbouring steps' copies overlap compute"
                        if flush is None else "serial per step on one stream, L2 flushed "
                        "before each step outside its events")}
        tp.tp_check_status(mb.ws)

    if rank != 0:
        return 0

    pk = peaks()
    roof, kernels = roofline_from_trace(recs, pk, w.name, clocks=clocks)
    peak, regime, _ = tensor_peak(pk, clocks)
    # the whole step's algorithmic bytes (every launch's operands once, outputs once) per
    # second, cold and warm L2: the HBM view of a latency-bound step (the pages' batch-32 case)
    step_bytes = sum(r["bytes"] for r in recs) / args.steps
    step_hbm = {"bytes_per_step": step_bytes,
                "cold_gbs": step_bytes / (ms / args.steps / 1e3) / 1e9,
                "warm_gbs": (step_bytes / (warm["ms_per_step"] / 1e3) / 1e9) if warm else None,
                "peak": pk["hbm_gbs"], "unit": "GB/s"}

    cpu = None
    if keep_host:
        cpu = cpu_baseline(w, mb.host, args.cpu_seconds)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "tokens": w.tokens, "hidden": w.hidden, "ffn": w.ffn,
                   "tp_degree": w.tp_degree, "reduce": args.reduce,
                   "sequence_parallel": bool(args.sp),
                   "pass": "fwd+bwd" if w.backward else "fwd",
                   "parallelism": "single GPU, all shards on it" if world == 1 else
                   f"{world} independent replicas (no exchange)",
                   "l2": l2_note,
                   "timing": "throughput from untraced steps; per-kernel figures from the "
                             "same number of steps traced with per-launch events"},
        "pct_of_peak": value / peak * 100.0 if w.dtype == "bf16" else None,
        "pct_of_peak_basis": (f"{regime} peak (see roofline.peak_source)" if w.dtype == "bf16"
                              else None),
        "clocks": clocks,
        "e2e": e2e,
        "warm_l2": warm,
        "step_hbm_view": step_hbm,
        "gpu_launches": len(recs),
        "gpu_launches_per_step": len(recs) / args.steps,
        "roofline": roof,
        "kernels": kernels,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
