#!/usr/bin/env python
"""Benchmark: MSDA forward + backward at Deformable-DETR encoder scale on GB300.

One step = one forward and one full backward (zero, accumulate, finish) of
the encoder workload (B=2, Q=S=22223, M=8, D=32, L=4, K=4; synthetic inputs
drawn by scale_deformable_attention_msda_gb300.workloads), with every input
resident in HBM. L2 is flushed (a 256 MiB write) between timed steps, outside
the timed events. Each kernel is bracketed by CUDA events on the launching
stream, so the step time and every kernel's time come from the device clock.

Printed (rank 0, one JSON line): queries/s for the whole job, ms per step,
per-kernel times and HBM fractions, the roofline of the dominant kernel, the
end-to-end number through the public API with host buffers (copies inside the
timed region), the fp64 CPU oracle timed on the host cores as a baseline, and
the SM clocks sampled during the run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--dtype bf16|f32|f16]
                  [--accum fp32_buffer|native|auto|fp16_buffer] [--impl ours|reference]
Under torchrun each rank runs its own replica (weak scaling); the time is the
maximum over ranks. --impl reference times the fp64 CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MSDA fwd+bwd queries/sec at encoder scale; achieved HBM GB/s vs GB300 peak"
UNIT = "queries/s"
FLUSH_BYTES = 256 << 20
FALLBACK_HBM_GBS = 6800.0
# L2 reduction throughput of this machine's GB300 for random 16-byte vector adds,
# GB/s of reduction data, by bytes each group of lanes adds per instruction
# (the 64 MiB footprint rows of profiles/gb300_memory_ceilings.md, recorded
# with a standalone microbenchmark). The backward is bound by this, not by HBM.
RED_CEILING_GBS = {64: 5902.0, 128: 7003.0}


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f32", "f16"])
    ap.add_argument("--accum", default="fp32_buffer", choices=["fp32_buffer", "native", "auto", "fp16_buffer"])
    ap.add_argument("--no-f32-line", action="store_true",
                    help="skip the second timed phase with fp32 storage (the line's f32_encoder)")
    ap.add_argument("--no-accum-lines", action="store_true",
                    help="skip the timed phases of the other 16-bit accumulators (the line's "
                         "accumulator_modes)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the benchmark line, time forward and backward over the "
                         "ablation grid (B=1, bf16: Q x K x L x dispatch order, plus the "
                         "4x4-patch contention workload), one JSON line per point")
    ap.add_argument("--configs", action="store_true",
                    help="instead of the benchmark line, time forward and backward (cold "
                         "and warm L2) on the decoder, encoder and Mask2Former "
                         "configurations and the sweep point Q=5000, K=4, L=4, with the "
                         "fp64 oracle on 1 thread and all cores, "
                         "one JSON line per configuration")
    ap.add_argument("--layer", action="store_true",
                    help="instead of the benchmark line, time the MultiScaleDeformableAttention "
                         "layer (projections + fused-softmax operator, bf16) forward and "
                         "backward on the encoder shape, and the operator's share of it")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be at least 3")
    return a


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


# ------------------------------------------------------------ multi-rank
# Each rank is an independent replica; the only exchange is the timing
# reduction below (no collective on the data path).

def reduce_max(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(device_index=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device_index is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device_index])
        else:
            dist.barrier()


def job_throughput(units_this_rank: float, seconds_this_rank: float, device=None) -> tuple:
    """(whole-job units per second, max seconds over ranks, total units)."""
    total = reduce_sum(units_this_rank, device)
    slowest = reduce_max(seconds_this_rank, device)
    return total / slowest, slowest, total


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 100 ms while the GPU works (read-only)."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, uuid=None):
        self.lines = []
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if uuid:
            cmd.insert(1, f"--id={uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "util": float(f[4]),
                             "reasons": [r for r, v in zip(self.REASONS, f[5:9]) if v == "Active"]})
            except ValueError:
                continue
        if not rows:
            return None
        busy = [r for r in rows if r["util"] > 0] or rows
        reasons = sorted({x for r in busy for x in r["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in busy),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(busy)}


def gather_roofline(samples: int, D: int, elt: int, forward_ms: float, sm_mhz: float,
                    n_sms: int) -> dict:
    """The forward's own bound: L1 data-pipe wavefronts. Every sample gathers
    4 corner vectors of D*elt bytes, each in ceil(D*elt/128) 128-byte lines
    (rows are D*elt-aligned), one wavefront per line; the pipe retires about
    one wavefront per cycle per SM (ncu: 80 % of its peak at 0.8 per cycle)."""
    lines = -(-D * elt // 128)
    wavefronts = 4 * samples * lines
    achieved = wavefronts / (forward_ms * 1e-3) / 1e9
    peak = n_sms * sm_mhz * 1e6 / 1e9
    return {"kernel": "msda_forward_kernel", "bound": "l1_wavefronts",
            "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "G wavefronts/s",
            "frac": round(achieved / peak, 4), "wavefronts_per_launch": wavefronts,
            "model": "one L1 data-pipe wavefront per 128-byte line of each gathered corner "
                     "vector (4 per sample); peak one wavefront per cycle per SM x SMs x "
                     "median SM clock under load"}


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


ACCUM_MODES = {"fp32_buffer": lambda b: b.MSDA_ACC_FP32_BUFFER,
               "native": lambda b: b.MSDA_ACC_NATIVE,
               "auto": lambda b: b.MSDA_ACC_AUTO,
               "fp16_buffer": lambda b: b.MSDA_ACC_FP16_BUFFER}


# Kernels one bench step launches, by the accumulator the backward resolved to:
# forward, zero (grad_value or workspace), accumulate, finish (16-bit data with
# the fp32 workspace); fp32 data and native 16-bit adds need no finish; the
# fp16 workspace's one call: zero + maxima, accumulate, finish.
LAUNCHES_PER_STEP = {"fp32_buffer": 4, "native": 3, "fp16_buffer": 4, "f32": 3}


def arithmetic_dtype(storage: str, resolved: str) -> str:
    """The type the step's arithmetic and grad_value accumulation run in:
    fp32 for fp32 storage and for 16-bit storage with the fp32 workspace; fp16
    for bf16 storage with the scaled fp16 workspace; the 16-bit type itself
    when grad_value is accumulated natively."""
    if storage == "f32" or resolved == "fp32_buffer":
        return "f32"
    return "f16" if resolved == "fp16_buffer" else storage


def resolved_accumulator(storage: str, mode: str, workspace_bytes: int) -> str:
    """What a backward call of `mode` accumulates grad_value in: fp32 storage
    adds fp32; the scaled fp16 workspace applies to bf16 data only (others add
    natively); AUTO and the fp32 buffer resolve to the workspace when the
    library asks for one."""
    if storage == "f32":
        return "fp32_buffer"
    if mode == "fp16_buffer":
        return "fp16_buffer" if storage == "bf16" else "native"
    return "fp32_buffer" if workspace_bytes > 0 else "native"

KERNEL_SOURCES = {"msda_forward_kernel": ("msda_common.cuh", "msda_forward.cu"),
                  "msda_backward_kernel": ("msda_common.cuh", "msda_backward.cuh")}


def kernel_source_hash(kernel: str) -> str:
    """sha256 prefix of the code of the source files that define `kernel`:
    comments and runs of whitespace are dropped first, so that editing a
    comment does not retire the ncu counters taken on the same code."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "scale_deformable_attention_msda_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        text = open(os.path.join(csrc, name), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(name.encode())
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


# The ncu summary that holds a kernel's counters for the bench's encoder run,
# by (kernel, storage dtype, accumulator): each is a different instantiation,
# and a run with no summary of its own reports no traffic.
PROFILE_FILES = {
    ("msda_forward_kernel", "bf16", "fp32_buffer"): "msda_forward_kernel_encoder.md",
    ("msda_forward_kernel", "bf16", "native"): "msda_forward_kernel_encoder.md",
    ("msda_backward_kernel", "bf16", "fp32_buffer"): "msda_backward_kernel_encoder.md",
    ("msda_backward_kernel", "bf16", "native"): "msda_backward_kernel_native_encoder.md",
    ("msda_forward_kernel", "bf16", "fp16_buffer"): "msda_forward_kernel_encoder.md",
    ("msda_backward_kernel", "bf16", "fp16_buffer"): "msda_backward_kernel_fp16_buffer_encoder.md",
    ("msda_forward_kernel", "f32", "fp32_buffer"): "msda_kernels_f32_encoder.md",
    ("msda_backward_kernel", "f32", "fp32_buffer"): "msda_kernels_f32_encoder.md",
}


def profiled_traffic(kernel: str, dtype: str = "bf16", accum: str = "fp32_buffer"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None.

    The summary (PROFILE_FILES) carries a line
    `traffic_bytes_per_launch: N  source_sha256: H`; the figure counts only
    while the kernel's sources still hash to H (else the kernel has changed
    since the counters were taken)."""
    import re
    name = PROFILE_FILES.get((kernel, dtype, accum))
    if name is None:
        return None
    path = os.path.join(ROOT, "profiles", name)
    try:
        text = open(path).read()
    except OSError:
        return None
    # a summary of several kernels qualifies each line with the kernel's name
    m = (re.search(r"traffic_bytes_per_launch \(" + re.escape(kernel) +
                   r"\):\s*(\d+)\s+source_sha256:\s*([0-9a-f]+)", text) or
         re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_sha256:\s*([0-9a-f]+)", text))
    if not m or kernel not in KERNEL_SOURCES:
        return None
    return int(m.group(1)) if m.group(2) == kernel_source_hash(kernel) else None


def issued_atomic_rows(p, block: int):
    """Per level, the vector adds the backward issues per launch: every
    distinct in-map corner row among the corners of each aligned block of
    `block` consecutive samples of one query-head (the kernel sums the
    weights of corners that share a row there and adds once), counted with
    numpy from the inputs, for the atomic roofline only. A block is counted
    under the level of its first sample (one level exactly when K is a
    multiple of `block`)."""
    import numpy as np
    loc = np.asarray(p["loc"], dtype=np.float64)                 # (B, Q, M, L, K, 2)
    H = np.asarray(p["shapes"])[:, 0][None, None, None, :, None]
    W = np.asarray(p["shapes"])[:, 1][None, None, None, :, None]
    start = np.asarray(p["starts"])[None, None, None, :, None]
    x0 = np.floor(loc[..., 0] * W - 0.5).astype(np.int64)
    y0 = np.floor(loc[..., 1] * H - 0.5).astype(np.int64)
    rows = []
    for dy in (0, 1):
        for dx in (0, 1):
            xx, yy = x0 + dx, y0 + dy
            ok = (xx >= 0) & (xx < W) & (yy >= 0) & (yy < H)
            rows.append(np.where(ok, start + yy * W + xx, -1))
    B, Q, M, L, K = x0.shape
    r = np.stack(rows, -1).reshape(B * Q * M, L * K, 4)
    n_blocks = (L * K + block - 1) // block
    pad = n_blocks * block - L * K
    if pad:
        r = np.concatenate([r, np.full((B * Q * M, pad, 4), -1, np.int64)], axis=1)
    r = np.sort(r.reshape(B * Q * M, n_blocks, block * 4), axis=-1)
    first = np.ones(r.shape, dtype=bool)
    first[..., 1:] = r[..., 1:] != r[..., :-1]
    per_block = np.count_nonzero(first & (r >= 0), axis=(0, 2))   # (n_blocks,)
    level_of_block = (np.arange(n_blocks) * block) // K
    return [int(per_block[level_of_block == l].sum()) for l in range(L)]


# ---------------------------------------------------------- CPU baseline

def cpu_baseline(p, seconds: float = 10.0, max_reps: int = 20, nthreads: int = 0):
    """The fp64 oracle, as it stands, on the host cores: forward + backward of
    the full workload, repeated for about `seconds`."""
    import numpy as np
    import oracle
    oracle.build()
    f64 = {k: np.ascontiguousarray(p[k], dtype=np.float64)
           for k in ("value", "loc", "attn", "grad_out")}
    B, Q = f64["loc"].shape[:2]
    times = []
    t_end = time.perf_counter() + seconds
    while len(times) < max_reps and (len(times) < 2 or time.perf_counter() < t_end):
        t0 = time.perf_counter()
        oracle.forward(f64["value"], p["shapes"], p["starts"], f64["loc"], f64["attn"],
                       nthreads=nthreads)
        oracle.backward(f64["value"], p["shapes"], p["starts"], f64["loc"], f64["attn"],
                        f64["grad_out"], nthreads=nthreads)
        times.append(time.perf_counter() - t0)
    t = statistics.median(times)
    return {"value": B * Q / t, "unit": UNIT, "cores": nthreads or (os.cpu_count() or 1),
            "kind": "oracle",
            "sample": f"full workload (B={B}, Q={Q}), forward+backward in fp64, "
                      f"median of {len(times)} repetitions"}


# ------------------------------------------------------------- our arm

def run_e2e(args, binding, torch, p, w, tdt, accum, shapes, starts, comp, dev):
    """Throughput through msda_forward + msda_backward with host buffers
    (see the caller): K pipelined steps, copies included."""
    names_in, names_out = ("value", "loc", "attn", "grad_out"), ("out", "gv", "gl", "ga")
    host_in = {k: torch.tensor(p[k], dtype=torch.float64).to(tdt).pin_memory() for k in names_in}
    sets = []
    for _ in range(2):
        d = {k: torch.empty(t.shape, dtype=tdt, device=dev) for k, t in host_in.items()}
        bb = binding.BackwardBuffers(d["value"], d["loc"], d["attn"], accum)
        o = {"out": torch.empty((w.B, w.Q, w.M * w.D), dtype=tdt, device=dev),
             "gv": bb.grad_value, "gl": bb.grad_sampling_locations,
             "ga": bb.grad_attention_weights}
        h = {k: torch.empty(t.shape, dtype=tdt).pin_memory() for k, t in o.items()}
        sets.append({"in": d, "buf": bb, "out": o, "host_out": h})
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in sets[0]["out"].values())
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of set b copied
    ev_done = [torch.cuda.Event() for _ in range(2)]   # kernels of set b finished
    ev_read = [torch.cuda.Event() for _ in range(2)]   # results of set b copied out

    def run(n):
        for i in range(n):
            b, st = i & 1, sets[i & 1]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_done[b])
                for k in names_in:
                    st["in"][k].copy_(host_in[k], non_blocking=True)
                ev_in[b].record(s_in)
            comp.wait_event(ev_in[b])
            if i >= 2:
                comp.wait_event(ev_read[b])
            d = st["in"]
            binding.msda_forward(d["value"], shapes, starts, d["loc"], d["attn"],
                                 out=st["out"]["out"], stream=comp)
            binding.msda_backward(d["value"], shapes, starts, d["loc"], d["attn"], d["grad_out"],
                                  accum=accum, grad_value=st["buf"].grad_value,
                                  grad_sampling_locations=st["buf"].grad_sampling_locations,
                                  grad_attention_weights=st["buf"].grad_attention_weights,
                                  workspace=st["buf"].workspace, stream=comp)
            ev_done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                for k in names_out:
                    st["host_out"][k].copy_(st["out"][k], non_blocking=True)
                ev_read[b].record(s_out)
        comp.wait_event(ev_read[(n - 1) & 1])
        if n >= 2:
            comp.wait_event(ev_read[(n - 2) & 1])

    run(3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_event(e0)
    run(args.e2e_steps)
    e1.record(comp)
    torch.cuda.synchronize()
    total_s = e0.elapsed_time(e1) / 1e3
    qps, slowest_s, _ = job_throughput(w.B * w.Q * args.e2e_steps, total_s, dev)
    return {"value": round(qps, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
            "ms_per_step": round(slowest_s * 1e3 / args.e2e_steps, 4),
            "pipeline": "H2D of step i+1 and D2H of step i-1 overlap step i's kernels "
                        "(two copy streams, two buffer sets)"}



def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    from scale_deformable_attention_msda_gb300 import binding, build, workloads as wl

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or not os.path.exists(build.LIBRARY):
        build.build()
    barrier(local_rank)
    binding.lib()

    accum = ACCUM_MODES[args.accum](binding)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    names = ("forward", "zero", "backward", "finish")

    def setup(dtype):
        """Operands of the encoder workload in `dtype`, resident in HBM."""
        tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "f16": torch.float16}[dtype]
        w = wl.encoder(dtype, variant=rank)
        p = wl.make_inputs(w)

        def up(a):
            return torch.tensor(a, dtype=torch.float64).to(tdt).to(dev)

        return {"w": w, "p": p, "tdt": tdt, "value": up(p["value"]), "loc": up(p["loc"]),
                "attn": up(p["attn"]), "gout": up(p["grad_out"]),
                "shapes": torch.tensor(p["shapes"], device=dev),
                "starts": torch.tensor(p["starts"], device=dev)}

    def timed(op, acc, acc_name, steps, warmup):
        """Warm-up, then `steps` timed steps (L2 flushed before each, outside
        the events); per-kernel event times in ms, and the accumulator the
        backward resolved to. The scaled fp16 workspace is taken only by the
        one-call msda_backward: its "backward" time then covers its prepare
        pass, the adds and its finish pass, and "zero" and "finish" are empty."""
        out = torch.empty((op["w"].B, op["w"].Q, op["w"].M * op["w"].D), dtype=op["tdt"], device=dev)
        buf = binding.BackwardBuffers(op["value"], op["loc"], op["attn"], acc)
        a = (op["value"], op["shapes"], op["starts"], op["loc"], op["attn"])
        storage = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[op["tdt"]]
        resolved = resolved_accumulator(storage, acc_name, buf.workspace_bytes)
        one_call = resolved == "fp16_buffer"

        def step(ev=None):
            if ev:
                ev[0].record(stream)
            binding.msda_forward(*a, out=out)
            if ev:
                ev[1].record(stream)
            if not one_call:
                binding.msda_backward_zero(buf, op["tdt"])
            if ev:
                ev[2].record(stream)
            if one_call:
                binding.msda_backward(*a, op["gout"], accum=acc, grad_value=buf.grad_value,
                                      grad_sampling_locations=buf.grad_sampling_locations,
                                      grad_attention_weights=buf.grad_attention_weights,
                                      workspace=buf.workspace)
            else:
                binding.msda_backward_accumulate(*a, op["gout"], buf)
            if ev:
                ev[3].record(stream)
            if not one_call:
                binding.msda_backward_finish(buf, op["tdt"])
            if ev:
                ev[4].record(stream)

        for _ in range(warmup):
            flush.fill_(1)
            step()
        torch.cuda.synchronize()
        barrier(local_rank)
        torch.cuda.synchronize()
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
        for i in range(steps):
            flush.fill_(i & 0xff)
            step(evs[i])
        torch.cuda.synchronize()
        barrier(local_rank)
        torch.cuda.synchronize()
        per = {n: [evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)]
               for j, n in enumerate(names)}
        step_ms = [evs[i][0].elapsed_time(evs[i][4]) for i in range(steps)]
        return per, step_ms, resolved

    peak, peak_kind = measured_hbm_peak()
    kernel_name = {"forward": "msda_forward_kernel", "backward": "msda_backward_kernel"}

    def roofline_of(w, mean, dtype, acc_name):
        """Roofline of the dominant kernel from its event times."""
        cb = wl.compulsory_bytes(w)
        algo = {"forward": cb["forward"], "backward": cb["backward"]}
        dominant = max(("forward", "backward"), key=lambda n: mean[n])
        achieved = algo[dominant] / (mean[dominant] * 1e-3) / 1e9
        traffic = profiled_traffic(kernel_name[dominant], dtype, acc_name)
        roof = {"bound": "hbm", "kernel": kernel_name[dominant], "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": traffic, "algorithmic_bytes": algo[dominant],
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                else "fallback 6.8 TB/s",
                "traffic_source": (f"stored ncu figure: profiles/{PROFILE_FILES[(kernel_name[dominant], dtype, acc_name)]}"
                                   " (dram__bytes_read.sum + dram__bytes_write.sum per launch, "
                                   "valid while the kernel sources hash as recorded there)")
                if traffic is not None else "none: no ncu summary of this kernel's current code"}
        if acc_name == "fp16_buffer" and dominant == "backward":
            roof["duration_covers"] = ("the one msda_backward call: zero + maxima, the kernel, "
                                       "finish")
        kernels = {}
        for n in names:
            k = {"ms": round(mean[n], 5)}
            if n in algo:
                gbs = algo[n] / (mean[n] * 1e-3) / 1e9
                k.update(algorithmic_bytes=algo[n], gbs=round(gbs, 1), hbm_frac=round(gbs / peak, 4))
            kernels[n] = k
        return roof, kernels, algo

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid) if rank == 0 else None

    op = setup(args.dtype)
    w, p = op["w"], op["p"]
    tdt, value, loc, attn, gout = op["tdt"], op["value"], op["loc"], op["attn"], op["gout"]
    shapes, starts = op["shapes"], op["starts"]
    per, step_ms, acc_name = timed(op, accum, args.accum, args.steps, args.warmup)
    total_s = sum(step_ms) / 1e3
    qps, slowest_s, total_units = job_throughput(w.B * w.Q * args.steps, total_s, dev)
    ms_per_step = slowest_s * 1e3 / args.steps
    mean = {n: statistics.fmean(v) for n, v in per.items()}

    # ---- the same step with fp32 storage (both precisions of the encoder
    # configuration on one line); fewer steps
    f32_line = None
    if args.dtype != "f32" and not args.no_f32_line:
        op32 = setup("f32")
        steps32 = max(1, min(args.steps, 500))
        per32, step32, _ = timed(op32, binding.MSDA_ACC_FP32_BUFFER, "fp32_buffer", steps32,
                                 args.warmup)
        qps32, slow32, _ = job_throughput(op32["w"].B * op32["w"].Q * steps32, sum(step32) / 1e3, dev)
        mean32 = {n: statistics.fmean(v) for n, v in per32.items()}
        roof32, kern32, _ = roofline_of(op32["w"], mean32, "f32", "fp32_buffer")
        f32_line = {"storage_dtype": "f32", "dtype": "f32", "grad_value_accumulator": "fp32 atomics",
                    "value": round(qps32, 1), "unit": UNIT, "steps": steps32,
                    "ms_per_step": round(slow32 * 1e3 / steps32, 5), "kernels": kern32,
                    "roofline": roof32, "gpu_launches": 3 * steps32,
                    "step": "msda_forward + msda_backward (zero, accumulate; fp32 data needs no "
                            "finish pass)"}
        del op32

    # ---- the same bf16 step with the other grad_value accumulators (the
    # accumulator switch measured in one run); fewer steps
    modes = None
    if args.dtype == "bf16" and not args.no_accum_lines:
        modes = {}
        for name in ("fp32_buffer", "native", "fp16_buffer"):
            if name == acc_name:
                continue
            steps_m = max(1, min(args.steps, 500))
            per_m, step_m, res_m = timed(op, ACCUM_MODES[name](binding), name, steps_m, args.warmup)
            qps_m, slow_m, _ = job_throughput(w.B * w.Q * steps_m, sum(step_m) / 1e3, dev)
            mean_m = {n: statistics.fmean(v) for n, v in per_m.items()}
            modes[name] = {"value": round(qps_m, 1), "unit": UNIT, "steps": steps_m,
                           "ms_per_step": round(slow_m * 1e3 / steps_m, 5),
                           "dtype": arithmetic_dtype("bf16", res_m),
                           "accumulator_resolved": res_m,
                           "kernels_ms": {n: round(mean_m[n], 5) for n in names},
                           "gpu_launches": LAUNCHES_PER_STEP[res_m] * steps_m}
        modes["note"] = ("same encoder step and inputs, bf16 storage; grad_value error against "
                         "the fp64 oracle is measured by the GPU tests, not here; fp16_buffer's "
                         "backward is one msda_backward call (zero and finish inside it)")
    clocks = sampler.stop() if sampler else None
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    gather = gather_roofline(w.samples, w.D, 2 if args.dtype != "f32" else 4, mean["forward"],
                             sm_mhz, n_sms)
    if f32_line is not None:
        f32_line["gather_roofline"] = gather_roofline(w.samples, w.D, 4,
                                                      f32_line["kernels"]["forward"]["ms"],
                                                      sm_mhz, n_sms)

    # ---- end to end through the public API, host buffers, copies timed.
    # Pipelined as a training input pipeline runs: step i's inputs go in on
    # one copy stream while step i-1 computes, step i-1's results come out on
    # another while step i computes, and two device buffer sets alternate
    # (events order every reuse). Every step copies its four inputs from
    # pinned host memory and its four results back; the timed region spans
    # all copies and kernels of all steps. No L2 flush: each step's inputs
    # arrive fresh by DMA.
    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, binding, torch, p, w, tdt, accum, shapes, starts, stream, dev)

    # ---- roofline of the dominant kernel
    roofline, kernels, _ = roofline_of(w, mean, args.dtype, acc_name)
    for n in names:
        kernels[n]["launches"] = args.steps
    cb = wl.compulsory_bytes(w)
    step_bytes = cb["forward"] + cb["backward"]
    # Atomic bytes the backward adds per launch (the distinct corner rows it
    # issues, at the target's element size) and the bytes one add instruction
    # covers per query-head. fp32 data and 16-bit data with the fp32
    # workspace use D/4 lanes of 4 fp32 channels while D/4 fits a warp (4 D
    # bytes per query-head; 16-byte lanes with 16-bit data write 2 D, in two
    # halves); native 16-bit mode and the fp16 workspace use D/8 lanes of 8
    # channels (2 D bytes).
    f32_target = acc_name == "fp32_buffer"
    narrow = f32_target and w.D // 4 <= 32
    lanes = w.D // 4 if narrow else w.D // 8
    acc_bytes = 4 if f32_target else 2
    rows_per_level = issued_atomic_rows(p, min(4, lanes))
    red_bytes = sum(rows_per_level) * w.D * acc_bytes
    group = (4 if narrow else 2) * w.D
    ceiling = RED_CEILING_GBS[128 if group >= 128 else 64]
    red_gbs = red_bytes / (mean["backward"] * 1e-3) / 1e9
    atomic_roofline = {"kernel": "msda_backward_kernel", "bound": "l2_reduction",
                       "achieved": round(red_gbs, 1), "peak": ceiling, "unit": "GB/s",
                       "frac": round(red_gbs / ceiling, 4), "atomic_bytes": red_bytes,
                       "atomic_bytes_unmerged": w.samples * 4 * w.D * acc_bytes,
                       "atomic_bytes_per_level": [n * w.D * acc_bytes for n in rows_per_level],
                       "peak_source": "measured red.global.add.v4 throughput, "
                                      f"{group}-byte groups (profiles/gb300_memory_ceilings.md)"}
    if acc_name == "fp16_buffer":
        atomic_roofline["duration_covers"] = "the one msda_backward call (prepare and finish passes too)"

    result = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(p)
        launches_per_step = LAUNCHES_PER_STEP["f32" if args.dtype == "f32" else acc_name]
        result = {
            "metric": METRIC, "value": round(qps, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": arithmetic_dtype(args.dtype, acc_name), "data": "synthetic",
            "config": {"workload": "deformable-detr encoder: B=2, Q=S=22223, M=8, D=32, L=4, K=4, "
                                   "levels (100,167),(50,84),(25,42),(13,21)",
                       "storage_dtype": args.dtype, "grad_value_accumulator": args.accum,
                       "accumulator_resolved": acc_name,
                       "global_batch": w.B * world, "queries_per_step": w.B * w.Q * world,
                       "parallelism": f"replicas x{world}" if world > 1 else "single gpu",
                       "l2": "flushed between timed steps (256 MiB write, outside the events)",
                       "step": "msda_forward + msda_backward (zero, accumulate, finish)"
                               if acc_name != "fp16_buffer" else
                               "msda_forward + msda_backward (one call: zero + maxima, "
                               "accumulate, finish)"},
            "step_hbm": {"compulsory_bytes": step_bytes,
                         "gbs": round(step_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                         "frac": round(step_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4)},
            "kernels": kernels,
            "roofline": roofline,
            "f32_encoder": f32_line,
            "accumulator_modes": modes,
            "atomic_roofline": atomic_roofline,
            "gather_roofline": gather,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "kernel_source_sha256": {k: kernel_source_hash(k) for k in KERNEL_SOURCES},
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        barrier(local_rank)
        dist.destroy_process_group()
    return result


# ------------------------------------------------------------ the sweep

def run_sweep(args):
    """Median forward / backward times (L2 flushed before each timed call) over
    the ablation grid: Q in {5000, 10000, 22223}, K in {2, 4, 8}, L in 1..4 of
    the encoder levels, linear / Morton / Hilbert dispatch, and the
    high-contention variant (every sample inside a 4x4-pixel patch per level).
    The backward is one msda_backward call into preallocated buffers (its
    zero, accumulate and finish steps), so every accumulator runs the same way."""
    import numpy as np
    import torch

    from scale_deformable_attention_msda_gb300 import binding, build, workloads as wl

    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "f16": torch.float16}[args.dtype]
    accum = ACCUM_MODES[args.accum](binding)
    reps = max(5, min(args.steps, 30))

    def time_point(w, order_kind):
        p = wl.make_inputs(w.with_dtype(args.dtype))
        up = lambda a: torch.tensor(a, dtype=torch.float64).to(tdt).to(dev)  # noqa: E731
        value, loc, attn, g = up(p["value"]), up(p["loc"]), up(p["attn"]), up(p["grad_out"])
        shapes = torch.tensor(p["shapes"], device=dev)
        starts = torch.tensor(p["starts"], device=dev)
        order = None
        if order_kind != "linear":
            order = torch.tensor(wl.query_order(w, order_kind), device=dev)
        out = torch.empty((w.B, w.Q, w.M * w.D), dtype=tdt, device=dev)
        buf = binding.BackwardBuffers(value, loc, attn, accum)
        tf, tb = [], []
        for i in range(reps + 3):
            flush.fill_(i & 0xff)
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            binding.msda_forward(value, shapes, starts, loc, attn, query_order=order, out=out)
            e[1].record()
            binding.msda_backward(value, shapes, starts, loc, attn, g, accum=accum,
                                  query_order=order, grad_value=buf.grad_value,
                                  grad_sampling_locations=buf.grad_sampling_locations,
                                  grad_attention_weights=buf.grad_attention_weights,
                                  workspace=buf.workspace)
            e[2].record()
            torch.cuda.synchronize()
            if i >= 3:
                tf.append(e[0].elapsed_time(e[1]))
                tb.append(e[1].elapsed_time(e[2]))
        cb = wl.compulsory_bytes(w.with_dtype(args.dtype))
        f, b = float(np.median(tf)), float(np.median(tb))
        return {"workload": w.name, "Q": w.Q, "K": w.K, "L": w.L, "order": order_kind,
                "dtype": args.dtype, "accum": args.accum, "forward_us": round(f * 1e3, 2),
                "backward_us": round(b * 1e3, 2),
                "queries_per_s": round(w.B * w.Q / ((f + b) * 1e-3), 1),
                "forward_hbm_frac": round(cb["forward"] / (f * 1e-3) / 1e9 / measured_hbm_peak()[0], 4),
                "backward_hbm_frac": round(cb["backward"] / (b * 1e-3) / 1e9 / measured_hbm_peak()[0], 4)}

    for w in wl.sweep_grid():
        for kind in ("linear", "morton", "hilbert"):
            print(json.dumps(time_point(w, kind)), flush=True)
    for Q in (5000, 10000, 22223):
        print(json.dumps(time_point(wl.sweep(Q, 4, 4, contention=True), "linear")), flush=True)


def run_configs(args):
    """Per configuration: median forward and backward call times (msda_forward,
    msda_backward = zero + accumulate + finish) over 50 calls after 10
    warm-up, cold (L2 flushed before each call) and warm (not flushed); their
    HBM fractions; and the fp64 oracle on the host, one thread and all cores."""
    import numpy as np
    import torch

    import oracle
    from scale_deformable_attention_msda_gb300 import binding, build, workloads as wl

    build.build()
    oracle.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    peak = measured_hbm_peak()[0]
    plan = [(wl.decoder, "f32", "fp32_buffer"), (wl.decoder, "bf16", "fp32_buffer"),
            (wl.decoder, "bf16", "native"), (wl.decoder, "bf16", "auto"),
            (wl.encoder, "f32", "fp32_buffer"), (wl.encoder, "bf16", "fp32_buffer"),
            (wl.encoder, "bf16", "native"), (wl.encoder, "bf16", "auto"),
            (wl.decoder, "bf16", "fp16_buffer"), (wl.encoder, "bf16", "fp16_buffer"),
            (wl.mask2former, "bf16", "fp32_buffer"), (wl.mask2former, "bf16", "native"),
            (wl.mask2former, "bf16", "fp16_buffer"),
            (lambda dt: wl.sweep(5000, 4, 4, dtype=dt), "bf16", "fp32_buffer")]
    for make, dtype, acc_name in plan:
        w = make(dtype)
        p = wl.make_inputs(w)
        tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "f16": torch.float16}[dtype]
        accum = ACCUM_MODES[acc_name](binding)
        up = lambda a: torch.tensor(a, dtype=torch.float64).to(tdt).to(dev)  # noqa: E731
        value, loc, attn, g = up(p["value"]), up(p["loc"]), up(p["attn"]), up(p["grad_out"])
        shapes = torch.tensor(p["shapes"], device=dev)
        starts = torch.tensor(p["starts"], device=dev)
        out = torch.empty((w.B, w.Q, w.M * w.D), dtype=tdt, device=dev)
        buf = binding.BackwardBuffers(value, loc, attn, accum)

        def fwd():
            binding.msda_forward(value, shapes, starts, loc, attn, out=out)

        def bwd():
            binding.msda_backward(value, shapes, starts, loc, attn, g, accum=accum,
                                  grad_value=buf.grad_value,
                                  grad_sampling_locations=buf.grad_sampling_locations,
                                  grad_attention_weights=buf.grad_attention_weights,
                                  workspace=buf.workspace)

        def median_us(fn, cold):
            ts = []
            for i in range(60):
                if cold:
                    flush.fill_(i & 0xff)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                if i >= 10:
                    ts.append(a.elapsed_time(b) * 1e3)
            return float(np.median(ts))

        t = {f"{n}_{c}_us": round(median_us(fn, c == "cold"), 2)
             for n, fn in (("forward", fwd), ("backward", bwd)) for c in ("cold", "warm")}
        cb = wl.compulsory_bytes(w)
        f64 = {k: np.ascontiguousarray(p[k], dtype=np.float64)
               for k in ("value", "loc", "attn", "grad_out")}

        def oracle_s(nthreads):
            r = {}
            for name, fn in (("forward", lambda: oracle.forward(
                                 f64["value"], p["shapes"], p["starts"], f64["loc"], f64["attn"],
                                 nthreads=nthreads)),
                             ("backward", lambda: oracle.backward(
                                 f64["value"], p["shapes"], p["starts"], f64["loc"], f64["attn"],
                                 f64["grad_out"], nthreads=nthreads))):
                ts = []
                while len(ts) < 3 and sum(ts) < 20.0:
                    t0 = time.perf_counter()
                    fn()
                    ts.append(time.perf_counter() - t0)
                r[name] = float(np.median(ts))
            return r

        one, allc = oracle_s(1), oracle_s(0)
        q = w.B * w.Q
        print(json.dumps({
            "config": w.name, "dtype": dtype, "accum": acc_name if dtype != "f32" else "fp32",
            "accum_resolved": resolved_accumulator(dtype, acc_name, buf.workspace_bytes)
                              if dtype != "f32" else "fp32",
            "B": w.B, "Q": w.Q, "S": w.S, "samples": w.samples, **t,
            "queries_per_s_cold": round(q / ((t["forward_cold_us"] + t["backward_cold_us"]) * 1e-6), 1),
            "forward_hbm_frac_cold": round(cb["forward"] / (t["forward_cold_us"] * 1e-6) / 1e9 / peak, 4),
            "backward_hbm_frac_cold": round(cb["backward"] / (t["backward_cold_us"] * 1e-6) / 1e9 / peak, 4),
            "oracle_1_thread_queries_per_s": round(q / (one["forward"] + one["backward"]), 1),
            "oracle_all_cores_queries_per_s": round(q / (allc["forward"] + allc["backward"]), 1),
            "oracle_cores": os.cpu_count() or 1}), flush=True)


# ------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 CPU oracle, as it stands, timed on the host cores."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    import numpy as np
    import oracle
    from scale_deformable_attention_msda_gb300 import workloads as wl

    oracle.build()
    w = wl.encoder(args.dtype)
    p = wl.make_inputs(w)
    f64 = {k: np.ascontiguousarray(p[k], dtype=np.float64) for k in ("value", "loc", "attn", "grad_out")}

    def step(n):
        oracle.forward(f64["value"], p["shapes"], p["starts"], f64["loc"][:, :n], f64["attn"][:, :n])
        oracle.backward(f64["value"], p["shapes"], p["starts"], f64["loc"][:, :n],
                        f64["attn"][:, :n], f64["grad_out"][:, :n])

    # size each step so that warmup + steps take about 90 s in all
    t0 = time.perf_counter()
    step(2048)
    t = time.perf_counter() - t0
    budget = 90.0 / (args.steps + args.warmup)
    n = int(min(w.Q, max(256, 2048 * budget / max(t, 1e-6))))
    for _ in range(args.warmup):
        step(n)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step(n)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    qps = w.B * n * args.steps / total
    cores = os.cpu_count() or 1
    result = {
        "impl": "reference", "metric": METRIC, "value": round(qps, 1), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total * 1e3 / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "deformable-detr encoder: B=2, Q=S=22223, M=8, D=32, L=4, K=4",
                   "sample_queries_per_batch": n, "storage_dtype": args.dtype},
        "cpu_baseline": {"value": round(qps, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {n} queries of each of the B={w.B} batches per step, "
                                   "forward+backward in fp64 against the full value tensor"},
        "e2e": {"value": round(qps, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(result), flush=True)
    return result


def run_layer(args):
    """The layer around the operator: MultiScaleDeformableAttention (dim 256,
    8 heads, 4 levels, 4 points; its four projections are cuBLAS matmuls) in
    bf16 on the encoder shape, forward + backward from a given output
    gradient, L2 flushed before each step; and, on the same operands, the
    operator alone (msda_forward_softmax + msda_backward_softmax)."""
    import numpy as np
    import torch

    from scale_deformable_attention_msda_gb300 import binding, build, layer as lay, workloads as wl

    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    w = wl.encoder("bf16")
    dim = w.M * w.D
    rng = np.random.Generator(np.random.PCG64(77))
    dt = torch.bfloat16
    net = lay.MultiScaleDeformableAttention(dim, w.M, w.L, w.K).to(dev, dt)
    query = torch.tensor(rng.standard_normal((w.B, w.Q, dim)), dtype=dt, device=dev).requires_grad_()
    value = torch.tensor(rng.standard_normal((w.B, w.S, dim)), dtype=dt, device=dev).requires_grad_()
    ref = torch.tensor(wl.reference_points(w, rng), dtype=torch.float32, device=dev)
    shapes = torch.tensor(wl.spatial_shapes(w.levels), device=dev)
    starts = torch.tensor(wl.level_start_index(w.levels), device=dev)
    gout = torch.tensor(rng.standard_normal((w.B, w.Q, dim)), dtype=dt, device=dev)

    def layer_step():
        net.zero_grad(set_to_none=True)
        query.grad = value.grad = None
        net(query, ref, value, shapes, starts).backward(gout)

    # the operator's operands, as the layer builds them
    with torch.no_grad():
        v = net.value_proj(value).view(w.B, w.S, w.M, w.D).contiguous()
        off = net.sampling_offsets(query).view(w.B, w.Q, w.M, w.L, w.K, 2)
        logits = net.attention_weights(query).view(w.B, w.Q, w.M, w.L, w.K).contiguous()
        wh = shapes.flip(-1).to(off.dtype)
        loc = (ref[:, :, None, None, None, :].to(off.dtype) +
               off / wh[None, None, None, :, None, :]).contiguous()
    g_op = torch.tensor(rng.standard_normal((w.B, w.Q, dim)), dtype=dt, device=dev)
    buf = binding.BackwardBuffers(v, loc, logits, binding.MSDA_ACC_FP32_BUFFER)
    out = torch.empty((w.B, w.Q, dim), dtype=dt, device=dev)

    def op_step():
        binding.msda_forward(v, shapes, starts, loc, logits, out=out, softmax=True)
        binding.msda_backward(v, shapes, starts, loc, logits, g_op, softmax=True,
                              grad_value=buf.grad_value,
                              grad_sampling_locations=buf.grad_sampling_locations,
                              grad_attention_weights=buf.grad_attention_weights,
                              workspace=buf.workspace)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for i in range(min(args.steps, 200)):
            flush.fill_(i & 255)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ts.sort()
        return ts[len(ts) // 2]

    layer_ms, op_ms = timed(layer_step), timed(op_step)
    print(json.dumps({
        "mode": "layer", "workload": f"MultiScaleDeformableAttention(dim={dim}, heads={w.M}, "
                                     f"levels={w.L}, points={w.K}) on the encoder shape "
                                     f"B={w.B}, Q=S={w.Q}",
        "dtype": "bf16", "steps": min(args.steps, 200), "warmup": args.warmup,
        "layer_fwd_bwd_ms": round(layer_ms, 4), "operator_fwd_bwd_ms": round(op_ms, 4),
        "operator_share": round(op_ms / layer_ms, 3),
        "layer_queries_per_s": round(w.B * w.Q / (layer_ms * 1e-3), 1),
        "l2": "flushed before each step (256 MiB write, outside the events)",
        "accumulator": "fp32_buffer", "data": "synthetic"}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.layer:
        run_layer(args)
        return
    if args.sweep:
        run_sweep(args)
    elif args.configs:
        run_configs(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
