#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on one GB300 per rank.

One *step* is one pass of the whole hot path over one batch of the
[B=2, H=16, N=8192, d=128] causal workload (the shape shared by the bf16
forward, the bf16 backward and the FP8 forward workloads):

  fwd      bf16 forward               attn_fwd          -> O, LSE
  bwd      bf16 backward              attn_bwd          -> dQ, dK, dV
  quant    E4M3 block quantization    attn_quantize_fp8 (q, k with Hadamard; v transposed)
  fwd_fp8  FP8 forward                attn_fwd_fp8      -> O8, LSE8

FLOPs are counted as 4*B*H*N^2*d per forward (halved for causal) and 2.5x that
for the backward; the quantization pass counts no FLOPs.  ``value`` is the
step's FLOPs divided by its device time (CUDA events on the launching stream),
summed over ranks; the inputs (q, k, v, dO: 256 MiB) are larger than the
129 MB L2, so no flush is inserted between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

``--impl reference`` times the fp64 CPU oracle instead (the slow plain
definition, on the host cores, on a bounded sample of the same workload).
Multi-GPU (torchrun): every rank runs its own full batch (weak scaling, no
collective on the data path); ranks meet only at the timing barriers.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as wl  # noqa: E402

WORKLOAD = wl.Workload("attn_step_bf16_causal_b2h16n8192d128", "bwd", 2, 16, 8192, 128, "bf16",
                       True, hadamard=True)
COMPONENTS = ("fwd", "bwd", "quant", "fwd_fp8")
LAUNCHES = {"fwd": 1, "bwd": 3, "quant": 3, "fwd_fp8": 1}  # kernels per component call


# Sources whose hash identifies the kernel an ncu traffic figure was taken on.
KERNEL_SOURCES = {
    "fwd": ["fwd.cu", "fwd_wide.cu", "fwd.cuh", "sm103_ptx.cuh", "tiles.cuh", "smem_attr.cuh"],
    "fwd_fp8": ["fwd.cu", "fwd.cuh", "sm103_ptx.cuh", "tiles.cuh", "smem_attr.cuh"],
    "bwd": ["bwd.cu", "bwd_wide.cu", "bwd.cuh", "sm103_ptx.cuh", "tiles.cuh", "smem_attr.cuh",
            "unit_ring.cuh"],
    "quant": ["fp8.cu", "fp8.cuh", "sm103_ptx.cuh"],
}


def sources_sha256(component):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[component]:
        with open(os.path.join(ROOT, "exact_attention_75_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(component):
    """DRAM bytes per launch of the component's main kernel from the committed
    ncu summary (profiles/traffic.json), or None when the kernel's sources have
    changed since that capture."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f).get(component)
    except Exception:
        return None
    if not rec or rec.get("sources_sha256") != sources_sha256(component):
        return None
    return rec.get("dram_bytes")


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained",
                                                      pk["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ------------------------------------------------------------ clocks -------

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------ ranks --------

def max_over_ranks(values):
    """Element-wise max of per-rank timings (a host-side timing reduction,
    not part of the data path).  NCCL needs the tensor on the GPU, gloo on
    the CPU."""
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor(values, dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


class CudaTimer:
    """Device timing on one stream with CUDA events."""

    def __init__(self, stream):
        self.stream = stream

    def sync(self):
        torch.cuda.synchronize()

    def mark(self):
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e

    def elapsed_ms(self, a, b):
        return a.elapsed_time(b)


def timed_region(steps, run_step, world, timer, on_start=None):
    """Time exactly `steps` calls of run_step: every rank meets at a barrier,
    the device is synchronised, the steps run between two timer marks, the
    device is synchronised again and the ranks meet once more.  Returns this
    rank's elapsed milliseconds."""
    if world > 1:
        torch.distributed.barrier()
    timer.sync()
    if on_start is not None:
        on_start()
    t0 = timer.mark()
    for _ in range(steps):
        run_step()
    t1 = timer.mark()
    timer.sync()
    if world > 1:
        torch.distributed.barrier()
    return timer.elapsed_ms(t0, t1)


def job_times(ms_step, e2e_ms, world):
    """Per-step times of the whole job: the slowest rank's."""
    if world > 1:
        ms_step, e2e_ms = max_over_ranks([ms_step, e2e_ms])
    return ms_step, e2e_ms


def job_value(step_flops, ms, world):
    """Whole-job TFLOP/s: every rank processes its own batch of step_flops
    (weak scaling) in the slowest rank's time ms."""
    return world * step_flops / (ms * 1e-3) / 1e12


def component_roofline(c, flops, nbytes, ms, peaks):
    """Roofline object of one component of the step: tensor-bound
    contractions against the measured dense bf16 peak (the E4M3 forward
    against twice that, the nominal FP8:bf16 ratio, as no FP8 peak is
    measured by the driver), the quantization pass against HBM bandwidth."""
    if flops > 0:
        ach = flops / (ms * 1e-3) / 1e12
        peak = peaks["bf16_tflops"] * (2 if c == "fwd_fp8" else 1)
        kind = f"{peaks['source']} bf16 burst" + (" x2 (nominal E4M3 ratio)" if c == "fwd_fp8"
                                                   else "")
        return {"bound": "tensor", "achieved": round(ach, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(ach / peak, 4), "traffic": measured_traffic(c),
                "algorithmic_bytes": nbytes, "peak_kind": kind}
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": measured_traffic(c),
            "algorithmic_bytes": nbytes, "peak_kind": f"{peaks['source']} HBM copy"}


def rank_env(gpus):
    """(rank, world, local_rank) from torchrun's environment (1 rank
    without it); --gpus must match the launched world size."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != gpus:
        raise SystemExit(f"bench.py: --gpus {gpus} but {world} rank(s) were launched "
                         f"(WORLD_SIZE={os.environ.get('WORLD_SIZE')})")
    return int(os.environ.get("RANK", "0")), world, int(os.environ.get("LOCAL_RANK", "0"))


def launch_ranks_if_needed(args):
    """--gpus N > 1 run as a plain process: launch N ranks (one per GPU of
    this node) through torch.distributed.run on 127.0.0.1 with the same
    arguments, wait for them and return True.  Under torchrun: False."""
    if args.gpus <= 1 or "WORLD_SIZE" in os.environ:
        return False
    import socket
    with socket.socket() as so:
        so.bind(("127.0.0.1", 0))
        port = so.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
    rc = subprocess.call(cmd)
    if rc != 0:
        raise SystemExit(rc)
    return True


def rank_workload(w: wl.Workload, rank: int) -> wl.Workload:
    """Weak scaling: rank r owns global heads [r*B*H, (r+1)*B*H) of a job of
    world*B*H independent heads; its slice is drawn with seed r."""
    return w.with_(seed=w.seed + rank)


# ------------------------------------------------------------ GPU arm -------

class Step:
    """All buffers of one step, resident on the device."""

    def __init__(self, attn, w: wl.Workload, dev, components, like=None):
        self.attn, self.w, self.dev, self.components = attn, w, dev, components
        if like is None:
            inp = wl.make_inputs(w, with_do=True)
            self.host = {n: inp[n].pin_memory() for n in ("q", "k", "v", "do")}
            self.signs = inp["signs"].to(dev)
        else:  # a second set of device buffers on the same pinned host inputs
            self.host, self.signs = like.host, like.signs
        self.q, self.k, self.v, self.do = (self.host[n].to(dev) for n in ("q", "k", "v", "do"))
        B, H, N, d = w.B, w.H, w.N, w.d
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
        if "bwd" in components:
            self.ws = torch.empty(attn.bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8,
                                  device=dev)
            self.dq, self.dk, self.dv = (torch.empty_like(self.q) for _ in range(3))
        if "quant" in components or "fwd_fp8" in components:
            nb = (N + 63) // 64
            self.q8 = torch.empty((B, H, N, d), dtype=torch.uint8, device=dev)
            self.k8 = torch.empty_like(self.q8)
            self.v8t = torch.empty((B, H, d, N), dtype=torch.uint8, device=dev)
            self.sq, self.sk, self.sv = (torch.empty((B, H, nb), dtype=torch.float32,
                                                     device=dev) for _ in range(3))
            self.o8 = torch.empty_like(self.q)
            self.lse8 = torch.empty_like(self.lse)

    def run(self, name):
        a, w = self.attn, self.w
        if name == "fwd":
            a.fwd(self.q, self.k, self.v, causal=w.causal, scale=w.scale, out=self.o,
                  lse=self.lse)
        elif name == "bwd":
            a.bwd(self.q, self.k, self.v, self.o, self.do, self.lse, causal=w.causal,
                  scale=w.scale, workspace=self.ws, dq=self.dq, dk=self.dk, dv=self.dv)
        elif name == "quant":
            L = a.lib()
            import ctypes
            s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            B, H, N, d = w.B, w.H, w.N, w.d
            for x, out, sc, sg, tr in ((self.q, self.q8, self.sq, self.signs, 0),
                                       (self.k, self.k8, self.sk, self.signs, 0),
                                       (self.v, self.v8t, self.sv, None, 1)):
                st = L.attn_quantize_fp8(ctypes.c_void_p(x.data_ptr()),
                                         ctypes.c_void_p(out.data_ptr()),
                                         ctypes.c_void_p(sc.data_ptr()), B, H, N, d, 64,
                                         ctypes.c_void_p(0 if sg is None else sg.data_ptr()),
                                         tr, s)
                if st != 0:
                    raise a.AttnError("attn_quantize_fp8", st)
        elif name == "fwd_fp8":
            a.fwd_fp8(self.q8, self.k8, self.v8t, self.sq, self.sk, self.sv, causal=w.causal,
                      scale=w.scale, out=self.o8, lse=self.lse8)

    def outputs(self):
        outs = [self.o, self.lse]
        if "bwd" in self.components:
            outs += [self.dq, self.dk, self.dv]
        if "fwd_fp8" in self.components:
            outs += [self.o8, self.lse8]
        return outs


def component_flops(w: wl.Workload):
    return {"fwd": w.fwd_flops(), "bwd": w.bwd_flops(), "quant": 0.0,
            "fwd_fp8": w.fwd_flops()}


def component_bytes(w: wl.Workload):
    """Algorithmic HBM bytes per launch of each component."""
    BH, N, d = w.B * w.H, w.N, w.d
    elems = BH * N * d
    return {"fwd": 4 * elems * 2 + BH * N * 4,
            "bwd": 8 * elems * 2 + BH * N * 4,
            "quant": 3 * (elems * 2 + elems + BH * ((N + 63) // 64) * 4),
            "fwd_fp8": 3 * elems + elems * 2 + BH * N * 4 + 3 * BH * ((N + 63) // 64) * 4}


SPLIT_KV_N = 4  # key splits of the split-KV measurement


def split_kv_timing(attn, st, w, stream, n_split, iters=20):
    """The split over the keys + merge on the same workload, timed apart from
    the step: attn_fwd_split (n_split runs of key blocks) and attn_merge,
    each with CUDA events on the launching stream after 3 warm-up calls."""
    BH, N, d = w.B * w.H, w.N, w.d
    o_part = torch.empty((n_split, w.B, w.H, N, d), dtype=st.q.dtype, device=st.q.device)
    l_part = torch.empty((n_split, w.B, w.H, N), dtype=torch.float32, device=st.q.device)
    o = torch.empty_like(st.q)
    lse = torch.empty((w.B, w.H, N), dtype=torch.float32, device=st.q.device)
    for _ in range(3):
        attn.fwd_split(st.q, st.k, st.v, n_split, causal=w.causal, out=o_part, lse=l_part)
        attn.merge(o_part, l_part, out=o, lse=lse)
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    ts, tm = [], []
    for _ in range(iters):
        e[0].record(stream)
        attn.fwd_split(st.q, st.k, st.v, n_split, causal=w.causal, out=o_part, lse=l_part)
        e[1].record(stream)
        attn.merge(o_part, l_part, out=o, lse=lse)
        e[2].record(stream)
        torch.cuda.synchronize()
        ts.append(e[0].elapsed_time(e[1]))
        tm.append(e[1].elapsed_time(e[2]))
    status = attn.poll_status()
    if status[0] != 0:
        raise RuntimeError(f"device status after the split-KV timing: {status}")
    ms_s, ms_m = statistics.mean(ts), statistics.mean(tm)
    # algorithmic bytes of the merge: read the partial O and LSE, write O, LSE
    merge_bytes = n_split * (BH * N * d * 2 + BH * N * 4) + BH * N * d * 2 + BH * N * 4
    return {"n_split": n_split, "fwd_split_ms": round(ms_s, 4), "merge_ms": round(ms_m, 4),
            "tflops": round(w.fwd_flops() / ((ms_s + ms_m) * 1e-3) / 1e12, 1),
            "merge_gbs": round(merge_bytes / (ms_m * 1e-3) / 1e9, 1),
            "merge_bytes": merge_bytes}


GQA_KV_HEADS = 4  # key/value heads of the grouped-query measurement


def gqa_timing(attn, st, w, stream, hkv, iters=10):
    """Forward + backward with grouped query heads on the step's workload
    (H query heads, hkv key/value heads: the first head of each group of the
    step's K, V, so no extra input draw), timed apart from the step."""
    G = w.H // hkv
    k = st.k[:, ::G].contiguous()
    v = st.v[:, ::G].contiguous()
    o, lse = attn.fwd(st.q, k, v, causal=w.causal)
    grads = attn.bwd(st.q, k, v, o, st.do, lse, causal=w.causal)
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    tf, tb = [], []
    for _ in range(iters):
        e[0].record(stream)
        attn.fwd(st.q, k, v, causal=w.causal, out=o, lse=lse)
        e[1].record(stream)
        attn.bwd(st.q, k, v, o, st.do, lse, causal=w.causal, dq=grads[0], dk=grads[1],
                 dv=grads[2])
        e[2].record(stream)
        torch.cuda.synchronize()
        tf.append(e[0].elapsed_time(e[1]))
        tb.append(e[1].elapsed_time(e[2]))
    status = attn.poll_status()
    if status[0] != 0:
        raise RuntimeError(f"device status after the GQA timing: {status}")
    mf, mb = statistics.mean(tf), statistics.mean(tb)
    return {"kv_heads": hkv, "fwd_ms": round(mf, 4), "bwd_ms": round(mb, 4),
            "fwd_tflops": round(w.fwd_flops() / (mf * 1e-3) / 1e12, 1),
            "bwd_tflops": round(w.bwd_flops() / (mb * 1e-3) / 1e12, 1),
            "note": "grouped query heads, timed apart from the step (not in value)"}


HEAD_DIMS = (64, 96, 192, 256)   # timed beside the step's d = 128
WIDE_BACKWARD = True             # the backward at d in {192, 256}


def head_dim_timing(attn, w, dev, stream, iters=10):
    """Forward + backward at the other head dims on the step's B, H, N,
    dtype and masking, timed apart from the step.  Inputs are standard
    normals drawn on the device from a seeded generator (timing only; parity
    at these head dims is in the tests)."""
    out = {}
    g = torch.Generator(device=dev).manual_seed(1234)
    for d in HEAD_DIMS:
        with_bwd = d <= 128 or WIDE_BACKWARD
        wd = w.with_(d=d)
        shape = (wd.B, wd.H, wd.N, d)
        q, k, v, do = (torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
                       .to(torch.bfloat16) for _ in range(4))
        o, lse = attn.fwd(q, k, v, causal=wd.causal, scale=wd.scale)
        grads = attn.bwd(q, k, v, o, do, lse, causal=wd.causal, scale=wd.scale) \
            if with_bwd else None
        torch.cuda.synchronize()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        tf, tb = [], []
        for _ in range(iters):
            e[0].record(stream)
            attn.fwd(q, k, v, causal=wd.causal, scale=wd.scale, out=o, lse=lse)
            e[1].record(stream)
            if with_bwd:
                attn.bwd(q, k, v, o, do, lse, causal=wd.causal, scale=wd.scale, dq=grads[0],
                         dk=grads[1], dv=grads[2])
            e[2].record(stream)
            torch.cuda.synchronize()
            tf.append(e[0].elapsed_time(e[1]))
            tb.append(e[1].elapsed_time(e[2]))
        status = attn.poll_status()
        if status[0] != 0:
            raise RuntimeError(f"device status after the d={d} timing: {status}")
        mf, mb = statistics.mean(tf), statistics.mean(tb)
        pk = load_peaks()["bf16_tflops"]
        r = {"fwd_ms": round(mf, 4), "fwd_tflops": round(wd.fwd_flops() / (mf * 1e-3) / 1e12, 1)}
        r["fwd_frac"] = round(r["fwd_tflops"] / pk, 4)
        if with_bwd:
            r.update({"bwd_ms": round(mb, 4),
                      "bwd_tflops": round(wd.bwd_flops() / (mb * 1e-3) / 1e12, 1)})
            r["bwd_frac"] = round(r["bwd_tflops"] / pk, 4)
        out[f"d{d}"] = r
        del q, k, v, do, o, lse, grads
    out["note"] = "bf16, the step's B, H, N and masking; timed apart from the step (not in value)"
    return out


def _timed(fn, stream, flush, iters, warmup=3):
    """Per-launch device times (ms) of fn on the stream, L2 flushed before
    each launch (outside the timed region)."""
    for _ in range(warmup):
        fn()
    ts = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(iters):
        flush.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return ts


def _summary(ts):
    q1, q2, q3 = statistics.quantiles(ts, n=4)
    return {"ms_median": round(q2, 4), "ms_iqr": [round(q1, 4), round(q3, 4)]}


def sweep_timing(attn, dev, stream, iters=20):
    """Forward at every configuration of the pages' workloads besides the
    step: the 256-token fp16 case, the fp16 d=64 and bf16 d=128 (inputs x0.5)
    sweeps over N with B*N = 16384, causal and not.  Inputs are seeded
    standard normals drawn on the device (timing only; parity is in the
    tests); L2 is flushed before every launch.  GB/s counts the algorithmic
    bytes (read Q, K, V, write O once; LSE fp32)."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    g = torch.Generator(device=dev).manual_seed(0)
    points = [wl.TINY_FWD_FP16]
    for causal in (True, False):
        points += wl.sweep_d64(causal)
    for causal in (True, False):
        points += wl.sweep_d128(causal)
    out = []
    for w in points:
        shape = (w.B, w.H, w.N, w.d)
        q, k, v = ((torch.randn(shape, generator=g, device=dev) * w.input_scale)
                   .to(w.torch_dtype) for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
        ts = _timed(lambda: attn.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse),
                    stream, flush, iters)
        status = attn.poll_status()
        if status[0] != 0:
            raise RuntimeError(f"device status after {w.name}: {status}")
        r = _summary(ts)
        nbytes = 4 * w.B * w.H * w.N * w.d * 2 + 4 * w.B * w.H * w.N
        r.update({"workload": w.name, "dtype": w.dtype, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                  "causal": w.causal,
                  "tflops": round(w.fwd_flops() / (r["ms_median"] * 1e-3) / 1e12, 1),
                  "gbs": round(nbytes / (r["ms_median"] * 1e-3) / 1e9, 1)})
        out.append(r)
        del q, k, v, o, lse
    return out


def tensor_peaks(dev, stream, iters=20):
    """Dense 8192^3 products through the libraries, the same way for both
    types: bf16 torch.matmul and E4M3 torch._scaled_mm (unit scales, bf16
    output).  A denominator for the E4M3 forward, not part of the path."""
    M = 8192
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    res = {}
    a = torch.randn(M, M, device=dev).to(torch.bfloat16)
    b = torch.randn(M, M, device=dev).to(torch.bfloat16)
    ts = _timed(lambda: torch.matmul(a, b), stream, flush, iters)
    res["bf16_tflops"] = round(2 * M ** 3 / (statistics.median(ts) * 1e-3) / 1e12, 1)
    try:
        a8, b8 = a.to(torch.float8_e4m3fn), b.to(torch.float8_e4m3fn)
        one = torch.ones((), dtype=torch.float32, device=dev)
        ts = _timed(lambda: torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one,
                                             out_dtype=torch.bfloat16), stream, flush, iters)
        res["e4m3_tflops"] = round(2 * M ** 3 / (statistics.median(ts) * 1e-3) / 1e12, 1)
    except Exception as e:  # the installed library may not offer the E4M3 product
        res["e4m3_unavailable"] = str(e).splitlines()[0][:200]
    res["note"] = "8192^3, median of 20 launches, L2 flushed; burst"
    return res


def decode_timing(attn, dev, stream, peaks, iters=20):
    """Decoding against a key/value cache, timed apart from the step: one
    query per sequence, 16 sequences x 16 heads, an 8192-row bf16 d=128
    cache, split over the keys into 8 runs (attn_fwd_kv) and merged
    (attn_merge); and the same with 2 key/value heads.  HBM-bound: the algorithmic bytes are the cache's K and V
    read once (plus q, the partials and O, under 0.1 %).  Inputs are seeded
    standard normals drawn on the device (timing only; parity is in the
    tests); L2 is flushed before every call."""
    w = wl.DECODE_BF16_D128
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    n_split = wl.DECODE_SPLITS
    for hkv in (w.H, wl.DECODE_GQA_KV_HEADS):
        g = torch.Generator(device=dev).manual_seed(0)
        q = torch.randn((w.B, w.H, wl.DECODE_NQ, w.d), generator=g, device=dev) \
            .to(torch.bfloat16)
        k, v = (torch.randn((w.B, hkv, w.N, w.d), generator=g, device=dev).to(torch.bfloat16)
                for _ in range(2))
        Op, Lp = attn.fwd_kv(q, k, v, n_split, causal=w.causal)
        O, L = attn.merge(Op, Lp)

        def step():
            attn.fwd_kv(q, k, v, n_split, causal=w.causal, out=Op, lse=Lp)
            attn.merge(Op, Lp, out=O, lse=L)

        ts = _timed(step, stream, flush, iters)
        status = attn.poll_status()
        if status[0] != 0:
            raise RuntimeError(f"device status after the decode timing: {status}")
        r = _summary(ts)
        kv_bytes = 2 * w.B * hkv * w.N * w.d * 2
        # Context for the fraction: the same bytes read by a plain library
        # reduction under the same flush (a short read-only kernel also pays
        # the flush's dirty lines being written back and its own ramp).
        kv = torch.cat([k.reshape(-1), v.reshape(-1)]).view(torch.int64)
        r["read_same_bytes_ms"] = round(statistics.median(
            _timed(lambda: kv.sum(), stream, flush, iters)), 4)
        del kv
        gbs = kv_bytes / (r["ms_median"] * 1e-3) / 1e9
        r.update({"workload": w.name, "kv_heads": hkv, "n_split": n_split,
                  "queries": wl.DECODE_NQ, "gbs": round(gbs, 1),
                  "roofline": {"bound": "hbm", "achieved": round(gbs, 1),
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": round(gbs / peaks["hbm_gbs"], 4),
                               "algorithmic_bytes": kv_bytes}})
        out["mha" if hkv == w.H else "gqa"] = r
        del q, k, v, Op, Lp, O, L
    out["note"] = ("fwd_kv (key splits, the warp-level decoding kernel: at most 16 query "
                   "rows per key/value head) + merge, L2 flushed, timed apart from the step "
                   "(not in value); gqa: 16 query heads on 2 key/value heads, a group's "
                   "8 queries in one unit; read_same_bytes_ms: torch.sum over the same K/V "
                   "bytes under the same flush")
    return out


def varlen_timing(attn, dev, stream, iters=10):
    """Forward + backward on the packed variable-length batch (16 heads,
    d = 128, bf16, causal, 16384 tokens per head in the seeded length mix),
    timed apart from the step.  FLOPs per sequence of L rows and head: the
    causal forward count 2 L^2 d, the backward 2.5x that."""
    lengths = wl.varlen_lengths()
    H, d = wl.VARLEN_HEADS, wl.VARLEN_D
    inp = wl.make_varlen_inputs(lengths, H, H, d, "bf16", seed=0)
    q, k, v, do, cu = (inp[n].to(dev) for n in ("q", "k", "v", "do", "cu_seqlens"))
    mx = max(lengths)
    o, lse = attn.fwd_varlen(q, k, v, cu, mx, causal=True)
    grads = attn.bwd_varlen(q, k, v, o, do, lse, cu, mx, causal=True)
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    tf, tb = [], []
    for _ in range(iters):
        e[0].record(stream)
        attn.fwd_varlen(q, k, v, cu, mx, causal=True, out=o, lse=lse)
        e[1].record(stream)
        attn.bwd_varlen(q, k, v, o, do, lse, cu, mx, causal=True, dq=grads[0], dk=grads[1],
                        dv=grads[2])
        e[2].record(stream)
        torch.cuda.synchronize()
        tf.append(e[0].elapsed_time(e[1]))
        tb.append(e[1].elapsed_time(e[2]))
    status = attn.poll_status()
    if status[0] != 0:
        raise RuntimeError(f"device status after the variable-length timing: {status}")
    ff = sum(2.0 * H * n * n * d for n in lengths)
    mf, mb = statistics.mean(tf), statistics.mean(tb)
    return {"lengths": lengths, "heads": H, "d": d, "fwd_ms": round(mf, 4),
            "bwd_ms": round(mb, 4), "fwd_tflops": round(ff / (mf * 1e-3) / 1e12, 1),
            "bwd_tflops": round(2.5 * ff / (mb * 1e-3) / 1e12, 1),
            "note": "packed variable-length batch (causal per sequence), timed apart from "
                    "the step (not in value)"}


def run_gpu(args, rank, world, local_rank):
    import exact_attention_75_gb300 as attn
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = WORKLOAD
    # Every component of the step runs; one the library rejects (for instance
    # with ATTN_ERR_UNSUPPORTED) fails the bench instead of shrinking the step.
    comps = list(COMPONENTS)
    st = Step(attn, rank_workload(w, rank), dev, comps)
    flops = component_flops(w)
    nbytes = component_bytes(w)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for c in comps:
            st.run(c)
    torch.cuda.synchronize()
    status = attn.poll_status()
    if status[0] != 0:
        raise RuntimeError(f"device status after warm-up: {status}")

    ev = {c: [] for c in comps}
    sampler = ClockSampler(local_rank)

    def one_step():
        for c in comps:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            st.run(c)
            e1.record(stream)
            ev[c].append((e0, e1))

    ms_total = timed_region(args.steps, one_step, world, CudaTimer(stream),
                            on_start=lambda: (sampler.start(), time.sleep(0.3)))
    clocks = sampler.stop()
    per = {c: statistics.mean(a.elapsed_time(b) for a, b in ev[c]) for c in comps}
    status = attn.poll_status()
    if status[0] != 0:
        raise RuntimeError(f"device status after timed region: {status}")

    # e2e through the public API with host buffers: every step copies its
    # inputs from pinned host memory and every output back, inside the timed
    # region.  Steps are pipelined over two sets of device buffers: the H2D
    # copy of step k+1 (one copy stream) and the D2H copy of step k (another)
    # run while step k computes.
    sets = [st, Step(attn, rank_workload(w, rank), dev, comps, like=st)]
    outs = [x.outputs() for x in sets]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs[0]]
    h2d = sum(st.host[n].numel() * st.host[n].element_size() for n in ("q", "k", "v", "do"))
    d2h = sum(o.numel() * o.element_size() for o in outs[0])
    # as many steps as the timed region (the first step's input copy and the
    # last step's output copy are not overlapped, so few steps understate the
    # pipelined rate)
    e2e_steps = max(3, args.steps)
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_round(nsteps, start):
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "comp", "out")}
        up.wait_event(start)
        down.wait_event(start)
        for k in range(nsteps):
            b = k % 2
            x = sets[b]
            with torch.cuda.stream(up):
                if k >= 2:
                    up.wait_event(ev["comp"][b])  # step k-2 has read these inputs
                for n in ("q", "k", "v", "do"):
                    getattr(x, n).copy_(x.host[n], non_blocking=True)
                ev["in"][b].record(up)
            stream.wait_event(ev["in"][b])
            if k >= 2:
                stream.wait_event(ev["out"][b])  # step k-2's outputs are on the host
            for c in comps:
                x.run(c)
            ev["comp"][b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev["comp"][b])
                for o, h in zip(outs[b], host_out):
                    h.copy_(o, non_blocking=True)
                ev["out"][b].record(down)
        stream.wait_stream(up)
        stream.wait_stream(down)

    torch.cuda.synchronize()
    warm = torch.cuda.Event()
    warm.record(stream)
    e2e_round(2, warm)  # untimed
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_round(e2e_steps, e0)
    e1 = torch.cuda.Event(enable_timing=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    del sets[1]

    split = split_kv_timing(attn, st, w, stream, n_split=SPLIT_KV_N)
    gqa = gqa_timing(attn, st, w, stream, GQA_KV_HEADS) if "bwd" in comps else None
    varlen = varlen_timing(attn, dev, stream) if "bwd" in comps else None
    head_dims = head_dim_timing(attn, w, dev, stream) if "bwd" in comps else None
    decode = decode_timing(attn, dev, stream, load_peaks())

    step_flops = sum(flops[c] for c in comps)
    ms_step, e2e_ms = job_times(ms_total / args.steps, e2e_ms, world)
    return dict(comps=comps, per=per, ms_step=ms_step, e2e_ms=e2e_ms, clocks=clocks, split=split,
                gqa=gqa, varlen=varlen, head_dims=head_dims, decode=decode,
                flops=flops, nbytes=nbytes, step_flops=step_flops, h2d=h2d, d2h=d2h,
                launches=sum(LAUNCHES[c] for c in comps) * args.steps)


# ------------------------------------------------------ oracle (CPU) arm -----

def cpu_oracle_sample(budget_s: float = 20.0):
    """Time the fp64 oracle (as it stands) on one head of the workload.

    Forward + backward of one (b, h) head at N = 8192, d = 128; repeated while
    the time budget lasts.  Returns (TFLOP/s, seconds, heads done, threads).
    """
    import oracle
    w = WORKLOAD.with_(B=1, H=1)
    inp = wl.make_inputs(w, with_do=True)
    q, k, v, do = (inp[n][0, 0].to(torch.float64).numpy() for n in ("q", "k", "v", "do"))
    heads = 0
    t0 = time.perf_counter()
    while True:
        oracle.attention_head(q, k, v, w.causal, w.scale)
        oracle.attention_backward_head(q, k, v, do, w.causal, w.scale)
        heads += 1
        if time.perf_counter() - t0 > budget_s / 2 or heads >= 8:
            break
    dt = time.perf_counter() - t0
    fl = heads * (w.fwd_flops() + w.bwd_flops())
    return fl / dt / 1e12, dt, heads, os.cpu_count()


# One entry point on one workload, for profiling a single kernel: the step's
# components on [2,16,8192,128] causal, and the other head dims' forward and
# backward on [2,16,8192,d] bf16 causal.
CASES = ("fwd", "bwd", "quant", "fwd_fp8", "fwd_d64", "bwd_d64", "fwd_d96", "bwd_d96",
         "fwd_d192", "bwd_d192", "fwd_d256", "bwd_d256", "merge", "decode", "decode_gqa",
         "fwd_fp16_d64_n512")


def run_case(name, steps, warmup):
    import exact_attention_75_gb300 as attn
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    if name in COMPONENTS:
        st = Step(attn, WORKLOAD, dev, list(COMPONENTS))
        for c in COMPONENTS:  # every input of the component defined
            st.run(c)
        fn = lambda: st.run(name)  # noqa: E731
        w = WORKLOAD
    elif name == "merge":
        # the split-KV merge of the step's workload: the partials of a 4-way
        # split of the keys, computed once, merged on every call
        w = WORKLOAD
        g = torch.Generator(device=dev).manual_seed(1234)
        q, k, v = (torch.randn((w.B, w.H, w.N, w.d), generator=g, device=dev)
                   .to(torch.bfloat16) for _ in range(3))
        op, lp = attn.fwd_split(q, k, v, SPLIT_KV_N, causal=w.causal, scale=w.scale)
        o, lse = attn.merge(op, lp)
        fn = lambda: attn.merge(op, lp, out=o, lse=lse)  # noqa: E731
    elif name == "fwd_fp16_d64_n512":
        # the shortest point of the fp16 d = 64 sweep: [32,16,512,64] causal
        w = wl.sweep_d64(True)[0]
        inp = wl.make_inputs(w)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        o, lse = attn.fwd(q, k, v, causal=w.causal, scale=w.scale)
        fn = lambda: attn.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)  # noqa
    elif name in ("decode", "decode_gqa"):
        # the decode batch's forward over the key splits (16 or 2 key/value
        # heads), without the merge
        w = wl.DECODE_BF16_D128
        hkv = w.H if name == "decode" else wl.DECODE_GQA_KV_HEADS
        g = torch.Generator(device=dev).manual_seed(1234)
        q = torch.randn((w.B, w.H, wl.DECODE_NQ, w.d), generator=g, device=dev) \
            .to(torch.bfloat16)
        k, v = (torch.randn((w.B, hkv, w.N, w.d), generator=g, device=dev).to(torch.bfloat16)
                for _ in range(2))
        op, lp = attn.fwd_kv(q, k, v, wl.DECODE_SPLITS, causal=w.causal, scale=w.scale)
        fn = lambda: attn.fwd_kv(q, k, v, wl.DECODE_SPLITS, causal=w.causal,  # noqa: E731
                                 scale=w.scale, out=op, lse=lp)
    elif name in CASES:
        kind, d = name.split("_d")
        w = WORKLOAD.with_(d=int(d))
        g = torch.Generator(device=dev).manual_seed(1234)
        shape = (w.B, w.H, w.N, w.d)
        q, k, v, do = (torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)
                       for _ in range(4))
        o, lse = attn.fwd(q, k, v, causal=w.causal, scale=w.scale)
        grads = [torch.empty_like(q) for _ in range(3)]
        if kind == "fwd":
            fn = lambda: attn.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)  # noqa
        else:
            fn = lambda: attn.bwd(q, k, v, o, do, lse, causal=w.causal, scale=w.scale,  # noqa
                                  dq=grads[0], dk=grads[1], dv=grads[2])
    else:
        raise SystemExit(f"unknown case {name}; one of {', '.join(CASES)}")
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    status = attn.poll_status()
    if status[0] != 0:
        raise RuntimeError(f"device status after case {name}: {status}")
    return {"case": name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": w.causal,
            "calls": steps, "ms_per_call": e0.elapsed_time(e1) / max(steps, 1)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None,
                    help="run one entry point on its workload (warmup + steps calls, for "
                         "profiling one kernel): " + ", ".join(CASES))
    ap.add_argument("--sweeps", action="store_true",
                    help="time the forward at every configuration and sweep point of the "
                         "workloads (one GPU) and print them instead of the step line")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    if launch_ranks_if_needed(args):
        return
    rank, world, local_rank = rank_env(args.gpus)
    peaks = load_peaks()
    w = WORKLOAD

    if args.case is not None:
        if rank == 0:
            print(json.dumps(run_case(args.case, args.steps, args.warmup)), flush=True)
        return

    if args.sweeps and args.impl == "gb300":
        if rank != 0:
            return
        import exact_attention_75_gb300 as attn
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        stream = torch.cuda.current_stream()
        sampler = ClockSampler(local_rank)
        sampler.start()
        sweeps = sweep_timing(attn, dev, stream)
        clocks = sampler.stop()
        line = {"metric": "attention fwd TFLOP/s per configuration", "impl": "gb300",
                "unit": "TFLOP/s", "higher_is_better": True, "n_gpus": 1, "data": "synthetic",
                "l2": "flushed (256 MiB write) before every launch", "clocks": clocks,
                "peaks": {"measured": peaks, "this_run": tensor_peaks(dev, stream)},
                "sweeps": sweeps}
        print(json.dumps(line), flush=True)
        return

    if args.impl == "reference":
        if rank != 0:
            return
        per_step = []
        for _ in range(args.warmup):  # untimed warm-up samples
            cpu_oracle_sample(budget_s=1.0)
        heads_total, t_total = 0, 0.0
        for _ in range(args.steps):
            tf, dt, heads, cores = cpu_oracle_sample(budget_s=min(20.0, 120.0 / args.steps))
            per_step.append(tf)
            heads_total += heads
            t_total += dt
        value = statistics.mean(per_step)
        sample = (f"fwd+bwd of {heads_total} (b,h) head(s) of the workload (N=8192, d=128, "
                  f"causal) in fp64 numpy over {args.steps} step(s)")
        line = {"metric": "attention fwd/bwd TFLOP/s", "value": value, "unit": "TFLOP/s",
                "impl": "reference", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": 1000 * t_total / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f64", "data": "synthetic",
                "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                           "causal": w.causal},
                "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores,
                                 "kind": "oracle", "sample": sample},
                "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl")
    r = run_gpu(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return

    comps, per = r["comps"], r["per"]
    value = job_value(r["step_flops"], r["ms_step"], world)
    e2e_val = job_value(r["step_flops"], r["e2e_ms"], world)
    breakdown = {}
    for c in comps:
        ms = per[c]
        tf = r["flops"][c] / (ms * 1e-3) / 1e12 if r["flops"][c] else None
        breakdown[c] = {"ms": round(ms, 4), "tflops": None if tf is None else round(tf, 1),
                        "gbs": round(r["nbytes"][c] / (ms * 1e-3) / 1e9, 1),
                        "roofline": component_roofline(c, r["flops"][c], r["nbytes"][c], ms,
                                                       peaks)}
    # dominant kernel = largest share of the step's time
    dom = max(comps, key=lambda c: per[c])
    roof = dict(breakdown[dom]["roofline"], kernel=dom)
    # the 16-bit part of the step alone (the E4M3 forward computes in FP8)
    bf16_comps = [c for c in ("fwd", "bwd") if c in comps]
    bf16_value = job_value(sum(r["flops"][c] for c in bf16_comps),
                           sum(per[c] for c in bf16_comps), world)
    line = {"metric": "attention fwd/bwd TFLOP/s", "value": round(value, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(r["ms_step"], 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+e4m3",
            "dtype_note": "value counts the bf16 forward and backward and the E4M3 forward "
                          "(the quantization pass counts no FLOPs); value_bf16 is the bf16 "
                          "forward + backward alone",
            "value_bf16": round(bf16_value, 2), "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "causal": w.causal, "components": comps,
                       "l2": "inputs (q,k,v,dO = 256 MiB) larger than L2; no flush",
                       "parallelism": f"replicas x{world}"},
            "breakdown": breakdown, "roofline": roof, "clocks": r["clocks"],
            "gpu_launches": r["launches"],
            "e2e": {"value": round(e2e_val, 2), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "note": "public API, pinned host buffers; each step's H2D and D2H copies "
                            "overlap the neighbouring steps' compute (two device buffer "
                            "sets, two copy streams)"}}
    if r.get("split"):
        sp = dict(r["split"])
        mb = sp.pop("merge_bytes")
        sp["note"] = ("split over the keys + merge, timed apart from the step (not in value); "
                      "tflops = forward FLOPs / (split forward + merge)")
        sp["merge_roofline"] = {"bound": "hbm", "achieved": sp["merge_gbs"],
                                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                "frac": round(sp["merge_gbs"] / peaks["hbm_gbs"], 4),
                                "algorithmic_bytes": mb}
        line["split_kv"] = sp
    if r.get("gqa"):
        line["gqa"] = r["gqa"]
    if r.get("varlen"):
        line["varlen"] = r["varlen"]
    if r.get("head_dims"):
        line["head_dims"] = r["head_dims"]
    if r.get("decode"):
        line["decode"] = r["decode"]
    if not args.no_cpu_baseline:
        tf, dt, heads, cores = cpu_oracle_sample()
        line["cpu_baseline"] = {"value": tf, "unit": "TFLOP/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"fp64 numpy fwd+bwd of {heads} head(s) "
                                          f"(N=8192, d=128, causal), {dt:.1f} s"}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
