#!/usr/bin/env python3
"""Benchmark of the GB300 SDPA backward: TFLOP/s and fraction of dense bf16 peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

One step = one full backward (preprocess -> main -> dQ kernel, which also
carries the GQA dK/dV group reduction)
over one batch of the workload, inputs resident in HBM. Each step is timed
with CUDA events on the launching stream; a 256 MiB buffer is written between
steps so that every step starts with a cold L2 (the flush is outside the event
pair). FLOPs are algorithmic: 2 * (3*D_qk + 2*D_v) per visible (query, key)
pair (= 10 * D per pair when D_qk = D_v), counted exactly from the mask.

Inputs: Q, K, V, dO are seeded draws (workloads.py); O and LSE are the fp64
oracle forward of those draws, computed in the CPU-baseline leg on rank 0
(which also times the oracle backward on a bounded sample of the workload)
and broadcast to the other ranks. The timed GPU path never calls the oracle.

Multi-GPU: the op does not shard across GPUs in this library; N ranks run N
independent replicas of the workload (weak scaling) and the step time is the
max over ranks. `--impl reference` times the fp64 oracle on the host cores
(the only reference this op has) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "SDPA backward TFLOP/s (bf16, 1xGB300) and fraction of dense tensor peak"
METRIC_FWD = "SDPA forward TFLOP/s (bf16, 1xGB300) and fraction of dense tensor peak"
DEFAULT_WORKLOAD = "causal_gqa_det"
L2_FLUSH_BYTES = 256 << 20


# ---------------------------------------------------------------- FLOP counting
def visible_pairs(w: workloads.Workload, lens) -> int:
    """Visible (query, key) pairs summed over batch rows and query heads: per query
    q the visible keys form the interval [q+diag-W, q+diag+R] clipped to [0, L_kv)."""
    total = 0
    for b in range(w.B):
        Lq = w.Sq if lens is None else min(int(lens[b]), w.Sq)
        Lk = w.Skv if lens is None else min(int(lens[b]), w.Skv)
        if Lq <= 0 or Lk <= 0:
            continue
        diag = (Lk - Lq) if w.bottom_right else 0
        q = np.arange(Lq, dtype=np.int64)
        lo = np.zeros(Lq, dtype=np.int64)
        hi = np.full(Lq, Lk - 1, dtype=np.int64)
        if w.causal:
            hi = np.minimum(hi, q + diag + max(w.window_right, 0))
        if w.window_left >= 0:
            lo = np.maximum(lo, q + diag - w.window_left)
        total += int(np.clip(hi - lo + 1, 0, None).sum()) * w.Hq
    return total


def flops_per_pair(w: workloads.Workload) -> int:
    return 2 * (3 * w.Dqk + 2 * w.Dv)


def fwd_flops_per_pair(w: workloads.Workload) -> int:
    """S = Q K^T and O = P V: 2 * (D_qk + D_v) per visible pair."""
    return 2 * (w.Dqk + w.Dv)


def main_kernel_flops_per_pair(w: workloads.Workload) -> int:
    """Algorithmic FLOPs of the main kernel per visible pair: all five GEMMs, or
    four on the two-kernel route, where dQ = dS K runs in the separate dQ kernel
    (the library takes that route for D_qk = 192 and 256, and for D_qk = 128 when
    deterministic). At D = 256 the kernel runs S and dP twice (once per half of
    the dK/dV columns); only the algorithmic four are counted."""
    if w.Dqk > 128 or (w.deterministic and w.Dqk == 128):
        return 2 * (2 * w.Dqk + 2 * w.Dv)
    return flops_per_pair(w)


def main_kernel_bytes_bias(w: workloads.Workload, pairs: int, bias, dbias_esz: int = 4) -> int:
    """Algorithmic DRAM bytes of one biased main-kernel launch: the bias at the
    visible pairs (its element size each), every dBias element written once
    (``dbias_esz`` bytes: 4 for fp32, 2 for the io-type dBias),
    and each Q, K, V, dO, dK, dV element moved once with the fp32 dQ accumulator
    read and written once (the reduction route; the stored-dS route moves bf16 dS
    instead, counted the same here)."""
    esz = bias.element_size()
    dbias = bias.numel() * dbias_esz
    qdo = 2 * w.B * w.Hq * w.Sq * w.Dqk * 2
    kv = w.B * w.Hkv * w.Skv * (w.Dqk + w.Dv) * 2
    dq_acc = 2 * w.B * w.Hq * w.Sq * w.Dqk * 4
    return pairs * esz + dbias + qdo + 2 * kv + dq_acc


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU works."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]

    def __init__(self, index: int, interval_ms: int = 50):
        self.index, self.interval = index, interval_ms
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", str(self.interval)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        rows = []
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[2], parts[3:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- distributed
def init_dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def broadcast_tensor(t: torch.Tensor, world: int):
    if world > 1:
        import torch.distributed as dist
        dist.broadcast(t, src=0)
    return t


# ---------------------------------------------------------------- CPU baseline (oracle)
def _problem(w, lens):
    import oracle
    return oracle.Problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv, scale=w.resolved_scale,
                          causal=w.causal,
                          bottom_right=w.bottom_right, window_left=w.window_left,
                          window_right=w.window_right,
                          seq_q_lens=None if lens is None else lens.numpy(),
                          seq_kv_lens=None if lens is None else lens.numpy())


def oracle_forward_inputs(w, t):
    """O (bf16) and LSE (fp32) of the workload from the fp64 oracle forward (with
    the additive bias t["bias"] when there is one)."""
    import oracle
    p = _problem(w, t["seq_q_lens"])
    bias = t.get("bias")
    q64, k64, v64 = (t[x].double().numpy() for x in ("q", "k", "v"))
    if t.get("qat"):  # NVFP4 QAT: the high-precision O of the fake-quantized inputs
        q64, k64, v64 = oracle.fake_nvfp4(q64), oracle.fake_nvfp4(k64), oracle.fake_nvfp4(v64)
    o64, lse64 = oracle.forward(p, q64, k64, v64,
                                bias=None if bias is None else bias.double().numpy())
    return torch.from_numpy(o64).to(t["q"].dtype), torch.from_numpy(lse64).float()


def _head_slice(w, t, o, lse, G_groups):
    """The first G_groups KV heads with their query heads (the sample unit)."""
    G = w.Hq // w.Hkv
    hq = G_groups * G
    return {k: v[:, :hq].contiguous() if k in ("q", "do") else v[:, :G_groups].contiguous()
            for k, v in (("q", t["q"]), ("do", t["do"]), ("k", t["k"]), ("v", t["v"]))}, \
        o[:, :hq].contiguous(), lse[:, :hq].contiguous(), hq


def oracle_backward_sample(w, t, o, lse, groups):
    """Runs the oracle backward on the first `groups` KV-head groups of every batch
    row; returns (seconds, algorithmic FLOPs of the sample)."""
    import oracle
    sl, os_, ls, hq = _head_slice(w, t, o, lse, groups)
    ws = w.with_(Hq=hq, Hkv=groups)
    p = _problem(ws, t["seq_q_lens"])
    args = [sl["q"].double().numpy(), sl["k"].double().numpy(), sl["v"].double().numpy(),
            os_.double().numpy(), sl["do"].double().numpy(), ls.double().numpy()]
    bias = t.get("bias")
    t0 = time.perf_counter()
    if t.get("qat"):
        oracle.qat_backward(p, *args)
    elif bias is None:
        oracle.backward(p, *args)
    else:  # the biased backward plus dBias, on the sample's heads
        b64 = bias[:, :hq].contiguous().double().numpy()
        oracle.backward(p, *args, bias=b64)
        oracle.dbias(p, *args, b64)
    dt = time.perf_counter() - t0
    return dt, visible_pairs(ws, t["seq_q_lens"]) * flops_per_pair(ws)


def cpu_baseline_fwd(w, t, target_s=12.0):
    """The fp64 oracle forward on the first KV-head groups of every batch row."""
    import oracle

    def sample(groups):
        G = w.Hq // w.Hkv
        ws = w.with_(Hq=groups * G, Hkv=groups)
        p = _problem(ws, t["seq_q_lens"])
        a = [t["q"][:, :groups * G].contiguous().double().numpy(),
             t["k"][:, :groups].contiguous().double().numpy(),
             t["v"][:, :groups].contiguous().double().numpy()]
        t0 = time.perf_counter()
        oracle.forward(p, *a)
        return time.perf_counter() - t0, visible_pairs(ws, t["seq_q_lens"]) * fwd_flops_per_pair(ws)

    dt, fl = sample(1)
    groups = max(1, min(w.Hkv, int(target_s / max(dt, 1e-3))))
    if groups > 1:
        dt, fl = sample(groups)
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle forward of {groups} of {w.Hkv} KV-head groups x B={w.B} "
                      f"({fl / 1e9:.2f} GFLOP algorithmic in {dt:.2f} s)"}


def run_gpu_fwd(args, w, t, rank, world, device):
    """Times sdpa_fwd: one kernel per step, so the step time is the kernel's."""
    import attention_backward_sdpa_gb300 as pkg
    pkg.load()
    lens = t["seq_q_lens"]
    d = {k: t[k].to(device) for k in ("q", "k", "v")}
    lq = None if lens is None else lens.to(device)
    lk = None if t["seq_kv_lens"] is None else t["seq_kv_lens"].to(device)
    o = torch.empty((w.B, w.Hq, w.Sq, w.Dv), dtype=t["q"].dtype, device=device)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=device)
    sink = workloads.sink_logits(w).to(device) if args.sink else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    kw = dict(scale=w.resolved_scale, causal=w.causal, bottom_right=w.bottom_right,
              window_left=w.window_left, window_right=w.window_right, seq_q_lens=lq,
              seq_kv_lens=lk, sink=sink, o=o, lse=lse)
    if "bias" in t:  # sdpa_fwd_bias
        d["bias"] = t["bias"].to(device)
        kw["bias"] = d["bias"]

    def step():
        pkg.sdpa_fwd(d["q"], d["k"], d["v"], **kw)

    pairs = visible_pairs(w, None if lens is None else lens.numpy())
    flops = pairs * fwd_flops_per_pair(w)
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(device)
        pkg.check_device_status()
        barrier(world)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize(device)
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        total_ms = sum(s.elapsed_time(e) for s, e in zip(starts, ends))
        # End to end with host buffers (as in run_gpu): Q, K, V (+ bias) in, O and
        # LSE out every step; E2E_IN_FLIGHT steps in flight, and one at a time.
        host_in = {k: v.cpu().pin_memory() for k, v in d.items()}
        h2d = sum(x.numel() * x.element_size() for x in host_in.values())
        d2h = sum(x.numel() * x.element_size() for x in (o, lse))
        e2e_steps = max(3, min(args.steps, 50))

        def new_slot():
            dd = {k: torch.empty_like(v) for k, v in d.items()}
            kws = dict(kw, o=torch.empty_like(o), lse=torch.empty_like(lse))
            if "bias" in dd:
                kws["bias"] = dd["bias"]
            return {"d": dd, "outs": [kws["o"], kws["lse"]],
                    "run": lambda: pkg.sdpa_fwd(dd["q"], dd["k"], dd["v"], **kws)}

        slot0 = {"d": d, "outs": [o, lse], "run": step}
        e2e_serial_s = e2e_time(device, host_in, [slot0], e2e_steps)
        e2e_s = e2e_time(device, host_in, [slot0] + [new_slot() for _ in range(E2E_IN_FLIGHT - 1)],
                         e2e_steps)
    pkg.check_device_status()
    ms_step = max_over_ranks(total_ms / args.steps, world, device)
    e2e_s = max_over_ranks(e2e_s, world, device)
    e2e_serial_s = max_over_ranks(e2e_serial_s, world, device)
    peak_tf, peak_hbm, peak_kind = peaks()
    achieved = flops / (ms_step * 1e-3) / 1e12
    return {
        "value": world * achieved, "ms_per_step": ms_step, "flops": flops,
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                     "frac": achieved / peak_tf, "traffic": None,
                     "kernel": {256: "sdpa_fwd_wide_kernel", 192: "sdpa_fwd_shared_kernel"}.get(
                         w.Dqk, "sdpa_fwd_kernel"),
                     "peak_kind": f"{peak_kind} bf16 burst", "kernel_gflop": flops / 1e9},
        "kernel_ms": {"fwd": round(ms_step, 5)},
        "e2e": {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps_in_flight": E2E_IN_FLIGHT,
                "serial_value": world * flops / e2e_serial_s / 1e12},
        "clocks": clocks.summary(),
        "gpu_launches": args.steps,
    }


def cpu_baseline_leg(w, t, target_s=12.0):
    import oracle
    t0 = time.perf_counter()
    o, lse = oracle_forward_inputs(w, t)
    fwd_s = time.perf_counter() - t0
    dt1, f1 = oracle_backward_sample(w, t, o, lse, 1)
    groups = max(1, min(w.Hkv, int(target_s / max(dt1, 1e-3))))
    if groups > 1:
        dt, fl = oracle_backward_sample(w, t, o, lse, groups)
    else:
        dt, fl = dt1, f1
    cb = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
          "kind": "oracle",
          "sample": f"fp64 oracle backward of {groups} of {w.Hkv} KV-head groups x B={w.B} "
                    f"({fl / 1e9:.2f} GFLOP algorithmic in {dt:.2f} s); oracle forward for the "
                    f"O/LSE inputs took {fwd_s:.1f} s"}
    return o, lse, cb


# ---------------------------------------------------------------- GPU leg
# DRAM bytes per launch of the main kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of the same bench command),
# valid only for the kernel sources they were taken on: the digest covers the
# kernel's source files, and a changed kernel reports null. D_qk = 192 and 256
# run sdpa_bwd_main_ds, every other head dim sdpa_bwd_main.
MAIN_SOURCES = {"sdpa_bwd_main": ("sdpa_bwd_main.cuh", "common.cuh", "ptx.cuh", "nvfp4.cuh", "bias.cuh"),
                "sdpa_bwd_main_ds": ("sdpa_bwd_main_ds.cu", "common.cuh", "ptx.cuh", "bias.cuh")}
MAIN_TRAFFIC = {
    "d37336d80f5254fa": {"causal_gqa_det": 134370304 + 513630464,
                         "causal_mha": 103112192 + 15115008,
                         "swa_causal_padded": 228067840 + 158214912,
                         "causal_mha/bias-B-f32": 456930816 + 540702464,
                         "causal_mha/qat": 102860544 + 14223872},
    "ffd89974697c001e": {"mla_br_causal": 132089088 + 263580416,
                         "mla_br_causal/bias-B-bf16": 430743808 + 1331224064,
                         "d256_causal": 302962176 + 301679616},
}


def main_kernel_name(w, tag=None) -> str:
    return "sdpa_bwd_main_ds" if w.Dqk > 128 else "sdpa_bwd_main"


def main_traffic(w, tag=None):
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "attention_backward_sdpa_gb300", "csrc")
    blob = b"".join(open(os.path.join(csrc, f), "rb").read() for f in MAIN_SOURCES[main_kernel_name(w, tag)])
    key = w.name if tag is None else f"{w.name}/{tag}"
    return MAIN_TRAFFIC.get(hashlib.sha256(blob).hexdigest()[:16], {}).get(key)


def bias_tag(t):
    """The traffic table's key suffix: 'bias-<batch>-<dtype>' for a biased run,
    'qat' for the NVFP4 QAT backward, 'f16' for fp16 io, else None."""
    if t.get("qat"):
        return "qat"
    if t["q"].dtype == torch.float16:
        return "f16"
    b = t.get("bias")
    if b is None:
        return None
    name = {torch.float32: "f32", torch.float16: "f16"}.get(b.dtype, "bf16")
    tag = f"bias-{'shared' if b.shape[0] == 1 and t['q'].shape[0] > 1 else 'B'}-{name}"
    dbt = t.get("dbias_dtype", torch.float32)
    return tag if dbt == torch.float32 else tag + "-dbias" + {torch.float16: "f16"}.get(dbt, "bf16")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return d.get("bf16_tflops"), d.get("hbm_gbs"), "measured"
    return 1900.0, 6800.0, "fallback"


E2E_IN_FLIGHT = 2  # steps in flight in the end-to-end measurement


def e2e_time(device, host_in, slots, n_steps):
    """Wall-clock seconds per step over n_steps steps through the public API with
    host buffers. Every step copies the inputs from pinned host memory into its
    slot's device buffers, runs the step and copies the outputs back into pinned
    host memory. Step i uses slot i % len(slots), each slot on a stream of its
    own with its own buffers and workspace, so with two slots one step's copies
    overlap the other's kernels (and the link carries both directions at once),
    as a training loop that stages its next batch does; with one slot the steps
    run one after another."""
    streams = [torch.cuda.Stream(device) for _ in slots]
    outs_h = [[torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in sl["outs"]] for sl in slots]
    torch.cuda.synchronize(device)
    t0 = time.perf_counter()
    for i in range(n_steps):
        j = i % len(slots)
        sl = slots[j]
        with torch.cuda.stream(streams[j]):
            for k, v in host_in.items():
                sl["d"][k].copy_(v, non_blocking=True)
            sl["run"]()
            for h, x in zip(outs_h[j], sl["outs"]):
                h.copy_(x, non_blocking=True)
    torch.cuda.synchronize(device)
    return (time.perf_counter() - t0) / n_steps


def run_gpu(args, w, t, o, lse, rank, world, device):
    import attention_backward_sdpa_gb300 as pkg
    pkg.load()
    lens = t["seq_q_lens"]
    d = {k: t[k].to(device) for k in ("q", "k", "v", "do")}
    d["o"], d["lse"] = o.to(device), lse.to(device)
    lq = None if lens is None else lens.to(device)
    lk = None if t["seq_kv_lens"] is None else t["seq_kv_lens"].to(device)
    dq, dk, dv = torch.empty_like(d["q"]), torch.empty_like(d["k"]), torch.empty_like(d["v"])
    ws = torch.empty(max(pkg.workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv,
                                            w.deterministic, causal=w.causal,
                                            bottom_right=w.bottom_right, window_left=w.window_left,
                                            window_right=w.window_right,
                                            padded=w.padded is not None), 256),
                     dtype=torch.uint8, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.current_stream(device)
    kw = dict(scale=w.resolved_scale, causal=w.causal, bottom_right=w.bottom_right,
              window_left=w.window_left, window_right=w.window_right,
              deterministic=w.deterministic, seq_q_lens=lq, seq_kv_lens=lk, dq=dq, dk=dk, dv=dv,
              workspace=ws)

    if args.sink:  # sink tokens: the same chain plus the dsink partials and reduce
        kw["sink"] = workloads.sink_logits(w).to(device)
        kw["dsink"] = torch.empty_like(kw["sink"])
    outs = [dq, dk, dv]
    if "bias" in t:  # additive bias: read by the main kernel, dBias written by it
        d["bias"] = t["bias"].to(device)
        kw["dbias_dtype"] = t["dbias_dtype"]
        kw["dbias"] = torch.empty(tuple(t["bias"].shape), dtype=t["dbias_dtype"], device=device)
        outs.append(kw["dbias"])

    qat_ws = None
    if t.get("qat"):
        qat_ws = torch.empty(max(pkg.nvfp4_qat_workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk,
                                                              w.Dv), 256), dtype=torch.uint8,
                             device=device)

    def run_with(dd, kws, qws):
        if qws is not None:
            pkg.sdpa_bwd_nvfp4_qat(dd["q"], dd["k"], dd["v"], dd["o"], dd["do"], dd["lse"],
                                   scale=w.resolved_scale, causal=w.causal,
                                   bottom_right=w.bottom_right, window_left=w.window_left,
                                   window_right=w.window_right, seq_q_lens=lq, seq_kv_lens=lk,
                                   dq=kws["dq"], dk=kws["dk"], dv=kws["dv"], workspace=qws)
            return
        pkg.sdpa_bwd(dd["q"], dd["k"], dd["v"], dd["o"], dd["do"], dd["lse"],
                     **(dict(kws, bias=dd["bias"]) if "bias" in dd else kws))

    def step():
        run_with(d, kw, qat_ws)

    def new_slot():
        """A second set of device inputs, outputs and workspace for the e2e loop."""
        dd = {k: torch.empty_like(v) for k, v in d.items()}
        kws = dict(kw, dq=torch.empty_like(dq), dk=torch.empty_like(dk), dv=torch.empty_like(dv),
                   workspace=torch.empty_like(ws))
        outs_s = [kws["dq"], kws["dk"], kws["dv"]]
        if args.sink:
            kws["dsink"] = torch.empty_like(kw["dsink"])
        if "bias" in d:
            kws["dbias"] = torch.empty_like(kw["dbias"])
            outs_s.append(kws["dbias"])
        qws = torch.empty_like(qat_ws) if qat_ws is not None else None
        return {"d": dd, "outs": outs_s, "run": lambda: run_with(dd, kws, qws)}

    def timed_loop(n, profile=False):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        if profile:
            pkg.profile_enable(True)
        for i in range(n):
            flush.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(device)
        prof = pkg.profile_read() if profile else None
        if profile:
            pkg.profile_enable(False)
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends)), prof

    pairs = visible_pairs(w, None if lens is None else lens.numpy())
    flops = pairs * flops_per_pair(w)
    main_flops = pairs * main_kernel_flops_per_pair(w)
    with ClockSampler(device.index if device.index is not None else 0) as clocks:
        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize(device)
        pkg.check_device_status()
        barrier(world)
        torch.cuda.synchronize(device)
        total_ms, _ = timed_loop(args.steps)
        torch.cuda.synchronize(device)
        barrier(world)
        pkg.check_device_status()
        # Per-kernel durations from the library's own events on the launch stream
        # (a second pass: the events between launches disable the PDL overlap).
        _, prof = timed_loop(args.steps, profile=True)
        # End to end through the public API with host buffers: pinned host -> device
        # copies of the inputs and a device -> host read of dQ/dK/dV (+ dBias)
        # every step; E2E_IN_FLIGHT steps in flight, and one at a time.
        host_in = {k: v.cpu().pin_memory() for k, v in d.items()}
        h2d = sum(x.numel() * x.element_size() for x in host_in.values())
        d2h = sum(x.numel() * x.element_size() for x in outs)
        e2e_steps = max(3, min(args.steps, 50))
        slot0 = {"d": d, "outs": outs, "run": step}
        e2e_serial_s = e2e_time(device, host_in, [slot0], e2e_steps)
        e2e_s = e2e_time(device, host_in, [slot0] + [new_slot() for _ in range(E2E_IN_FLIGHT - 1)],
                         e2e_steps)
    pkg.check_device_status()
    ms_step = max_over_ranks(total_ms / args.steps, world, device)
    e2e_s = max_over_ranks(e2e_s, world, device)
    e2e_serial_s = max_over_ranks(e2e_serial_s, world, device)
    peak_tf, peak_hbm, peak_kind = peaks()
    main_ms = prof["main"][0] / max(prof["main"][1], 1)
    achieved = main_flops / (main_ms * 1e-3) / 1e12
    value = world * flops / (ms_step * 1e-3) / 1e12
    kernel_ms = {k: round(v[0] / max(v[1], 1), 5) for k, v in prof.items() if v[1]}
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
            "frac": achieved / peak_tf, "traffic": main_traffic(w, bias_tag(t)),
            "kernel": main_kernel_name(w, bias_tag(t)), "peak_kind": f"{peak_kind} bf16 burst",
            "kernel_gflop": main_flops / 1e9}
    if "bias" in t:
        # With a bias the main kernel streams the bias and the fp32 dBias: it is
        # bound by HBM, against the measured copy bandwidth.
        nbytes = main_kernel_bytes_bias(w, pairs, t["bias"], t["dbias_dtype"].itemsize)
        gbs = nbytes / (main_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peak_hbm, "unit": "GB/s",
                "frac": gbs / peak_hbm, "traffic": main_traffic(w, bias_tag(t)),
                "kernel": main_kernel_name(w, bias_tag(t)), "peak_kind": f"{peak_kind} HBM copy",
                "algorithmic_bytes": nbytes, "tensor_tflops": achieved,
                "tensor_frac": achieved / peak_tf}
    return {
        "value": value, "ms_per_step": ms_step, "flops": flops,
        "roofline": roof,
        "kernel_ms": kernel_ms,
        "e2e": {"value": world * flops / e2e_s / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps_in_flight": E2E_IN_FLIGHT,
                "serial_value": world * flops / e2e_serial_s / 1e12},
        "clocks": clocks.summary(),
        # preprocess + main + dQ kernel (+ the three fake quantizations with QAT,
        # + dsink with sink tokens)
        "gpu_launches": (3 + (3 if t.get("qat") else 0) + (1 if args.sink else 0)) * args.steps,
    }


def run_reference(args, w, rank, world):
    """The fp64 oracle on the host cores, bounded samples of the workload per step."""
    if rank != 0:
        return
    import oracle
    t = workloads.generate(w)
    o, lse = oracle_forward_inputs(w, t)
    times, fl = [], 0
    for i in range(args.warmup + args.steps):
        dt, fl = oracle_backward_sample(w, t, o, lse, 1)
        if i >= args.warmup:
            times.append(dt)
    dt = sum(times) / len(times)
    v = fl / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H_q": w.Hq, "H_kv": w.Hkv, "S_q": w.Sq,
                       "S_kv": w.Skv, "D_qk": w.Dqk, "D_v": w.Dv, "causal": w.causal,
                       "bottom_right": w.bottom_right, "window_left": w.window_left,
                       "deterministic": w.deterministic,
                       "sample": "first KV-head group of every batch row per step"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"fp64 oracle backward of 1 of {w.Hkv} KV-head groups "
                                       f"x B={w.B} per step ({fl / 1e9:.2f} GFLOP)"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--sink", action="store_true",
                    help="time sdpa_bwd_sink (sink-token logits, dsink output) instead of sdpa_bwd")
    ap.add_argument("--bias", default="none", choices=["none", "B", "1"],
                    help="add a bias of B batches or 1 shared batch: sdpa_bwd_bias (dBias written "
                         "in fp32), or sdpa_fwd_bias with --pass fwd")
    ap.add_argument("--bias-dtype", default="bf16", choices=["bf16", "f16", "f32"])
    ap.add_argument("--dbias-dtype", default="f32", choices=["f32", "bf16", "f16"],
                    help="element type of the dBias output (bf16/f16: the io-type dBias)")
    ap.add_argument("--io", default="bf16", choices=["bf16", "f16"],
                    help="element type of Q, K, V, O, dO and the gradients (f16: sdpa_bwd_typed)")
    ap.add_argument("--qat", action="store_true",
                    help="time sdpa_bwd_nvfp4_qat (NVFP4 fake-quantized Q/K/V, P fake-quantized "
                         "for dV; D = 128, non-deterministic)")
    ap.add_argument("--pass", dest="pass_", default="bwd", choices=["bwd", "fwd"],
                    help="bwd: the backward chain (default); fwd: sdpa_fwd, the forward (O, LSE)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the oracle backward (O/LSE still come from the oracle forward)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    args.steps = max(args.steps, 1)
    w = workloads.WORKLOADS[args.workload]
    # option checks first: no process group or device is touched for a bad line
    if args.io == "f16" and args.qat:
        ap.error("--io f16: QAT needs bf16")
    if args.qat and (w.Dqk != 128 or w.Dv != 128 or w.deterministic or args.bias != "none"
                     or args.sink or args.pass_ != "bwd"):
        ap.error("--qat: a D = 128 non-deterministic workload, backward, no bias or sink")
    rank, world, local = init_dist()
    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return 0
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    io = torch.float16 if args.io == "f16" else torch.bfloat16
    t = workloads.generate(w, io)
    if args.qat:
        t["qat"] = True
    if args.bias != "none":
        dts = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
        t["bias"] = workloads.bias_tensor(w, 1 if args.bias == "1" else w.B, dts[args.bias_dtype])
        t["dbias_dtype"] = dts[args.dbias_dtype]
    if args.pass_ == "fwd":
        cb = cpu_baseline_fwd(w, t) if (rank == 0 and not args.no_cpu_baseline) else None
        r = run_gpu_fwd(args, w, t, rank, world, device)
        if rank == 0:
            print(json.dumps(result_line(args, w, world, r, cb, METRIC_FWD)), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    o = torch.empty((w.B, w.Hq, w.Sq, w.Dv), dtype=io)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32)
    cb = None
    if rank == 0:
        if args.no_cpu_baseline:
            o, lse = oracle_forward_inputs(w, t)
        else:
            o, lse, cb = cpu_baseline_leg(w, t)
    if world > 1:
        o_d, l_d = o.to(device), lse.to(device)
        broadcast_tensor(o_d, world)
        broadcast_tensor(l_d, world)
        o, lse = o_d.cpu(), l_d.cpu()
    r = run_gpu(args, w, t, o, lse, rank, world, device)
    if rank == 0:
        print(json.dumps(result_line(args, w, world, r, cb, METRIC)), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def result_line(args, w, world, r, cb, metric):
    """The JSON line of a GPU run (rank 0)."""
    return {"metric": metric, "value": r["value"], "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": args.io,
            "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H_q": w.Hq, "H_kv": w.Hkv, "S_q": w.Sq,
                       "S_kv": w.Skv, "D_qk": w.Dqk, "D_v": w.Dv, "causal": w.causal,
                       "bottom_right": w.bottom_right, "window_left": w.window_left,
                       "deterministic": w.deterministic, "seed": w.seed,
                       "pass": args.pass_, "sink": bool(args.sink), "nvfp4_qat": bool(args.qat),
                       "bias": None if args.bias == "none" else
                       {"batch": args.bias, "dtype": args.bias_dtype, "dbias": args.dbias_dtype},
                       "gflop_per_step": r["flops"] / 1e9,
                       "l2": "256 MiB buffer written between timed steps",
                       "parallelism": f"replicas{world}" if world > 1 else "single"},
            "roofline": r["roofline"], "cpu_baseline": cb, "e2e": r["e2e"],
            "gpu_launches": r["gpu_launches"], "kernel_ms": r["kernel_ms"],
            "clocks": r["clocks"]}


if __name__ == "__main__":
    sys.exit(main())
