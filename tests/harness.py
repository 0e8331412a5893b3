"""Shared helpers of the parity tests: seeded inputs, oracle forward/backward,
the GPU call through the C ABI, and the tolerance check."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Parity bar for bf16 I/O with fp32 accumulation, per gradient tensor.
REL_FRO_TOL = 1e-2
MAX_ABS_TOL = 3e-2  # times max|ref|


def problem_of(w: workloads.Workload, lens=None) -> oracle.Problem:
    return oracle.Problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv, scale=w.resolved_scale,
                          causal=w.causal, bottom_right=w.bottom_right,
                          window_left=w.window_left, window_right=w.window_right,
                          seq_q_lens=None if lens is None else lens.numpy(),
                          seq_kv_lens=None if lens is None else lens.numpy())


def f64(x: torch.Tensor) -> np.ndarray:
    return x.double().numpy()


def make_case(w: workloads.Workload, sink: bool = False, bias=None, io=torch.bfloat16):
    """Seeded inputs plus O (bf16) and LSE (fp32) from the oracle forward; with
    ``sink`` the forward takes the workload's sink logits (case["sink"]); with
    ``bias`` = (batch, dtype) an additive bias of that batch (1 or B) and element
    type (case["bias"]), which the oracle sees exactly as the GPU does. ``io``
    is the element type of Q, K, V, dO and O (bf16 or fp16)."""
    t = workloads.generate(w, io)
    t["sink"] = workloads.sink_logits(w) if sink else None
    t["bias"] = None if bias is None else workloads.bias_tensor(w, bias[0], bias[1])
    p = oracle.Problem(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv, scale=w.resolved_scale,
                       causal=w.causal, bottom_right=w.bottom_right, window_left=w.window_left,
                       window_right=w.window_right,
                       seq_q_lens=None if t["seq_q_lens"] is None else t["seq_q_lens"].numpy(),
                       seq_kv_lens=None if t["seq_kv_lens"] is None else t["seq_kv_lens"].numpy())
    o64, lse64 = oracle.forward(p, f64(t["q"]), f64(t["k"]), f64(t["v"]),
                                None if t["sink"] is None else t["sink"].double().numpy(),
                                bias=None if t["bias"] is None else f64(t["bias"]))
    t["o"] = torch.from_numpy(o64).to(io)
    t["lse"] = torch.from_numpy(lse64).float()
    t["problem"] = p
    t["workload"] = w
    return t


def _bias64(case):
    return None if case.get("bias") is None else f64(case["bias"])


def oracle_backward(case):
    p = case["problem"]
    return oracle.backward(p, f64(case["q"]), f64(case["k"]), f64(case["v"]), f64(case["o"]),
                           f64(case["do"]), case["lse"].double().numpy(), bias=_bias64(case))


def oracle_dbias(case, rows=None):
    """dBias from the bf16 inputs and fp32 LSE the GPU sees: in full, or at the
    flat bias rows ``rows`` ((bb * Hq + h) * Sq + q) as a (len(rows), Skv) array."""
    p = case["problem"]
    args = (p, f64(case["q"]), f64(case["k"]), f64(case["v"]), f64(case["o"]), f64(case["do"]),
            case["lse"].double().numpy(), _bias64(case))
    return oracle.dbias(*args) if rows is None else oracle.dbias_rows(*args, rows)


def oracle_dsink(case):
    """(dsink, sum of |terms|) per head from the bf16 O / dO and fp32 LSE the GPU sees."""
    p = case["problem"]
    lse = case["lse"].double().numpy()
    dl = oracle.delta(p, f64(case["o"]), f64(case["do"]))
    sink = case["sink"].double().numpy()
    ds = oracle.dsink(p, sink, lse, dl)
    mag = oracle.dsink(p, sink, lse, np.abs(dl))  # -sum of |terms|
    return ds, -mag


def oracle_sampled(case, q_rows, kv_rows):
    p = case["problem"]
    return oracle.backward_sampled(p, f64(case["q"]), f64(case["k"]), f64(case["v"]),
                                   f64(case["o"]), f64(case["do"]), case["lse"].double().numpy(),
                                   q_rows, kv_rows, bias=_bias64(case))


def to_device(case, dev="cuda"):
    d = {k: case[k].to(dev) for k in ("q", "k", "v", "o", "do", "lse")}
    d["sink"] = None if case.get("sink") is None else case["sink"].to(dev)
    d["bias"] = None if case.get("bias") is None else case["bias"].to(dev)
    for k in ("seq_q_lens", "seq_kv_lens"):
        d[k] = None if case[k] is None else case[k].to(dev)
    return d


def gpu_backward(case, dev_tensors=None, poison=True, **overrides):
    import attention_backward_sdpa_gb300 as pkg
    w = case["workload"]
    d = dev_tensors or to_device(case)
    outs = {}
    if poison:  # every output element must be written by the library
        outs = {"dq": torch.full_like(d["q"], float("nan")),
                "dk": torch.full_like(d["k"], float("nan")),
                "dv": torch.full_like(d["v"], float("nan"))}
    kw = dict(scale=w.resolved_scale, causal=w.causal, bottom_right=w.bottom_right,
              window_left=w.window_left, window_right=w.window_right,
              deterministic=w.deterministic, seq_q_lens=d["seq_q_lens"],
              seq_kv_lens=d["seq_kv_lens"])
    kw.update(overrides)
    res = pkg.sdpa_bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"], **kw, **outs)
    pkg.check_device_status()
    return res


def errors(gpu: np.ndarray, ref: np.ndarray):
    """(relative Frobenius error, max abs error / max|ref|)."""
    diff = gpu - ref
    nref = np.linalg.norm(ref)
    mref = np.abs(ref).max() if ref.size else 0.0
    rel = np.linalg.norm(diff) / nref if nref > 0 else np.linalg.norm(diff)
    mx = np.abs(diff).max() / mref if mref > 0 else (np.abs(diff).max() if diff.size else 0.0)
    return float(rel), float(mx)


def assert_close(name, gpu: np.ndarray, ref: np.ndarray):
    assert np.all(np.isfinite(gpu)), f"{name}: non-finite values in GPU output"
    rel, mx = errors(gpu, ref)
    assert rel <= REL_FRO_TOL and mx <= MAX_ABS_TOL, \
        f"{name}: rel_fro={rel:.3e} (<= {REL_FRO_TOL}), max_abs/max|ref|={mx:.3e} (<= {MAX_ABS_TOL})"
    return rel, mx
