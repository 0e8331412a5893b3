"""Head dim 256 (D_qk = D_v = 256) against the fp64 oracle (GPU).

The pages list 256 among the served head sizes ("SDPA Backward (SM120)",
"Head-size support and tile configs"). Here dK and dV alone would fill tensor
memory, so the main kernel's work units each accumulate one half of their
columns (both halves recompute S and dP over the full head dim) and dQ comes
from the stored dS tiles (the two-kernel route, deterministic by construction).
The cases cover both causal alignments with S_q != S_kv, GQA partial sets, a
left window with per-batch lengths, a right band, fp16 io, a bias with its
dBias, a sink with dsink, a full-size shape on sampled rows, and bitwise
reproducibility. Every output element is compared (NaN-poisoned before the call).
The forward at this size runs on its own kernel (one O accumulator shared by
the two softmax warpgroups, which agree on each row's reference every tile); it
is checked on the same cases, with sinks, biases, fp16 io, the full-size shape
and a forward-then-backward step.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import (assert_close, gpu_backward, make_case, oracle_backward, oracle_dbias,
                     oracle_dsink, to_device)

pytestmark = pytest.mark.gpu

W = workloads.Workload

CASES = {
    "d256_br_causal_long_kv": W("d256_br_causal_long_kv", 1, 2, 2, 200, 333, 256, 256, causal=True,
                                bottom_right=True, seed=90),
    "d256_tl_causal_long_q": W("d256_tl_causal_long_q", 1, 2, 2, 333, 200, 256, 256, causal=True,
                               seed=91),
    "d256_dense_gqa": W("d256_dense_gqa", 2, 4, 2, 190, 250, 256, 256, seed=92),
    "d256_padded_window": W("d256_padded_window", 2, 2, 2, 300, 300, 256, 256, causal=True,
                            window_left=100, padded=(40, 300), seed=93),
    "d256_band_right_det": W("d256_band_right_det", 1, 3, 1, 260, 260, 256, 256, causal=True,
                             window_right=50, deterministic=True, seed=94),
    "d256_single_query": W("d256_single_query", 1, 2, 2, 1, 300, 256, 256, causal=True,
                           bottom_right=True, seed=95),
}


def _compare(case, outs):
    for name, g, r in zip(("dq", "dk", "dv"), outs, oracle_backward(case)):
        assert_close(f"{case['workload'].name} {name}", g.double().cpu().numpy(), r)


@pytest.mark.parametrize("name", sorted(CASES))
def test_d256_parity(name):
    case = make_case(CASES[name])
    _compare(case, gpu_backward(case))


def test_d256_padded_rows_are_exact_zeros_and_bitwise():
    case = make_case(CASES["d256_padded_window"])
    d = to_device(case)
    first = [t.clone() for t in gpu_backward(case, d)]
    _compare(case, first)
    for b, L in enumerate(case["seq_q_lens"].tolist()):
        for t in first:
            assert torch.all(t[b, :, L:] == 0)
    for _ in range(9):
        again = gpu_backward(case, d)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("name", ["d256_br_causal_long_kv", "d256_dense_gqa"])
def test_d256_f16_parity(name):
    case = make_case(CASES[name], io=torch.float16)
    outs = gpu_backward(case)
    assert outs[0].dtype == torch.float16
    _compare(case, outs)


@pytest.mark.parametrize("kind,dtype", [("B", torch.bfloat16), ("1", torch.float32)])
def test_d256_bias_parity(kind, dtype):
    w = CASES["d256_dense_gqa"] if kind == "1" else CASES["d256_padded_window"]
    case = make_case(w, bias=(1 if kind == "1" else w.B, dtype))
    d = to_device(case)
    dbias = torch.full(tuple(d["bias"].shape), float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv, db = gpu_backward(case, d, bias=d["bias"], dbias=dbias)
    _compare(case, (dq, dk, dv))
    assert_close("dbias", db.double().cpu().numpy(), oracle_dbias(case))


def test_d256_sink_parity():
    from test_parity_gpu import _dsink_close
    case = make_case(CASES["d256_tl_causal_long_q"], sink=True)
    d = to_device(case)
    dq, dk, dv, dsink = gpu_backward(case, d, sink=d["sink"])
    _compare(case, (dq, dk, dv))
    ref, mag = oracle_dsink(case)
    _dsink_close(dsink.double().cpu().numpy(), ref, mag)


def test_d256_full_size_sampled():
    """The benchmark's head-dim-256 shape (B1 H16 S4096, causal) on sampled rows."""
    from test_parity_gpu import _sampled_check
    _sampled_check(make_case(workloads.WORKLOADS["d256_causal"]))


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("sink", [False, True])
def test_d256_forward_parity(name, sink):
    from test_parity_gpu import _check_fwd, _gpu_fwd
    case = make_case(CASES[name], sink=sink)
    o, lse = _gpu_fwd(case, to_device(case))
    _check_fwd(case, o, lse)


@pytest.mark.parametrize("kind,dtype", [("B", torch.bfloat16), ("1", torch.float32), ("B", torch.float16)])
def test_d256_forward_bias_parity(kind, dtype):
    from test_parity_gpu import _check_fwd, _gpu_fwd
    w = CASES["d256_dense_gqa"] if kind == "1" else CASES["d256_padded_window"]
    case = make_case(w, bias=(1 if kind == "1" else w.B, dtype))
    o, lse = _gpu_fwd(case, to_device(case))
    _check_fwd(case, o, lse)


def test_d256_forward_f16_io_with_bias():
    """fp16 io and an fp16 bias: the one forward variant the cases above leave out."""
    from test_parity_gpu import _check_fwd, _gpu_fwd
    w = CASES["d256_dense_gqa"]
    case = make_case(w, bias=(w.B, torch.float16), io=torch.float16)
    o, lse = _gpu_fwd(case, to_device(case))
    assert o.dtype == torch.float16
    _check_fwd(case, o, lse)


@pytest.mark.parametrize("name", ["d256_br_causal_long_kv", "d256_padded_window"])
def test_d256_forward_f16_parity(name):
    from test_parity_gpu import _check_fwd, _gpu_fwd
    case = make_case(CASES[name], io=torch.float16)
    o, lse = _gpu_fwd(case, to_device(case))
    assert o.dtype == torch.float16
    _check_fwd(case, o, lse)


def test_d256_forward_full_size_sampled_and_bitwise():
    """The benchmark's head-dim-256 shape: sampled rows against the oracle, and
    the same bits on a second call (each item's rows come from one CTA)."""
    from test_parity_gpu import _check_fwd, _gpu_fwd
    w = workloads.WORKLOADS["d256_causal"]
    case = make_case(w)
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    rng = np.random.default_rng(w.seed + 7)
    rows = np.unique(rng.integers(0, w.B * w.Hq * w.Sq, 4096))
    _check_fwd(case, o, lse, rows)
    o2, lse2 = _gpu_fwd(case, d)
    assert torch.equal(o.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(lse, lse2)


def test_d256_forward_then_backward():
    """A training step at head dim 256: the GPU forward's O/LSE into the GPU
    backward, against the oracle backward of the same O/LSE."""
    from test_parity_gpu import _gpu_fwd
    case = make_case(CASES["d256_padded_window"])
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    case["o"], case["lse"] = o.cpu(), lse.cpu()
    _compare(case, gpu_backward(case))
