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


def test_d256_forward_is_refused():
    """The forward kernel serves D_v up to 128: at 256 the call is refused."""
    import attention_backward_sdpa_gb300 as pkg
    case = make_case(CASES["d256_dense_gqa"])
    d = to_device(case)
    with pytest.raises(pkg.SdpaError) as err:
        pkg.sdpa_fwd(d["q"], d["k"], d["v"])
    assert err.value.code == 2  # SDPA_ERR_UNSUPPORTED
