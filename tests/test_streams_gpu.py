"""Calls in flight on two streams at once (GPU).

A training loop that stages its next batch while the current one computes has
two calls in flight on two streams. Each backward call owns its workspace
(allocated in stream order when none is given) and each forward launch its own
ticket slot, so a call's results must not depend on what runs beside it: the
same bits as the call made alone (the deterministic and stored-dS backward
routes, and the forward, whose rows each come from one CTA), and the oracle's
values on the dQ-reduction route, whose adds may land in any order.
"""
import pytest
import torch

import workloads
from harness import assert_close, gpu_backward, make_case, oracle_backward, to_device

pytestmark = pytest.mark.gpu

W = workloads.Workload
CASES = [
    W("streams_det", 2, 4, 2, 300, 300, 128, 128, causal=True, deterministic=True, seed=120),
    W("streams_reduction", 2, 4, 4, 333, 333, 64, 64, causal=True, window_left=100, seed=121),
    W("streams_d256", 1, 4, 2, 260, 260, 256, 256, causal=True, bottom_right=True, seed=122),
    W("streams_mla", 1, 4, 2, 300, 280, 192, 128, causal=True, window_left=120, seed=123),
]


def _mask_kw(w, d):
    return dict(scale=w.resolved_scale, causal=w.causal, bottom_right=w.bottom_right,
                window_left=w.window_left, window_right=w.window_right,
                seq_q_lens=d["seq_q_lens"], seq_kv_lens=d["seq_kv_lens"])


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_backward_calls_on_two_streams(w):
    import attention_backward_sdpa_gb300 as pkg
    case = make_case(w)
    d = to_device(case)
    alone = [t.clone() for t in gpu_backward(case, d)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    torch.cuda.synchronize()
    results = []
    for rep in range(2):
        for s in streams:
            with torch.cuda.stream(s):
                results.append(pkg.sdpa_bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"],
                                            deterministic=w.deterministic, **_mask_kw(w, d)))
    torch.cuda.synchronize()
    pkg.check_device_status()
    exact = w.deterministic or w.Dqk > 128
    for outs in results:
        for name, g, a, r in zip(("dq", "dk", "dv"), outs, alone, oracle_backward(case)):
            assert_close(f"{w.name} {name}", g.double().cpu().numpy(), r)
            if exact:
                assert torch.equal(g.view(torch.int16), a.view(torch.int16)), name


@pytest.mark.parametrize("w", [CASES[0], CASES[2], CASES[3]], ids=lambda w: w.name)
def test_forward_calls_on_two_streams(w):
    """One case per forward kernel (each takes tickets from counters of its own)."""
    import attention_backward_sdpa_gb300 as pkg
    from test_parity_gpu import _check_fwd
    case = make_case(w)
    d = to_device(case)
    o0, lse0 = pkg.sdpa_fwd(d["q"], d["k"], d["v"], **_mask_kw(w, d))
    torch.cuda.synchronize()
    _check_fwd(case, o0, lse0)
    streams = [torch.cuda.Stream() for _ in range(2)]
    results = []
    for rep in range(3):
        for s in streams:
            with torch.cuda.stream(s):
                results.append(pkg.sdpa_fwd(d["q"], d["k"], d["v"], **_mask_kw(w, d)))
    torch.cuda.synchronize()
    pkg.check_device_status()
    for o, lse in results:
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
        assert torch.equal(lse, lse0)
