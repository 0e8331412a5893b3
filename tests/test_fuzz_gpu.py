"""Seeded random sweep of the backward against the fp64 oracle (GPU).

The SDPA agent guide page ("Hard rules") records a tensor-memory race that was
found only by fuzzing masked configurations. These cases draw shapes and masks
at random from a fixed seed: sequence lengths that are not tile multiples,
S_q != S_kv, causal in both alignments, left and right windows, per-batch
lengths (including empty rows), GQA/MQA ratios, every served head-dim pair
both io types and both determinism modes. Every element of dQ/dK/dV is
compared with the oracle at the parity bar; outputs are NaN-poisoned, so an
element left unwritten fails.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import assert_close, gpu_backward, make_case, oracle_backward

pytestmark = pytest.mark.gpu

N_CASES = 24
HEAD_DIMS = [(64, 64), (128, 128), (192, 128), (32, 32), (96, 96), (8, 8), (256, 256)]


def _draw(i):
    rng = np.random.default_rng(1000 + i)
    Dqk, Dv = HEAD_DIMS[int(rng.integers(len(HEAD_DIMS)))]
    Hkv = int(rng.integers(1, 3))
    G = int(rng.choice([1, 2, 3, 4]))
    B = int(rng.integers(1, 3))
    Sq = int(rng.integers(1, 420))
    Skv = int(rng.integers(1, 420)) if rng.random() < 0.5 else Sq
    causal = bool(rng.random() < 0.7)
    kw = dict(causal=causal, bottom_right=bool(rng.random() < 0.5),
              window_left=int(rng.integers(0, 300)) if rng.random() < 0.4 else -1,
              window_right=int(rng.integers(0, 80)) if causal and rng.random() < 0.3 else -1,
              deterministic=bool(rng.random() < 0.4), seed=2000 + i)
    if rng.random() < 0.4:
        lo = int(rng.integers(0, min(Sq, Skv) + 1))
        if Sq == Skv:
            kw["padded"] = (lo, Sq)
    w = workloads.Workload(f"fuzz{i}", B, G * Hkv, Hkv, Sq, Skv, Dqk, Dv, **kw)
    io = torch.float16 if rng.random() < 0.25 else torch.bfloat16
    return w, io


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_backward_parity(i):
    w, io = _draw(i)
    case = make_case(w, io=io)
    dq, dk, dv = gpu_backward(case)  # the binding takes the io type from the tensors
    torch.cuda.synchronize()
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), oracle_backward(case)):
        assert_close(f"{w} {name}", g.double().cpu().numpy(), r)


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_forward_parity(i):
    """The forward on the same draws: O at the parity bar, LSE within 1e-3 (natural
    log units, relative to its magnitude), -inf exactly on rows with no key."""
    from test_parity_gpu import _check_fwd, _gpu_fwd
    from harness import to_device
    w, io = _draw(i)
    case = make_case(w, io=io)
    o, lse = _gpu_fwd(case, to_device(case))
    _check_fwd(case, o, lse)
