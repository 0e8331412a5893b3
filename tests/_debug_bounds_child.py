"""Child process of test_debug_bounds.py: runs shapes on every dQ route and
both forward kernels through the debug-bounds library (selected by
SDPA_BWD_LIBRARY before the binding loads it), checks that no kernel reported
an out-of-range access and that the gradients, O and LSE match the fp64 oracle.
Not collected by pytest on its own."""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

import torch  # noqa: E402

import attention_backward_sdpa_gb300 as pkg  # noqa: E402
import workloads  # noqa: E402
from harness import assert_close, gpu_backward, make_case, oracle_backward, to_device  # noqa: E402
from test_parity_gpu import _check_fwd, _gpu_fwd  # noqa: E402

W = workloads.Workload
SHAPES = [
    W("one_query", 1, 2, 2, 1, 70, 64, 64, seed=81),                                  # a single row
    W("dense_65", 1, 2, 1, 65, 65, 128, 128, seed=82),                                # reduction route, ragged
    W("causal_127_d96", 2, 2, 2, 127, 127, 96, 96, causal=True, seed=83),             # zero-filled columns
    W("window_129_det", 1, 4, 2, 129, 129, 128, 128, causal=True, window_left=50,
      deterministic=True, seed=84),                                                   # two-kernel route, band
    W("padded_relay", 2, 2, 2, 200, 200, 64, 64, causal=True, padded=(1, 200),
      deterministic=True, seed=85),                                                   # ordered relay
    W("mla_br", 1, 2, 2, 150, 200, 192, 128, causal=True, bottom_right=True, seed=86),  # D_qk 192
    W("gqa_partials_det", 1, 8, 2, 300, 300, 128, 128, causal=True, deterministic=True,
      seed=87),                                                                       # partial dK/dV sets
    W("padded_br_det", 2, 2, 2, 190, 260, 128, 128, causal=True, bottom_right=True,
      padded=(1, 260), deterministic=True, seed=88),                                  # full-rectangle band
    W("d256_gqa_window", 2, 4, 2, 140, 200, 256, 256, causal=True, window_left=60,
      padded=(1, 140), seed=89),                                                      # D 256, half-column units
]

assert pkg.library_path() == os.environ["SDPA_BWD_LIBRARY"]
for w in SHAPES:
    case = make_case(w)
    res = gpu_backward(case)  # raises SdpaError on SDPA_ERR_BOUNDS or SDPA_ERR_TIMEOUT
    torch.cuda.synchronize()
    for name, g, r in zip(("dq", "dk", "dv"), res, oracle_backward(case)):
        assert_close(f"{w.name} {name}", g.double().cpu().numpy(), r)
    o, lse = _gpu_fwd(case, to_device(case))  # checks the status word too
    _check_fwd(case, o, lse)
    print("ok", w.name, flush=True)
print("DEBUG_BOUNDS_OK", len(SHAPES))
