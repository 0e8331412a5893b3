"""The allocation-free entry point (sdpa_bwd_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory where they run the
backward (for example a plugin of a framework that owns the whole device
memory pool). Its scratch is a fixed 16 MiB array inside the library, so these
checks make two calls in a row on different problems (the array keeps the
previous call's contents) and compare each with the workspace-taking
sdpa_bwd on the same inputs, within the parity tolerance of the other tests.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import workloads
from harness import assert_close, make_case, to_device

pytestmark = pytest.mark.gpu

W = workloads.Workload
SDPA_ERR_WORKSPACE = 4
LIMIT_BYTES = 16 << 20


def _lib():
    import attention_backward_sdpa_gb300 as pkg
    lib = pkg.load(build_if_missing=True)
    vp, i = ctypes.c_void_p, ctypes.c_int
    lib.sdpa_bwd_noalloc.argtypes = [vp] * 9 + [i] * 7 + [ctypes.c_float] + [i] * 5 + [vp, vp, vp]
    lib.sdpa_bwd_noalloc.restype = i
    return lib, pkg


def _call_noalloc(lib, w, d, outs):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sdpa_bwd_noalloc(p(d["q"]), p(d["k"]), p(d["v"]), p(d["o"]), p(d["do"]),
                                p(d["lse"]), p(outs[0]), p(outs[1]), p(outs[2]), w.B, w.Hq, w.Hkv,
                                w.Sq, w.Skv, w.Dqk, w.Dv, ctypes.c_float(w.resolved_scale),
                                int(w.causal), int(w.bottom_right), w.window_left, w.window_right,
                                int(w.deterministic), p(d["seq_q_lens"]), p(d["seq_kv_lens"]),
                                stream)


CASES = [
    W("noalloc_gqa", 1, 4, 2, 384, 384, 128, 128, causal=True, window_left=200, seed=31),
    W("noalloc_padded", 2, 2, 2, 300, 300, 64, 64, causal=True, bottom_right=True,
      padded=(100, 300), deterministic=True, seed=32),
]


def test_noalloc_matches_sdpa_bwd_on_two_calls_in_a_row():
    lib, pkg = _lib()
    for w in CASES:
        assert pkg.workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv, w.deterministic) \
            <= LIMIT_BYTES
    cases = [make_case(w) for w in CASES]
    devs = [to_device(c) for c in cases]
    for w, d in zip(CASES, devs):  # two calls in a row, different problems
        outs = [torch.full_like(d["q"], float("nan")), torch.full_like(d["k"], float("nan")),
                torch.full_like(d["v"], float("nan"))]
        assert _call_noalloc(lib, w, d, outs) == 0
        pkg.check_device_status()
        ref = pkg.sdpa_bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"],
                           scale=w.resolved_scale, causal=w.causal, bottom_right=w.bottom_right,
                           window_left=w.window_left, window_right=w.window_right,
                           deterministic=w.deterministic, seq_q_lens=d["seq_q_lens"],
                           seq_kv_lens=d["seq_kv_lens"])
        torch.cuda.synchronize()
        for name, g, r in zip(("dq", "dk", "dv"), outs, ref):
            assert_close(name, g.double().cpu().numpy(), r.double().cpu().numpy())


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib, pkg = _lib()
    w = W("too_big", 2, 16, 16, 2048, 2048, 128, 128, causal=True)
    assert pkg.workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv) > LIMIT_BYTES
    fake = {k: None for k in ("seq_q_lens", "seq_kv_lens")}
    buf = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    for k in ("q", "k", "v", "o", "do"):
        fake[k] = buf
    fake["lse"] = torch.empty(4, dtype=torch.float32, device="cuda")
    assert _call_noalloc(lib, w, fake, [buf, buf, buf]) == SDPA_ERR_WORKSPACE
