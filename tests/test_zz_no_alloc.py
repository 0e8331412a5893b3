"""The allocation-free entry point (sdpa_bwd_noalloc), called through the C ABI.

It serves callers that cannot allocate device memory where they run the
backward (for example a plugin of a framework that owns the whole device
memory pool). Its scratch is a fixed 16 MiB array inside the library, shared
by every call and keeping what the previous call left. So the check makes a
series of calls in a row on different problems, one per dQ route that carves
its scratch from the array (the fp32 accumulator of the reduction route, the
ordered relay's counters, the stored dS tiles and the zero tile of the
two-kernel route at head dims 128, 192 and 256, the GQA partial sets), each after a larger call has left
stale data in the array. Each result is compared with the fp64 oracle and with
the workspace-taking sdpa_bwd on the same inputs, within the parity tolerance
of the other tests; deterministic calls must equal sdpa_bwd bit for bit.
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

import workloads
from harness import assert_close, make_case, oracle_backward, to_device

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


# In call order. The first fills half the array, so every later call starts
# from another call's leftovers.
CASES = [
    # reduction route (fp32 dQ accumulator), GQA with a sliding window
    W("noalloc_gqa", 1, 8, 2, 1000, 1000, 128, 128, causal=True, window_left=300, seed=31),
    # ordered relay (D 64, deterministic): turn counters and the accumulator
    W("noalloc_padded", 2, 2, 2, 300, 300, 64, 64, causal=True, bottom_right=True,
      padded=(100, 300), deterministic=True, seed=32),
    # two-kernel route (D 128, deterministic): the band of stored dS tiles, the
    # zero tile, GQA partial sets
    W("noalloc_det128", 1, 4, 2, 320, 320, 128, 128, causal=True, deterministic=True, seed=33),
    # two-kernel route at D_qk 192 / D_v 128: stored dS tiles, GQA partial sets
    W("noalloc_mla", 1, 4, 2, 260, 260, 192, 128, causal=True, bottom_right=True, seed=34),
    # the reduction route once more (D 64), after the dS calls
    W("noalloc_dense", 1, 2, 1, 200, 330, 64, 64, seed=35),
    # head dim 256: stored dS tiles of the half-column units, GQA partial sets
    W("noalloc_d256", 1, 4, 2, 200, 200, 256, 256, causal=True, window_left=90, seed=36),
]


def test_noalloc_matches_oracle_and_sdpa_bwd_on_calls_in_a_row():
    lib, pkg = _lib()
    for w in CASES:
        assert pkg.workspace_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv, w.deterministic,
                                  causal=w.causal, bottom_right=w.bottom_right,
                                  window_left=w.window_left, window_right=w.window_right,
                                  padded=w.padded is not None) <= LIMIT_BYTES
    cases = [make_case(w) for w in CASES]
    devs = [to_device(c) for c in cases]
    for rep in range(2):  # the whole series twice: every call follows another
        for w, c, d in zip(CASES, cases, devs):
            outs = [torch.full_like(d["q"], float("nan")), torch.full_like(d["k"], float("nan")),
                    torch.full_like(d["v"], float("nan"))]
            assert _call_noalloc(lib, w, d, outs) == 0, w.name
            pkg.check_device_status()
            ref = pkg.sdpa_bwd(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"],
                               scale=w.resolved_scale, causal=w.causal,
                               bottom_right=w.bottom_right, window_left=w.window_left,
                               window_right=w.window_right, deterministic=w.deterministic,
                               seq_q_lens=d["seq_q_lens"], seq_kv_lens=d["seq_kv_lens"])
            torch.cuda.synchronize()
            exact = oracle_backward(c)
            for name, g, r, e in zip(("dq", "dk", "dv"), outs, ref, exact):
                g64 = g.double().cpu().numpy()
                assert_close(f"{w.name} {name} vs oracle", g64, e)
                assert_close(f"{w.name} {name} vs sdpa_bwd", g64, r.double().cpu().numpy())
                if w.deterministic:
                    assert torch.equal(g, r), f"{w.name} {name}: not bitwise equal to sdpa_bwd"


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
