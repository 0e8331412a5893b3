"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Small cases compare every element of dQ/dK/dV; they span several 128-row tiles
with ragged tails and cover each mask kind, GQA/MQA, both causal alignments,
S_q != S_kv, padding (including empty batch rows) and the deterministic relay.
The five benchmark workloads run at full size and are compared on sampled rows
that the oracle computes one by one. Outputs are NaN-poisoned before every call,
so an element the library fails to write fails the test.
"""
import numpy as np
import pytest
import torch

import workloads
from harness import (assert_close, errors, gpu_backward, make_case, oracle_backward,
                     oracle_dbias, oracle_dsink, oracle_sampled, to_device)

pytestmark = pytest.mark.gpu

W = workloads.Workload


def _full_compare(w):
    case = make_case(w)
    dq, dk, dv = gpu_backward(case)
    ref = oracle_backward(case)
    res = {}
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        res[name] = assert_close(name, g.double().cpu().numpy(), r)
    return case, (dq, dk, dv), ref


SMALL = {
    "tiny_dense": workloads.WORKLOADS["tiny_dense"],
    "tiny_causal": workloads.WORKLOADS["tiny_dense"].with_(causal=True),
    "d128_causal_ragged": W("d128_causal_ragged", 1, 2, 2, 300, 300, 128, 128, causal=True, seed=10),
    "d128_dense_ragged": W("d128_dense_ragged", 2, 2, 2, 190, 250, 128, 128, seed=11),
    "br_causal_long_kv": W("br_causal_long_kv", 1, 2, 2, 200, 333, 128, 128, causal=True,
                           bottom_right=True, seed=12),
    "br_causal_long_q": W("br_causal_long_q", 1, 2, 2, 333, 200, 128, 128, causal=True,
                          bottom_right=True, seed=13),
    "tl_causal_long_q": W("tl_causal_long_q", 1, 2, 2, 333, 200, 64, 64, causal=True, seed=14),
    "window_causal": W("window_causal", 1, 2, 2, 400, 400, 128, 128, causal=True, window_left=100,
                       seed=15),
    "window_only": W("window_only", 1, 2, 2, 300, 280, 128, 128, window_left=150,
                     bottom_right=True, seed=16),
    "causal_band_right": W("causal_band_right", 1, 2, 2, 260, 260, 128, 128, causal=True,
                           window_right=50, seed=17),
    "gqa": W("gqa", 2, 4, 2, 256, 256, 128, 128, causal=True, seed=18),
    "mqa_d64": W("mqa_d64", 1, 3, 1, 200, 170, 64, 64, causal=True, bottom_right=True, seed=19),
    "padded_window": W("padded_window", 3, 2, 2, 300, 300, 128, 128, causal=True,
                       window_left=64, padded=(1, 300), seed=20),
    "custom_scale": W("custom_scale", 1, 2, 2, 150, 150, 128, 128, causal=True, scale=0.05,
                      seed=21),
    "single_query": W("single_query", 1, 2, 2, 1, 300, 128, 128, causal=True, bottom_right=True,
                      seed=22),
    "single_key": W("single_key", 1, 2, 2, 130, 1, 64, 64, seed=23),
    "gqa_det": W("gqa_det", 1, 4, 2, 520, 520, 128, 128, causal=True, deterministic=True, seed=24),
    "window_det": W("window_det", 2, 2, 1, 600, 600, 128, 128, causal=True, window_left=200,
                    deterministic=True, seed=25),
    # deterministic D=64: the ordered relay of dQ reductions on turn counters
    "det_d64_relay": W("det_d64_relay", 2, 4, 2, 300, 300, 64, 64, causal=True,
                       deterministic=True, seed=38),
    "det_d64_window": W("det_d64_window", 1, 2, 2, 400, 330, 64, 64, causal=True,
                        bottom_right=True, window_left=90, deterministic=True, seed=39),
    # deterministic D=128: the 128-row-tile main kernel (odd 64-row tile counts
    # exercise its half-filled last tile)
    "det_padded_odd": W("det_padded_odd", 2, 2, 2, 300, 300, 128, 128, causal=True,
                        padded=(30, 300), deterministic=True, seed=32),
    "det_br_long_kv": W("det_br_long_kv", 1, 2, 2, 200, 333, 128, 128, causal=True,
                        bottom_right=True, deterministic=True, seed=33),
    "det_dense_ragged": W("det_dense_ragged", 2, 2, 1, 130, 250, 128, 128, deterministic=True,
                          seed=34),
    "det_window_only": W("det_window_only", 1, 2, 2, 300, 280, 128, 128, window_left=150,
                         bottom_right=True, deterministic=True, seed=35),
    "mla_br_causal_ragged": W("mla_br_causal_ragged", 1, 2, 2, 300, 333, 192, 128, causal=True,
                              bottom_right=True, seed=28),
    "mla_dense": W("mla_dense", 2, 2, 2, 190, 250, 192, 128, seed=29),
    "mla_gqa_window": W("mla_gqa_window", 1, 4, 2, 400, 400, 192, 128, causal=True,
                        window_left=100, seed=30),
    "mla_padded_det": W("mla_padded_det", 2, 2, 2, 300, 300, 192, 128, causal=True,
                        padded=(50, 300), deterministic=True, seed=31),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_full_parity(name):
    _full_compare(SMALL[name])


def test_padded_rows_are_exact_zeros():
    w = SMALL["padded_window"]
    case, (dq, dk, dv), _ = _full_compare(w)
    lens = case["seq_q_lens"].tolist()
    for b, L in enumerate(lens):
        assert torch.all(dq[b, :, L:] == 0)
        assert torch.all(dk[b, :, L:] == 0) and torch.all(dv[b, :, L:] == 0)


def test_zero_length_batch_row():
    w = W("zero_len", 2, 2, 2, 200, 200, 128, 128, causal=True, seed=26)
    case = make_case(w)
    lens = torch.tensor([0, 150], dtype=torch.int32)
    case["seq_q_lens"] = lens
    case["seq_kv_lens"] = lens.clone()
    case["problem"].seq_q_lens = lens.numpy()
    case["problem"].seq_kv_lens = lens.numpy()
    # O/LSE consistent with the lengths
    import oracle
    from harness import f64
    o64, lse64 = oracle.forward(case["problem"], f64(case["q"]), f64(case["k"]), f64(case["v"]))
    case["o"] = torch.from_numpy(o64).to(torch.bfloat16)
    case["lse"] = torch.from_numpy(lse64).float()
    dq, dk, dv = gpu_backward(case)
    ref = oracle_backward(case)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(name, g.double().cpu().numpy(), r)
    assert torch.all(dq[0] == 0) and torch.all(dk[0] == 0) and torch.all(dv[0] == 0)


def test_adversarial_key_growth_masked():
    """Keys scaled by growth**(key // 128) make the probability mass jump between
    key tiles; a masked entry leaking into a gradient shows as ref == 0, gpu != 0.
    (Where the oracle's zero comes from cancellation, e.g. a row that sees one key
    has dS = P*(dP - delta) = 0 exactly in fp64, the fp32 GPU result is ~1e-8, so
    the check is relative to the tensor's scale: a leaked probability is O(1).)"""
    w = W("growth", 1, 2, 2, 384, 384, 128, 128, causal=True, window_left=150, seed=27)
    case = make_case(w)
    growth = torch.tensor(1.5) ** (torch.arange(384) // 128).float()
    case["k"] = (case["k"].float() * growth[None, None, :, None]).to(torch.bfloat16)
    import oracle
    from harness import f64
    o64, lse64 = oracle.forward(case["problem"], f64(case["q"]), f64(case["k"]), f64(case["v"]))
    case["o"] = torch.from_numpy(o64).to(torch.bfloat16)
    case["lse"] = torch.from_numpy(lse64).float()
    dq, dk, dv = gpu_backward(case)
    ref = oracle_backward(case)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = g.double().cpu().numpy()
        assert_close(name, g, r)
        leak = np.abs(g[r == 0]).max(initial=0.0)
        assert leak <= 1e-5 * np.abs(r).max(), f"{name}: {leak:.3e} where the oracle is exactly zero"


@pytest.mark.parametrize("name", ["window_det", "det_d64_relay"])
def test_deterministic_bitwise_small(name):
    w = SMALL[name]
    case = make_case(w)
    d = to_device(case)
    first = gpu_backward(case, d)
    for _ in range(5):
        again = gpu_backward(case, d)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------- full-size workloads
_CASES = {}


def _case(name):
    if name not in _CASES:
        _CASES[name] = make_case(workloads.WORKLOADS[name])
    return _CASES[name]


def _sample_rows(w, lens, rng, n_rand=24):
    """Flat query rows and key rows to check: tile edges, ends, padding, random."""
    q_rows, kv_rows = [], []
    edges = [0, 1, 127, 128, 129, 255, 256, w.Sq // 2, w.Sq - 129, w.Sq - 128, w.Sq - 1]
    for b in range(w.B):
        L = w.Sq if lens is None else int(lens[b])
        pick = set(e for e in edges if 0 <= e < w.Sq)
        pick |= {max(L - 1, 0), min(L, w.Sq - 1)}
        for h in (0, w.Hq - 1):
            q_rows += [(b * w.Hq + h) * w.Sq + q for q in sorted(pick)]
        for hk in (0, w.Hkv - 1):
            kv_rows += [(b * w.Hkv + hk) * w.Skv + k for k in sorted(pick) if k < w.Skv]
    q_rows += list(rng.integers(0, w.B * w.Hq * w.Sq, n_rand))
    kv_rows += list(rng.integers(0, w.B * w.Hkv * w.Skv, n_rand))
    return np.unique(np.array(q_rows)), np.unique(np.array(kv_rows))


@pytest.mark.parametrize("name", workloads.ORDER)
def test_workload_sampled_parity(name):
    _sampled_check(_case(name))


# Shapes large enough that the main kernel's work units span several query
# heads of a KV group (their dK/dV summed in tensor memory; the host takes the
# largest group size that leaves 1.5 units per SM): two heads per unit with no
# partial sets left (G = 2: 16 key tiles x 2 x 16 groups = 512 units), and two
# heads per unit with two partial sets to reduce (G = 4, deterministic route:
# 16 x 1 x 8 x 2 = 256 units, while four heads per unit would leave 128).
GROUPED = {
    "group2_nopart": W("group2_nopart", 2, 32, 16, 2048, 2048, 128, 128, causal=True, seed=36),
    "group2_part2_det": W("group2_part2_det", 1, 32, 8, 2048, 2048, 128, 128, causal=True,
                          deterministic=True, seed=37),
}


@pytest.mark.parametrize("name", sorted(GROUPED))
def test_grouped_units_sampled_parity(name):
    _sampled_check(make_case(GROUPED[name]))


def _sampled_check(case):
    w = case["workload"]
    dq, dk, dv = gpu_backward(case)
    lens = None if case["seq_q_lens"] is None else case["seq_q_lens"].numpy()
    q_rows, kv_rows = _sample_rows(w, lens, np.random.default_rng(w.seed))
    rq, rk, rv = oracle_sampled(case, q_rows, kv_rows)
    gq = dq.reshape(-1, w.Dqk)[torch.from_numpy(q_rows).cuda()].double().cpu().numpy()
    gk = dk.reshape(-1, w.Dqk)[torch.from_numpy(kv_rows).cuda()].double().cpu().numpy()
    gv = dv.reshape(-1, w.Dv)[torch.from_numpy(kv_rows).cuda()].double().cpu().numpy()
    assert_close("dq", gq, rq)
    assert_close("dk", gk, rk)
    assert_close("dv", gv, rv)
    for g in (dq, dk, dv):
        assert torch.isfinite(g).all()
    if lens is not None:
        for b, L in enumerate(lens):
            assert torch.all(dq[b, :, L:] == 0) and torch.all(dk[b, :, L:] == 0)
            assert torch.all(dv[b, :, L:] == 0)


def test_workload_deterministic_bitwise_10_runs():
    case = _case("causal_gqa_det")
    d = to_device(case)
    first = gpu_backward(case, d)
    for _ in range(9):
        again = gpu_backward(case, d, poison=True)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ---------------------------------------------------------------- sink tokens
# With a sink the forward's LSE includes it; dQ/dK/dV come out of the same
# kernels and dsink from the preprocess partials plus the fixed-order reduce.
SINK_CASES = {
    "d128_causal_ragged": SMALL["d128_causal_ragged"],
    "gqa_det": SMALL["gqa_det"],
    "det_padded_odd": SMALL["det_padded_odd"],
    "padded_nondet": SMALL["det_padded_odd"].with_(name="padded_nondet", deterministic=False),
    "mla_gqa_window": SMALL["mla_gqa_window"],
    "tl_causal_long_q_d64": SMALL["tl_causal_long_q"],
    "mid_gqa": W("mid_gqa", 2, 8, 2, 1024, 1024, 128, 128, causal=True, seed=40),
}


def _dsink_close(gpu, ref, mag):
    err = np.abs(gpu - ref)
    # fp32 delta, exp2 and sums against fp64: a few ulp of the terms' magnitude
    assert np.all(err <= 1e-4 * mag + 1e-6), f"dsink: err {err.max():.3e}, mag {mag.max():.3e}"


@pytest.mark.parametrize("name", sorted(SINK_CASES))
def test_sink_parity(name):
    case = make_case(SINK_CASES[name], sink=True)
    d = to_device(case)
    dq, dk, dv, dsink = gpu_backward(case, d, sink=d["sink"])
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)
    ref, mag = oracle_dsink(case)
    _dsink_close(dsink.double().cpu().numpy(), ref, mag)
    # The sink enters dQ/dK/dV only through the LSE: the plain call gives the same bits
    dq2, dk2, dv2 = gpu_backward(case, d)
    if case["workload"].deterministic or case["workload"].Dqk == 192:
        for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_dsink_bitwise_reproducible():
    case = make_case(SINK_CASES["mid_gqa"], sink=True)
    d = to_device(case)
    first = gpu_backward(case, d, sink=d["sink"])[3].clone()
    for _ in range(9):
        again = gpu_backward(case, d, sink=d["sink"])[3]
        assert torch.equal(first.view(torch.int32), again.view(torch.int32))


# ---------------------------------------------------------------- forward
# The fused forward against the oracle forward: O (bf16) within the gradient
# tolerance, LSE within 1e-3 (fp32 scores of bf16 products, ex2.approx), rows
# without a visible key exactly -inf (or the sink).
FWD_CASES = {
    "tiny_dense": SMALL["tiny_dense"],
    "d128_causal_ragged": SMALL["d128_causal_ragged"],
    "br_causal_long_kv": SMALL["br_causal_long_kv"],
    "br_causal_long_q": SMALL["br_causal_long_q"],
    "tl_causal_long_q_d64": SMALL["tl_causal_long_q"],
    "window_causal": SMALL["window_causal"],
    "window_only": SMALL["window_only"],        # warps whose rows split across mask paths
    "d128_dense_ragged": SMALL["d128_dense_ragged"],
    "gqa_det": SMALL["gqa_det"],
    "det_padded_odd": SMALL["det_padded_odd"],
    "single_query": SMALL["single_query"],
    "mla_gqa_window": SMALL["mla_gqa_window"],
    "mla_padded_det": SMALL["mla_padded_det"],
}


def _check_fwd(case, o, lse, rows=None):
    ro = case["o"].double().numpy()
    rl = case["lse"].double().numpy()
    go = o.double().cpu().numpy()
    gl = lse.double().cpu().numpy()
    if rows is not None:
        ro, rl = ro.reshape(-1, ro.shape[-1])[rows], rl.reshape(-1)[rows]
        go, gl = go.reshape(-1, go.shape[-1])[rows], gl.reshape(-1)[rows]
    assert_close("o", go, ro)
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(gl)), "LSE: -inf rows differ"
    assert np.all(gl[~fin] == rl[~fin])
    err = np.abs(gl[fin] - rl[fin])
    assert err.size == 0 or err.max() <= 1e-3 * max(1.0, np.abs(rl[fin]).max()), f"lse err {err.max():.3e}"


def _gpu_fwd(case, d):
    import attention_backward_sdpa_gb300 as pkg
    w = case["workload"]
    o, lse = pkg.sdpa_fwd(d["q"], d["k"], d["v"], scale=w.resolved_scale, causal=w.causal,
                          bottom_right=w.bottom_right, window_left=w.window_left,
                          window_right=w.window_right, seq_q_lens=d["seq_q_lens"],
                          seq_kv_lens=d["seq_kv_lens"], sink=d.get("sink"), bias=d.get("bias"),
                          o=torch.full((w.B, w.Hq, w.Sq, w.Dv), float("nan"), dtype=d["q"].dtype,
                                       device="cuda"),
                          lse=torch.full((w.B, w.Hq, w.Sq), float("nan"), device="cuda"))
    pkg.check_device_status()
    return o, lse


@pytest.mark.parametrize("name", sorted(FWD_CASES))
@pytest.mark.parametrize("sink", [False, True])
def test_forward_parity(name, sink):
    case = make_case(FWD_CASES[name], sink=sink)
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    _check_fwd(case, o, lse)


@pytest.mark.parametrize("name", workloads.ORDER)
def test_forward_full_size(name):
    case = _case(name)
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    w = case["workload"]
    rng = np.random.default_rng(w.seed + 7)
    rows = np.unique(rng.integers(0, w.B * w.Hq * w.Sq, 4096))
    _check_fwd(case, o, lse, rows)


def test_forward_then_backward_matches_oracle():
    """A training step: the GPU forward's O/LSE into the GPU backward, against the
    oracle backward of the same O/LSE."""
    case = make_case(SMALL["gqa_det"])
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    case["o"], case["lse"] = o.cpu(), lse.cpu()
    dq, dk, dv = gpu_backward(case)
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)


# ---------------------------------------------------------------- additive bias
# The bias joins the scores before the softmax (the oracle forward gives the
# LSE of the biased scores); dQ/dK/dV and the fp32 dBias are checked against
# the oracle with the gradient bar. dBias comes back NaN-poisoned, so every
# element must be written: visited tiles by the main kernel (masked pairs as
# 0), the others by the preprocess. "1" marks one bias batch shared by B > 1
# batch rows (dBias summed atomically), "B" a bias per batch row.
BIAS_CASES = {
    "d128_causal_ragged_B_bf16": (SMALL["d128_causal_ragged"], "B", torch.bfloat16),
    "gqa_shared_f32": (SMALL["gqa"], "1", torch.float32),
    "gqa_det_B_bf16": (SMALL["gqa_det"], "B", torch.bfloat16),          # stored-dS route
    "det_padded_odd_B_f32": (SMALL["det_padded_odd"], "B", torch.float32),
    "padded_window_shared_bf16": (SMALL["padded_window"], "1", torch.bfloat16),
    "tl_causal_long_q_d64_B_bf16": (SMALL["tl_causal_long_q"], "B", torch.bfloat16),
    "det_d64_relay_B_f32": (SMALL["det_d64_relay"], "B", torch.float32),
    "window_only_B_bf16": (SMALL["window_only"], "B", torch.bfloat16),
    "single_key_d64_B_f32": (SMALL["single_key"], "B", torch.float32),
    "d128_dense_ragged_shared_bf16": (SMALL["d128_dense_ragged"], "1", torch.bfloat16),
    "br_causal_long_kv_B_f32": (SMALL["br_causal_long_kv"], "B", torch.float32),
    # D_qk 192 / D_v 128 (the MLA kernel)
    "mla_br_causal_ragged_B_bf16": (SMALL["mla_br_causal_ragged"], "B", torch.bfloat16),
    "mla_dense_shared_f32": (SMALL["mla_dense"], "1", torch.float32),
    "mla_gqa_window_B_f32": (SMALL["mla_gqa_window"], "B", torch.float32),
    "mla_padded_det_B_bf16": (SMALL["mla_padded_det"], "B", torch.bfloat16),
}


def _bias_case(w, kind, dtype):
    return make_case(w, bias=(1 if kind == "1" else w.B, dtype))


def _gpu_bias(case, d):
    dbias = torch.full(tuple(d["bias"].shape), float("nan"), dtype=torch.float32, device="cuda")
    out = gpu_backward(case, d, bias=d["bias"], dbias=dbias)
    assert len(out) == 4 and out[3] is dbias
    return out


@pytest.mark.parametrize("name", sorted(BIAS_CASES))
def test_bias_parity(name):
    case = _bias_case(*BIAS_CASES[name])
    d = to_device(case)
    dq, dk, dv, dbias = _gpu_bias(case, d)
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)
    rb = oracle_dbias(case)
    gb = dbias.double().cpu().numpy()
    assert_close("dbias", gb, rb)
    # masked pairs and padding carry exact zeros
    masked = ~_visible_mask(case)
    if masked.any():
        assert np.all(gb[np.broadcast_to(masked, gb.shape)] == 0.0)


def _visible_mask(case):
    """(bias_batch, 1, Sq, Skv) pairs visible in every batch row the bias serves."""
    w = case["workload"]
    p = case["problem"]
    qi = np.arange(w.Sq)[:, None]
    ki = np.arange(w.Skv)[None, :]
    vis = []
    for b in range(w.B):
        Lq = w.Sq if p.seq_q_lens is None else int(p.seq_q_lens[b])
        Lk = w.Skv if p.seq_kv_lens is None else int(p.seq_kv_lens[b])
        diag = (Lk - Lq) if w.bottom_right else 0
        m = (qi < Lq) & (ki < Lk)
        if w.causal:
            m &= ki <= qi + diag + max(w.window_right, 0)
        if w.window_left >= 0:
            m &= ki >= qi + diag - w.window_left
        vis.append(m)
    vis = np.stack(vis)[:, None]
    if case["bias"].shape[0] == 1:
        vis = vis.any(0, keepdims=True)
    return vis


def test_bias_without_dbias_matches():
    """bias_grad=False computes the same dQ/dK/dV without writing a dBias."""
    case = _bias_case(*BIAS_CASES["gqa_det_B_bf16"])
    d = to_device(case)
    a = _gpu_bias(case, d)
    b = gpu_backward(case, d, bias=d["bias"], bias_grad=False)
    assert len(b) == 3
    for x, y in zip(a[:3], b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_bias_with_sink():
    case = make_case(SMALL["det_padded_odd"], sink=True, bias=(2, torch.float32))
    d = to_device(case)
    dbias = torch.full(tuple(d["bias"].shape), float("nan"), dtype=torch.float32, device="cuda")
    dq, dk, dv, dsink, db = gpu_backward(case, d, sink=d["sink"], bias=d["bias"], dbias=dbias)
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)
    assert_close("dbias", db.double().cpu().numpy(), oracle_dbias(case))
    ref, mag = oracle_dsink(case)
    _dsink_close(dsink.double().cpu().numpy(), ref, mag)


@pytest.mark.parametrize("name", ["gqa_det_B_bf16", "det_d64_relay_B_f32", "mla_padded_det_B_bf16"])
def test_dbias_bitwise_reproducible(name):
    """A per-batch dBias is written once per element: bitwise reproducible
    (10 runs), like dQ/dK/dV in deterministic mode."""
    case = _bias_case(*BIAS_CASES[name])
    d = to_device(case)
    first = [t.clone() for t in _gpu_bias(case, d)]
    for _ in range(9):
        again = _gpu_bias(case, d)
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# Full-size bias cases: the causal MHA workload with one bias shared by both
# batch rows (atomic dBias), and a grouped shape whose work units carry two
# query heads (G = 8, 8 key tiles x 8 groups x 4 parts x 2 >= 1.5 units per SM).
BIAS_FULL = {
    "causal_mha_shared_bf16": (workloads.WORKLOADS["causal_mha"], "1", torch.bfloat16),
    "grouped_B_f32": (W("bias_groups", 1, 64, 8, 1024, 1024, 128, 128, causal=True, seed=41), "B",
                      torch.float32),
}


@pytest.mark.parametrize("name", sorted(BIAS_FULL))
def test_bias_full_size_sampled(name):
    case = _bias_case(*BIAS_FULL[name])
    w = case["workload"]
    d = to_device(case)
    dq, dk, dv, dbias = _gpu_bias(case, d)
    q_rows, kv_rows = _sample_rows(w, None, np.random.default_rng(w.seed))
    rq, rk, rv = oracle_sampled(case, q_rows, kv_rows)
    assert_close("dq", dq.reshape(-1, w.Dqk)[torch.from_numpy(q_rows).cuda()].double().cpu().numpy(), rq)
    assert_close("dk", dk.reshape(-1, w.Dqk)[torch.from_numpy(kv_rows).cuda()].double().cpu().numpy(), rk)
    assert_close("dv", dv.reshape(-1, w.Dv)[torch.from_numpy(kv_rows).cuda()].double().cpu().numpy(), rv)
    nb = dbias.shape[0]
    rows = np.unique(np.array([(bb * w.Hq + h) * w.Sq + q for bb in range(nb) for h in (0, w.Hq - 1)
                               for q in (0, 63, 64, 127, 128, w.Sq // 2 + 5, w.Sq - 1)] +
                              list(np.random.default_rng(w.seed + 1).integers(0, nb * w.Hq * w.Sq, 16))))
    rb = oracle_dbias(case, rows)
    gb = dbias.reshape(-1, w.Skv)[torch.from_numpy(rows).cuda()].double().cpu().numpy()
    assert_close("dbias", gb, rb)
    assert torch.isfinite(dbias).all()


# Forward with a bias: O and LSE of the biased scores against the oracle forward
# with the same bias (16-byte bias rows and ragged ones, per-batch and shared,
# bf16 and fp32, every head-dim pair).
FWD_BIAS_CASES = {
    "d128_causal_ragged_B_bf16": (SMALL["d128_causal_ragged"], "B", torch.bfloat16),  # S_kv 300
    "d128_dense_ragged_shared_f32": (SMALL["d128_dense_ragged"], "1", torch.float32),
    "gqa_B_f32": (SMALL["gqa"], "B", torch.float32),
    "padded_window_shared_bf16": (SMALL["padded_window"], "1", torch.bfloat16),
    "tl_causal_long_q_d64_B_f32": (SMALL["tl_causal_long_q"], "B", torch.float32),   # S_kv 200
    "window_only_B_bf16": (SMALL["window_only"], "B", torch.bfloat16),               # S_kv 280
    "mla_gqa_window_B_bf16": (SMALL["mla_gqa_window"], "B", torch.bfloat16),
    "single_query_B_f32": (SMALL["single_query"], "B", torch.float32),
}


@pytest.mark.parametrize("name", sorted(FWD_BIAS_CASES))
def test_forward_bias_parity(name):
    case = _bias_case(*FWD_BIAS_CASES[name])
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    _check_fwd(case, o, lse)


def test_forward_bias_minus_infinity_rows():
    """A bias of -inf on every key of some rows empties them (O = 0, LSE = -inf);
    -inf on some keys removes just those."""
    w = SMALL["d128_causal_ragged"]
    bias = workloads.bias_tensor(w, 1, torch.float32)
    bias[0, 0, 5:9, :] = float("-inf")       # whole rows
    bias[0, 1, :, 7::3] = float("-inf")      # a comb of keys
    case = make_case(w, bias=(1, torch.float32))
    case["bias"] = bias
    import oracle
    from harness import f64
    o64, lse64 = oracle.forward(case["problem"], f64(case["q"]), f64(case["k"]), f64(case["v"]),
                                bias=bias.double().numpy())
    case["o"] = torch.from_numpy(o64).to(torch.bfloat16)
    case["lse"] = torch.from_numpy(lse64).float()
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    _check_fwd(case, o, lse)
    assert torch.all(lse[0, 0, 5:9] == float("-inf")) and torch.all(o[0, 0, 5:9] == 0)


@pytest.mark.parametrize("name", ["gqa_B_f32", "d128_causal_ragged_B_bf16"])
def test_forward_then_backward_with_bias(name):
    """sdpa_fwd_bias then sdpa_bwd_bias on the GPU's own O/LSE match the oracle's
    forward and backward."""
    case = _bias_case(*FWD_BIAS_CASES[name])
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    d["o"], d["lse"] = o, lse
    dq, dk, dv, dbias = _gpu_bias(case, d)
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)
    assert_close("dbias", dbias.double().cpu().numpy(), oracle_dbias(case))


# ---------------------------------------------------------------- NVFP4 QAT
# The fake quantization is a rounding: the GPU's must equal the oracle's bit
# for bit. The QAT backward (quantized Q, K, V in the GEMMs, P fake-quantized
# over 16-key blocks for dV only) is checked against the oracle's with the
# gradient bar; O_hp / LSE come from the oracle's QAT forward.
def test_nvfp4_fake_quant_bitwise():
    import attention_backward_sdpa_gb300 as pkg
    import oracle
    g = torch.Generator("cpu").manual_seed(50)
    n_blocks = 8192
    mag = 10.0 ** (torch.rand(n_blocks, 1, generator=g) * 10 - 6)   # 1e-6 .. 1e4 per block
    x = (torch.randn(n_blocks, 16, generator=g) * mag)
    x[:64] = 0.0                                                      # zero blocks
    x[64:128] *= 1e6                                                  # saturated scales
    x[128:192, :8] = 0.0                                              # half-empty blocks
    xb = x.to(torch.bfloat16)
    y = pkg.nvfp4_fake_quant(xb.cuda()).cpu()
    ref64 = torch.from_numpy(oracle.fake_nvfp4(xb.double().numpy()))
    ref = ref64.to(torch.bfloat16)
    assert torch.equal(ref.double(), ref64)  # every fake-quantized value is exact in bf16
    diff = (y.view(torch.int16) != ref.view(torch.int16)).nonzero()
    assert diff.numel() == 0, f"{diff.shape[0]} values differ, first at {diff[:4].tolist()}"


QAT_CASES = {
    "mha_causal_ragged": W("qat_mha_causal", 1, 2, 2, 300, 300, 128, 128, causal=True, seed=51),
    "mha_dense_cross": W("qat_mha_dense", 2, 2, 2, 190, 250, 128, 128, seed=52),
    "gqa_causal": W("qat_gqa", 1, 4, 2, 256, 256, 128, 128, causal=True, seed=53),
    "padded_window": W("qat_padded_window", 2, 2, 2, 300, 300, 128, 128, causal=True,
                       window_left=100, padded=(100, 300), seed=54),
}


def _qat_case(w):
    import oracle
    from harness import f64
    t = workloads.generate(w)
    p = oracle.Problem(
        w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.Dqk, w.Dv, scale=w.resolved_scale, causal=w.causal,
        bottom_right=w.bottom_right, window_left=w.window_left, window_right=w.window_right,
        seq_q_lens=None if t["seq_q_lens"] is None else t["seq_q_lens"].numpy(),
        seq_kv_lens=None if t["seq_kv_lens"] is None else t["seq_kv_lens"].numpy())
    o_hp, lse, _ = oracle.qat_forward(p, f64(t["q"]), f64(t["k"]), f64(t["v"]))
    t["o"] = torch.from_numpy(o_hp).to(torch.bfloat16)
    t["lse"] = torch.from_numpy(lse).float()
    t["problem"], t["workload"] = p, w
    return t


def _gpu_qat(case, d):
    import attention_backward_sdpa_gb300 as pkg
    w = case["workload"]
    nan = float("nan")
    out = pkg.sdpa_bwd_nvfp4_qat(d["q"], d["k"], d["v"], d["o"], d["do"], d["lse"],
                                 scale=w.resolved_scale, causal=w.causal,
                                 bottom_right=w.bottom_right, window_left=w.window_left,
                                 window_right=w.window_right, seq_q_lens=d["seq_q_lens"],
                                 seq_kv_lens=d["seq_kv_lens"], dq=torch.full_like(d["q"], nan),
                                 dk=torch.full_like(d["k"], nan), dv=torch.full_like(d["v"], nan))
    pkg.check_device_status()
    return out


@pytest.mark.parametrize("name", sorted(QAT_CASES))
def test_nvfp4_qat_parity(name):
    import oracle
    from harness import f64
    case = _qat_case(QAT_CASES[name])
    d = to_device(case)
    dq, dk, dv = _gpu_qat(case, d)
    rq, rk, rv = oracle.qat_backward(case["problem"], f64(case["q"]), f64(case["k"]), f64(case["v"]),
                                     f64(case["o"]), f64(case["do"]), case["lse"].double().numpy())
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)
    # dV really used the quantized P: the plain backward's dV is further away
    _, _, pv = oracle.backward(case["problem"], oracle.fake_nvfp4(f64(case["q"])),
                               oracle.fake_nvfp4(f64(case["k"])), oracle.fake_nvfp4(f64(case["v"])),
                               f64(case["o"]), f64(case["do"]), case["lse"].double().numpy())
    g = dv.double().cpu().numpy()
    assert np.linalg.norm(g - rv) < 0.5 * np.linalg.norm(g - pv)


def test_nvfp4_qat_forward_then_backward():
    """Fake quantization and sdpa_fwd on the GPU give O_hp / LSE; the QAT
    backward on them matches the oracle's QAT forward + backward."""
    import attention_backward_sdpa_gb300 as pkg
    import oracle
    from harness import f64
    case = _qat_case(QAT_CASES["gqa_causal"])
    w = case["workload"]
    d = to_device(case)
    o, lse = pkg.sdpa_fwd_nvfp4_qat(d["q"], d["k"], d["v"], scale=w.resolved_scale, causal=w.causal)
    _check_fwd(case, o, lse)
    d["o"], d["lse"] = o, lse
    dq, dk, dv = _gpu_qat(case, d)
    rq, rk, rv = oracle.qat_backward(case["problem"], f64(case["q"]), f64(case["k"]), f64(case["v"]),
                                     f64(case["o"]), f64(case["do"]), case["lse"].double().numpy())
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)


# ---------------------------------------------------------------- fp16 io
# The same chain with fp16 Q, K, V, O, dO, dQ, dK, dV (fp16 MMA operands, P and
# dS rounded to fp16, fp32 accumulation), against the oracle on the fp16 values.
F16_CASES = {
    "d128_causal_ragged": SMALL["d128_causal_ragged"],
    "gqa_det": SMALL["gqa_det"],                    # stored-dS route, dQ-from-dS kernel
    "gqa": SMALL["gqa"],                            # GQA partial sets, reduction route
    "tl_causal_long_q_d64": SMALL["tl_causal_long_q"],
    "det_d64_relay": SMALL["det_d64_relay"],
    "padded_window": SMALL["padded_window"],
    "window_only": SMALL["window_only"],
    "mla_br_causal_ragged": SMALL["mla_br_causal_ragged"],
    "mla_gqa_window": SMALL["mla_gqa_window"],
}


@pytest.mark.parametrize("name", sorted(F16_CASES))
def test_f16_parity(name):
    case = make_case(F16_CASES[name], io=torch.float16)
    d = to_device(case)
    dq, dk, dv = gpu_backward(case, d)
    assert dq.dtype == torch.float16 and dk.dtype == torch.float16
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)


@pytest.mark.parametrize("name", ["d128_causal_ragged", "mla_gqa_window", "tl_causal_long_q_d64",
                                  "padded_window"])
def test_f16_forward_parity(name):
    case = make_case(F16_CASES[name], io=torch.float16)
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    assert o.dtype == torch.float16
    _check_fwd(case, o, lse)


def test_f16_sink_and_bitwise():
    case = make_case(SMALL["det_padded_odd"], sink=True, io=torch.float16)
    d = to_device(case)
    first = gpu_backward(case, d, sink=d["sink"])
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", first[0].double().cpu().numpy(), rq)
    ref, mag = oracle_dsink(case)
    _dsink_close(first[3].double().cpu().numpy(), ref, mag)
    first = [t.clone() for t in first]
    for _ in range(9):
        again = gpu_backward(case, d, sink=d["sink"])
        for a, b in zip(first, again):
            assert torch.equal(a.view(torch.int16) if a.dtype != torch.float32 else a.view(torch.int32),
                               b.view(torch.int16) if b.dtype != torch.float32 else b.view(torch.int32))


def test_f16_full_size_sampled():
    """causal_mha's shape with fp16 io, sampled rows against the oracle."""
    w = workloads.WORKLOADS["causal_mha"]
    case = make_case(w, io=torch.float16)
    dq, dk, dv = gpu_backward(case)
    q_rows, kv_rows = _sample_rows(w, None, np.random.default_rng(7))
    rq, rk, rv = oracle_sampled(case, q_rows, kv_rows)
    assert_close("dq", dq.reshape(-1, w.Dqk)[torch.from_numpy(q_rows).cuda()].double().cpu().numpy(), rq)
    assert_close("dk", dk.reshape(-1, w.Dqk)[torch.from_numpy(kv_rows).cuda()].double().cpu().numpy(), rk)
    assert_close("dv", dv.reshape(-1, w.Dv)[torch.from_numpy(kv_rows).cuda()].double().cpu().numpy(), rv)


# ---------------------------------------------------------------- head dim 32
# D = 32 runs on the 64-column kernels: TMA loads zero-fill columns 32..63 (so
# the extra columns add nothing to any product) and TMA stores drop them; the
# dQ accumulator keeps 64-column rows.
D32_CASES = {
    "d32_causal_ragged": W("d32_causal_ragged", 1, 2, 2, 300, 300, 32, 32, causal=True, seed=60),
    "d32_gqa_det_relay": W("d32_gqa_det", 1, 4, 2, 260, 260, 32, 32, causal=True, deterministic=True,
                           seed=61),
    "d32_padded_window": W("d32_padded_window", 2, 2, 2, 300, 300, 32, 32, causal=True, window_left=90,
                           padded=(100, 300), seed=62),
    "d32_dense_cross_gqa": W("d32_dense_cross", 2, 2, 1, 190, 250, 32, 32, seed=63),
}


@pytest.mark.parametrize("name", sorted(D32_CASES))
def test_d32_parity(name):
    case = make_case(D32_CASES[name])
    d = to_device(case)
    dq, dk, dv = gpu_backward(case, d)
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)


@pytest.mark.parametrize("name", ["d32_causal_ragged", "d32_padded_window"])
def test_d32_forward_parity(name):
    case = make_case(D32_CASES[name])
    d = to_device(case)
    o, lse = _gpu_fwd(case, d)
    _check_fwd(case, o, lse)


def test_d32_f16_bias_and_bitwise():
    w = D32_CASES["d32_causal_ragged"]
    case = make_case(w, io=torch.float16)
    d = to_device(case)
    dq, dk, dv = gpu_backward(case, d)
    for g, r, n in zip((dq, dk, dv), oracle_backward(case), ("dq", "dk", "dv")):
        assert_close(n, g.double().cpu().numpy(), r)
    case = make_case(w, bias=(1, torch.float32))
    d = to_device(case)
    dq, dk, dv, db = _gpu_bias(case, d)
    for g, r, n in zip((dq, dk, dv), oracle_backward(case), ("dq", "dk", "dv")):
        assert_close(n, g.double().cpu().numpy(), r)
    assert_close("dbias", db.double().cpu().numpy(), oracle_dbias(case))
    case = make_case(D32_CASES["d32_gqa_det_relay"])
    d = to_device(case)
    first = [t.clone() for t in gpu_backward(case, d)]
    for _ in range(9):
        for a, b in zip(first, gpu_backward(case, d)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# Other multiples of 8 up to 128 run on the next larger kernel (64 or 128
# columns) the same way; in deterministic mode those on the 128-column kernel
# take the ordered relay (the stored-dS route is for exactly 128).
DPAD_CASES = {
    "d8_causal": W("d8_causal", 1, 2, 2, 150, 150, 8, 8, causal=True, seed=64),
    "d40_gqa_window": W("d40_gqa_window", 1, 4, 2, 260, 230, 40, 40, causal=True, bottom_right=True,
                        window_left=70, seed=65),
    "d72_dense_cross": W("d72_dense_cross", 2, 2, 2, 190, 250, 72, 72, seed=66),
    "d96_det_relay": W("d96_det", 1, 4, 2, 260, 260, 96, 96, causal=True, deterministic=True, seed=67),
    "d120_padded": W("d120_padded", 2, 2, 2, 300, 300, 120, 120, causal=True, padded=(100, 300), seed=68),
}


@pytest.mark.parametrize("name", sorted(DPAD_CASES))
def test_padded_head_dim_parity(name):
    case = make_case(DPAD_CASES[name])
    d = to_device(case)
    dq, dk, dv = gpu_backward(case, d)
    rq, rk, rv = oracle_backward(case)
    assert_close("dq", dq.double().cpu().numpy(), rq)
    assert_close("dk", dk.double().cpu().numpy(), rk)
    assert_close("dv", dv.double().cpu().numpy(), rv)
    o, lse = _gpu_fwd(case, d)
    _check_fwd(case, o, lse)


def test_padded_head_dim_f16_and_bitwise():
    case = make_case(DPAD_CASES["d40_gqa_window"], io=torch.float16)
    d = to_device(case)
    for g, r, n in zip(gpu_backward(case, d), oracle_backward(case), ("dq", "dk", "dv")):
        assert_close(n, g.double().cpu().numpy(), r)
    case = make_case(DPAD_CASES["d96_det_relay"])
    d = to_device(case)
    first = [t.clone() for t in gpu_backward(case, d)]
    for _ in range(9):
        for a, b in zip(first, gpu_backward(case, d)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# fp16 io with an additive bias (fp16 or fp32 bias elements), backward and forward.
F16_BIAS_CASES = {
    "d128_causal_ragged_B_f16": (SMALL["d128_causal_ragged"], "B", torch.float16),
    "gqa_shared_f32": (SMALL["gqa"], "1", torch.float32),
    "gqa_det_B_f16": (SMALL["gqa_det"], "B", torch.float16),
    "mla_gqa_window_B_f16": (SMALL["mla_gqa_window"], "B", torch.float16),
}


@pytest.mark.parametrize("name", sorted(F16_BIAS_CASES))
def test_f16_bias_parity(name):
    w, kind, dt = F16_BIAS_CASES[name]
    case = make_case(w, bias=(1 if kind == "1" else w.B, dt), io=torch.float16)
    d = to_device(case)
    dq, dk, dv, dbias = _gpu_bias(case, d)
    assert dq.dtype == torch.float16
    for g, r, n in zip((dq, dk, dv), oracle_backward(case), ("dq", "dk", "dv")):
        assert_close(n, g.double().cpu().numpy(), r)
    assert_close("dbias", dbias.double().cpu().numpy(), oracle_dbias(case))
    o, lse = _gpu_fwd(case, d)
    _check_fwd(case, o, lse)


# The io-type dBias (bf16 / fp16 elements): written directly for a per-batch
# bias (half the bytes), summed in fp32 and cast for a shared one.
DBIAS16_CASES = {
    "d128_causal_ragged_B_bf16out": (SMALL["d128_causal_ragged"], "B", torch.bfloat16, torch.bfloat16),
    "gqa_shared_f16out": (SMALL["gqa"], "1", torch.float32, torch.float16),
    "padded_window_B_bf16out": (SMALL["padded_window"], "B", torch.bfloat16, torch.bfloat16),
    "mla_dense_shared_bf16out": (SMALL["mla_dense"], "1", torch.bfloat16, torch.bfloat16),
    "d40_f16io_B_f16out": (DPAD_CASES["d40_gqa_window"], "B", torch.float16, torch.float16),
}


@pytest.mark.parametrize("name", sorted(DBIAS16_CASES))
def test_io_type_dbias(name):
    w, kind, bdt, odt = DBIAS16_CASES[name]
    io = torch.float16 if bdt == torch.float16 and odt == torch.float16 else torch.bfloat16
    case = make_case(w, bias=(1 if kind == "1" else w.B, bdt), io=io)
    d = to_device(case)
    dbias = torch.full(tuple(d["bias"].shape), float("nan"), dtype=odt, device="cuda")
    dq, dk, dv, db = gpu_backward(case, d, bias=d["bias"], dbias=dbias, dbias_dtype=odt)
    assert db is dbias and db.dtype == odt
    for g, r, n in zip((dq, dk, dv), oracle_backward(case), ("dq", "dk", "dv")):
        assert_close(n, g.double().cpu().numpy(), r)
    gb = db.double().cpu().numpy()
    assert_close("dbias", gb, oracle_dbias(case))
    masked = ~_visible_mask(case)
    if masked.any():
        assert np.all(gb[np.broadcast_to(masked, gb.shape)] == 0.0)
