"""Pins for the fp64 oracle, independent of the oracle itself.

Each check below fixes the oracle to something it does not compute the same
way: central finite differences of its own forward, algebraic invariants,
closed forms worked by hand, brute-force counts against closed forms, and a
float64 autograd run of torch's scaled_dot_product_attention (a library
special case). A dropped delta term, a wrong sign, a transposed operand or an
off-by-one in a mask edge each fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import Problem

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _inputs(p: Problem, seed=0, qscale=1.0):
    rng = np.random.default_rng(seed)
    q = _rand(rng, p.B, p.Hq, p.Sq, p.Dqk) * qscale
    k = _rand(rng, p.B, p.Hkv, p.Skv, p.Dqk)
    v = _rand(rng, p.B, p.Hkv, p.Skv, p.Dv)
    do = _rand(rng, p.B, p.Hq, p.Sq, p.Dv)
    return q, k, v, do


# Tiny problems spanning every mask kind, GQA/MQA, S_q != S_kv and D_qk != D_v.
FD_CASES = {
    "dense": Problem(1, 2, 2, 5, 7, 4, 3),
    "causal_tl": Problem(1, 2, 1, 6, 6, 4, 4, causal=True),
    "causal_br_long_q": Problem(1, 2, 2, 7, 4, 3, 5, causal=True, bottom_right=True),
    "causal_br_long_kv": Problem(1, 2, 2, 4, 9, 5, 3, causal=True, bottom_right=True),
    "causal_band_r2": Problem(1, 2, 2, 6, 8, 4, 4, causal=True, window_right=2),
    "window_causal": Problem(1, 2, 2, 8, 8, 4, 3, causal=True, window_left=2),
    "window_only": Problem(1, 2, 2, 7, 9, 3, 3, window_left=3, bottom_right=True),
    "padded": Problem(2, 2, 2, 6, 7, 4, 4, causal=True, bottom_right=True,
                      seq_q_lens=np.array([4, 6]), seq_kv_lens=np.array([5, 3])),
    "gqa": Problem(1, 4, 2, 5, 6, 4, 4, causal=True),
    "mqa_scale": Problem(1, 3, 1, 5, 5, 6, 4, scale=0.37),
}


def _loss(oracle_mod, p, q, k, v, do):
    o, _ = oracle_mod.forward(p, q, k, v)
    return float(np.sum(o * do))


def _central_differences(oracle_mod, p, q, k, v, do, h=1e-6):
    """dL/dQ, dL/dK, dL/dV of L = sum(O * dO), element by element, from the forward alone."""
    out = []
    for which, tensor in (("q", q), ("k", k), ("v", v)):
        fd = np.zeros_like(tensor)
        it = np.nditer(tensor, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            plus = tensor.copy()
            plus[idx] += h
            minus = tensor.copy()
            minus[idx] -= h
            args[which] = plus
            lp = _loss(oracle_mod, p, args["q"], args["k"], args["v"], do)
            args[which] = minus
            lm = _loss(oracle_mod, p, args["q"], args["k"], args["v"], do)
            fd[idx] = (lp - lm) / (2 * h)
        out.append(fd)
    return out


def _fd_tol(fd):
    return 2e-7 * max(1.0, float(np.abs(fd).max()))


@pytest.mark.parametrize("name", sorted(FD_CASES))
def test_backward_matches_central_differences(oracle_mod, name):
    """dL/dQ, dL/dK, dL/dV of L = sum(O * dO) by central differences of the forward."""
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=sum(map(ord, name)))
    o, lse = oracle_mod.forward(p, q, k, v)
    grads = oracle_mod.backward(p, q, k, v, o, do, lse)
    fds = _central_differences(oracle_mod, p, q, k, v, do)
    for grad, fd, which in zip(grads, fds, "qkv"):
        np.testing.assert_allclose(grad, fd, rtol=0, atol=_fd_tol(fd), err_msg=f"d{which}")


def test_finite_difference_pin_rejects_planted_mistakes(oracle_mod):
    """The pin above has teeth: backward results with a planted mistake (made on
    the CPU by feeding the oracle a wrong argument, or by altering its output)
    miss the central differences by far more than the tolerance."""
    import dataclasses
    p = Problem(1, 2, 2, 6, 6, 4, 4, causal=True, window_left=3, scale=0.6)
    q, k, v, do = _inputs(p, seed=11)
    o, lse = oracle_mod.forward(p, q, k, v)
    fds = _central_differences(oracle_mod, p, q, k, v, do)
    good = oracle_mod.backward(p, q, k, v, o, do, lse)
    wider = dataclasses.replace(p, window_left=4)
    kq = oracle_mod.backward(p, k, q, v, o, do, lse)  # Q and K exchanged: S transposed
    mutants = {
        "dropped delta": oracle_mod.backward(p, q, k, v, np.zeros_like(o), do, lse),
        "sign of dS": (-good[0], -good[1], good[2]),
        "scale missing from dK": (good[0], good[1] / p.scale, good[2]),
        "transposed scores": (kq[1], kq[0], kq[2]),
        "window edge off by one": oracle_mod.backward(wider, q, k, v, o, do, lse),
    }
    for grad, fd in zip(good, fds):
        assert np.abs(grad - fd).max() <= _fd_tol(fd)
    for what, grads in mutants.items():
        miss = max(np.abs(g - fd).max() / _fd_tol(fd) for g, fd in zip(grads, fds))
        assert miss > 100, what


@pytest.mark.parametrize("name", ["dense", "causal_br_long_q", "padded", "gqa", "window_causal"])
def test_row_sum_invariants(oracle_mod, name):
    """With exact O: each row of dS sums to 0, so sum_k dK_k = 0 per (b, kv head);
    and sum_k dV_k equals the sum of dO over the group's non-empty query rows."""
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=3)
    o, lse = oracle_mod.forward(p, q, k, v)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    G = p.Hq // p.Hkv
    nonempty = np.isfinite(lse)
    for b in range(p.B):
        for hk in range(p.Hkv):
            np.testing.assert_allclose(dk[b, hk].sum(0), 0.0, atol=1e-12)
            heads = range(hk * G, hk * G + G)
            expect = sum(do[b, h][nonempty[b, h]].sum(0) for h in heads)
            np.testing.assert_allclose(dv[b, hk].sum(0), expect, atol=1e-12)


def test_dq_invariant_under_key_shift(oracle_mod):
    """Adding one vector c to every key row shifts each score row by a constant,
    so P is unchanged and (rows of dS summing to 0) dQ is unchanged."""
    p = Problem(1, 2, 2, 6, 9, 5, 4, causal=True, bottom_right=True)
    q, k, v, do = _inputs(p, seed=7)
    c = np.random.default_rng(1).standard_normal(p.Dqk)
    res = []
    for kk in (k, k + c):
        o, lse = oracle_mod.forward(p, q, kk, v)
        res.append(oracle_mod.backward(p, q, kk, v, o, do, lse))
    np.testing.assert_allclose(res[0][0], res[1][0], atol=1e-11)
    np.testing.assert_allclose(res[0][2], res[1][2], atol=1e-11)


def test_gqa_equals_replicated_mha(oracle_mod):
    """GQA with H_kv heads == MHA with each KV head repeated G times (query head h
    reads KV head h // G); dK/dV of a KV head == the sum over its group."""
    G, Hkv = 3, 2
    pg = Problem(2, G * Hkv, Hkv, 6, 7, 4, 5, causal=True, bottom_right=True)
    pm = Problem(2, G * Hkv, G * Hkv, 6, 7, 4, 5, causal=True, bottom_right=True)
    q, k, v, do = _inputs(pg, seed=11)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    og, lg = oracle_mod.forward(pg, q, k, v)
    om, lm = oracle_mod.forward(pm, q, kr, vr)
    np.testing.assert_allclose(og, om, atol=1e-13)
    np.testing.assert_allclose(lg, lm, atol=1e-13)
    dqg, dkg, dvg = oracle_mod.backward(pg, q, k, v, og, do, lg)
    dqm, dkm, dvm = oracle_mod.backward(pm, q, kr, vr, om, do, lm)
    np.testing.assert_allclose(dqg, dqm, atol=1e-13)
    np.testing.assert_allclose(dkg, dkm.reshape(2, Hkv, G, 7, 4).sum(2), atol=1e-12)
    np.testing.assert_allclose(dvg, dvm.reshape(2, Hkv, G, 7, 5).sum(2), atol=1e-12)


def test_fully_masked_rows_give_exact_zeros(oracle_mod):
    """Padded query rows and rows left empty by a bottom-right diagonal have
    LSE = -inf, O = 0 and exactly zero dQ; padded key rows get exactly zero dK/dV."""
    p = Problem(2, 2, 1, 8, 5, 4, 4, causal=True, bottom_right=True,
                seq_q_lens=np.array([8, 3]), seq_kv_lens=np.array([5, 2]))
    q, k, v, do = _inputs(p, seed=5)
    o, lse = oracle_mod.forward(p, q, k, v)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    # b=0: L_q=8, L_kv=5, diag=-3 -> rows q<3 see no key. b=1: L_q=3, L_kv=2, diag=-1.
    for b, (lq, lk, empty) in enumerate([(8, 5, [0, 1, 2]), (3, 2, [0])]):
        dead_q = sorted(set(empty) | set(range(lq, 8)))
        assert np.all(np.isneginf(lse[b][:, dead_q]))
        assert np.all(o[b][:, dead_q] == 0.0)
        assert np.all(dq[b][:, dead_q] == 0.0)
        live = [i for i in range(8) if i not in dead_q]
        assert np.all(np.isfinite(lse[b][:, live]))
        assert np.all(dk[b][:, lk:] == 0.0) and np.all(dv[b][:, lk:] == 0.0)


def test_single_visible_key_closed_form(oracle_mod):
    """With one key, P = 1 and dS = 0: dQ = dK = 0 and dV = sum_q dO_q; O = V."""
    p = Problem(1, 2, 1, 5, 1, 4, 3)
    q, k, v, do = _inputs(p, seed=2)
    o, lse = oracle_mod.forward(p, q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v[:, :1], o.shape), atol=1e-15)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    assert np.abs(dq).max() < 1e-15 and np.abs(dk).max() < 1e-15
    np.testing.assert_allclose(dv[0, 0, 0], do[0].sum(axis=(0, 1)), atol=1e-13)


def test_zero_query_gives_uniform_attention(oracle_mod):
    """Q = 0 makes every visible score 0, so O_q is the mean of the visible V rows
    and LSE_q = log(number of visible keys)."""
    p = Problem(1, 1, 1, 4, 6, 3, 2, causal=True, bottom_right=True)
    _, k, v, _ = _inputs(p, seed=4)
    q = np.zeros((1, 1, 4, 3))
    o, lse = oracle_mod.forward(p, q, k, v)
    for i in range(4):
        n = i + 3  # diag = 2: row i sees keys 0..i+2
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].mean(0), atol=1e-15)
        assert abs(lse[0, 0, i] - math.log(n)) < 1e-15


def test_two_keys_worked_by_hand(oracle_mod):
    g = json.load(open(os.path.join(HERE, "golden", "two_keys_by_hand.json")))
    p = Problem(1, 1, 1, 1, 2, 1, 1, scale=1.0)
    i = g["inputs"]
    q = np.array(i["q"]).reshape(1, 1, 1, 1)
    k = np.array(i["k"]).reshape(1, 1, 2, 1)
    v = np.array(i["v"]).reshape(1, 1, 2, 1)
    do = np.array(i["do"]).reshape(1, 1, 1, 1)
    o, lse = oracle_mod.forward(p, q, k, v)
    e = g["expected"]
    assert abs(lse.item() - e["lse"]) < 1e-14 and abs(o.item() - e["o"]) < 1e-14
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    assert abs(dq.item() - e["dq"]) < 1e-14
    np.testing.assert_allclose(dk.ravel(), e["dk"], atol=1e-14)
    np.testing.assert_allclose(dv.ravel(), e["dv"], atol=1e-14)


def _pairs_causal_window(L, W):
    """Visible pairs of one head, square causal top-left with left window W, length L:
    row q sees min(q + 1, W + 1) keys."""
    if L <= W + 1:
        return L * (L + 1) // 2
    return (W + 1) * (W + 2) // 2 + (L - W - 1) * (W + 1)


def test_visible_counts_match_closed_forms(oracle_mod):
    # Square top-left causal: S(S+1)/2 per head.
    p = Problem(2, 3, 3, 37, 37, 8, 8, causal=True)
    assert oracle_mod.count_visible(p) == 2 * 3 * 37 * 38 // 2
    # Bottom-right causal, S_q < S_kv: row q sees q + (S_kv - S_q) + 1 keys.
    p = Problem(1, 2, 1, 5, 12, 8, 8, causal=True, bottom_right=True)
    assert oracle_mod.count_visible(p) == 2 * sum(q + 7 + 1 for q in range(5))
    # Right band R = 3 on a square causal mask: row q sees min(q + 4, S) keys.
    p = Problem(1, 1, 1, 10, 10, 8, 8, causal=True, window_right=3)
    assert oracle_mod.count_visible(p) == sum(min(q + 4, 10) for q in range(10))
    # Causal + left window W with padding: closed form per batch length.
    lens = np.array([40, 200, 65, 129])
    p = Problem(4, 2, 2, 200, 200, 8, 8, causal=True, window_left=64,
                seq_q_lens=lens, seq_kv_lens=lens)
    assert oracle_mod.count_visible(p) == 2 * sum(_pairs_causal_window(int(L), 64) for L in lens)
    # Window with W = 1 and top-left causal: every row but the first sees 2 keys.
    p = Problem(1, 1, 1, 9, 9, 8, 8, causal=True, window_left=1)
    assert oracle_mod.count_visible(p) == 2 * 9 - 1
    # Non-causal left window only (keys to the right stay visible).
    p = Problem(1, 1, 1, 6, 6, 8, 8, window_left=2)
    assert oracle_mod.count_visible(p) == sum(6 - max(0, q - 2) for q in range(6))


def _torch_mask(p: Problem):
    """Boolean (B, 1, Sq, Skv) mask from tril/triu bands of torch (not the oracle's predicate)."""
    masks = []
    for b in range(p.B):
        Lq = p.Sq if p.seq_q_lens is None else int(p.seq_q_lens[b])
        Lk = p.Skv if p.seq_kv_lens is None else int(p.seq_kv_lens[b])
        diag = (Lk - Lq) if p.bottom_right else 0
        m = torch.ones(p.Sq, p.Skv, dtype=torch.bool)
        if p.causal:
            m &= torch.ones(p.Sq, p.Skv, dtype=torch.bool).tril(diag + max(p.window_right, 0))
        if p.window_left >= 0:
            m &= torch.ones(p.Sq, p.Skv, dtype=torch.bool).triu(diag - p.window_left)
        m[Lq:, :] = False
        m[:, Lk:] = False
        masks.append(m)
    return torch.stack(masks)[:, None]


@pytest.mark.parametrize("name", ["dense", "causal_tl", "causal_br_long_kv", "window_causal",
                                  "window_only", "padded", "gqa", "mqa_scale", "causal_band_r2"])
def test_matches_torch_sdpa_float64(oracle_mod, name):
    """Forward and backward against torch SDPA in float64 with autograd, on rows
    that see at least one key (torch returns NaN on empty rows)."""
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=9)
    o, lse = oracle_mod.forward(p, q, k, v)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    G = p.Hq // p.Hkv
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    mask = _torch_mask(p)
    rows = mask.any(-1)  # (B, 1, Sq)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1), attn_mask=mask,
        scale=p.resolved_scale)
    live = rows.expand(-1, p.Hq, -1)
    tdo = torch.tensor(do) * live[..., None]
    out = torch.where(live[..., None], out, torch.zeros_like(out))
    (out * tdo).sum().backward()
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    scores = (tq.detach() @ tk.detach().repeat_interleave(G, 1).transpose(-1, -2)) * p.resolved_scale
    tl = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), -1)
    np.testing.assert_allclose(lse[live.numpy()], tl[live].numpy(), atol=1e-12)
    # The oracle's dO on empty rows does not matter (P = 0 there); zero it to compare.
    do_live = do * live[..., None].numpy()
    dq2, dk2, dv2 = oracle_mod.backward(p, q, k, v, o, do_live, lse)
    np.testing.assert_allclose(dq2, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk2, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv2, tv.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dq, dq2, atol=1e-12)  # dO on empty rows has no effect


def test_sampled_rows_equal_full_backward(oracle_mod):
    p = FD_CASES["padded"]
    q, k, v, do = _inputs(p, seed=13)
    o, lse = oracle_mod.forward(p, q, k, v)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    qi = np.array([0, 5, 7, 13, 23])
    ki = np.array([1, 6, 9, 27])
    sq, sk, sv = oracle_mod.backward_sampled(p, q, k, v, o, do, lse, qi, ki)
    np.testing.assert_array_equal(sq, dq.reshape(-1, p.Dqk)[qi])
    np.testing.assert_array_equal(sk, dk.reshape(-1, p.Dqk)[ki])
    np.testing.assert_array_equal(sv, dv.reshape(-1, p.Dv)[ki])


def test_negative_infinite_lse_gives_zero_probability(oracle_mod):
    """A row whose given LSE is -inf replays P = 0 (not NaN/inf) even when keys are
    visible: its dQ is exactly 0 and it adds nothing to dK/dV (same result as
    zeroing that row's dO)."""
    p = Problem(1, 2, 1, 5, 6, 4, 4, causal=True, bottom_right=True)
    q, k, v, do = _inputs(p, seed=21)
    o, lse = oracle_mod.forward(p, q, k, v)
    lse_cut = lse.copy()
    lse_cut[0, 1, 3] = -np.inf
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse_cut)
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    assert np.all(dq[0, 1, 3] == 0.0)
    do_cut = do.copy()
    do_cut[0, 1, 3] = 0.0
    _, dk_ref, dv_ref = oracle_mod.backward(p, q, k, v, o, do_cut, lse)
    # with dO zeroed the row still has P != 0 but dP = 0 and delta = 0, so dS = 0 and P*dO = 0
    np.testing.assert_allclose(dk, dk_ref, atol=1e-13)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-13)


# ---------------------------------------------------------------- sink tokens
# A per-query-head sink logit joins every row's softmax denominator without a
# value row ("SDPA Backward (SM120)", Capabilities: sink tokens; kernel chain
# step `dsink`). The pins below fix the oracle's sink forward and dsink to
# central differences of L = sum(O * dO), to the no-sink limit and to a closed
# form, none of which the oracle computes that way.
SINK_CASES = ["dense", "causal_br_long_kv", "padded", "gqa", "window_causal"]


def _sink(p, seed):
    return np.random.default_rng(seed).standard_normal(p.Hq) * 0.8


@pytest.mark.parametrize("name", SINK_CASES)
def test_dsink_matches_central_differences(oracle_mod, name):
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=11)
    sink = _sink(p, 12)
    o, lse = oracle_mod.forward(p, q, k, v, sink)
    ds = oracle_mod.dsink(p, sink, lse, oracle_mod.delta(p, o, do))
    h = 1e-6
    fd = np.zeros(p.Hq)
    for i in range(p.Hq):
        sp, sm = sink.copy(), sink.copy()
        sp[i] += h
        sm[i] -= h
        op, _ = oracle_mod.forward(p, q, k, v, sp)
        om, _ = oracle_mod.forward(p, q, k, v, sm)
        fd[i] = float(np.sum((op - om) * do)) / (2 * h)
    np.testing.assert_allclose(ds, fd, rtol=0, atol=2e-7 * max(1.0, np.abs(fd).max()))


@pytest.mark.parametrize("name", ["causal_br_long_kv", "padded", "gqa"])
def test_sink_backward_matches_central_differences(oracle_mod, name):
    """With a sink the forward's LSE carries it, and dQ/dK/dV from the same
    formulas still match central differences of L = sum(O * dO)."""
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=13)
    sink = _sink(p, 14)
    o, lse = oracle_mod.forward(p, q, k, v, sink)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse)
    h = 1e-6
    for tensor, grad, which in ((q, dq, "q"), (k, dk, "k"), (v, dv, "v")):
        fd = np.zeros_like(tensor)
        it = np.nditer(tensor, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            for sgn in (1, -1):
                t = tensor.copy()
                t[idx] += sgn * h
                args[which] = t
                o2, _ = oracle_mod.forward(p, args["q"], args["k"], args["v"], sink)
                fd[idx] += sgn * float(np.sum(o2 * do)) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=0, atol=2e-7 * max(1.0, float(np.abs(fd).max())),
                                   err_msg=f"d{which}")


def test_sink_at_minus_infinity_is_no_sink(oracle_mod):
    p = FD_CASES["padded"]
    q, k, v, do = _inputs(p, seed=15)
    o0, lse0 = oracle_mod.forward(p, q, k, v)
    sink = np.full(p.Hq, -np.inf)
    o1, lse1 = oracle_mod.forward(p, q, k, v, sink)
    np.testing.assert_array_equal(o1, o0)
    np.testing.assert_array_equal(lse1, lse0)
    assert np.all(oracle_mod.dsink(p, sink, lse1, oracle_mod.delta(p, o1, do)) == 0.0)


def test_sink_single_key_closed_form(oracle_mod):
    """One key with score s and a sink logit c: LSE = log(e^s + e^c),
    O = V / (1 + e^(c - s)), and with delta = dO . O,
    dsink = -sum_q e^(c - LSE_q) delta_q."""
    p = Problem(1, 1, 1, 3, 1, 2, 2, scale=1.0)
    q = np.array([[[[0.5, -1.0], [2.0, 0.25], [-0.75, 0.0]]]])
    k = np.array([[[[1.0, 0.5]]]])
    v = np.array([[[[2.0, -3.0]]]])
    do = np.array([[[[1.0, 0.5], [-2.0, 1.5], [0.25, 0.25]]]])
    c = 0.4
    o, lse = oracle_mod.forward(p, q, k, v, np.array([c]))
    ds = oracle_mod.dsink(p, np.array([c]), lse, oracle_mod.delta(p, o, do))
    want_ds = 0.0
    for i in range(3):
        s = float(q[0, 0, i] @ k[0, 0, 0])
        assert abs(lse[0, 0, i] - math.log(math.exp(s) + math.exp(c))) < 1e-14
        w = 1.0 / (1.0 + math.exp(c - s))
        np.testing.assert_allclose(o[0, 0, i], w * v[0, 0, 0], atol=1e-15)
        want_ds -= (1.0 - w) * float(w * v[0, 0, 0] @ do[0, 0, i])
    assert abs(ds[0] - want_ds) < 1e-14


# ---- additive bias (Capabilities list: a (1|B, H_q, S_q, S_kv) tensor added
# after the scale and before the softmax, with its gradient dBias). The pins
# fix the oracle's biased forward, its backward and dBias to central
# differences, to torch's float attention mask under float64 autograd (which
# also differentiates the mask), to the mask it can stand in for, to softmax
# shift invariance and to one extra head dimension.
BIAS_CASES = ["dense", "causal_br_long_kv", "padded", "gqa", "window_causal"]


def _bias(p, seed, batch):
    return np.random.default_rng(seed).standard_normal((batch, p.Hq, p.Sq, p.Skv)) * 0.7


@pytest.mark.parametrize("batch1", [False, True])
@pytest.mark.parametrize("name", BIAS_CASES)
def test_dbias_matches_central_differences(oracle_mod, name, batch1):
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=21)
    bias = _bias(p, 22, 1 if batch1 else p.B)
    o, lse = oracle_mod.forward(p, q, k, v, bias=bias)
    db = oracle_mod.dbias(p, q, k, v, o, do, lse, bias)
    assert db.shape == bias.shape
    h = 1e-6
    fd = np.zeros_like(bias)
    it = np.nditer(bias, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        bp, bm = bias.copy(), bias.copy()
        bp[idx] += h
        bm[idx] -= h
        op, _ = oracle_mod.forward(p, q, k, v, bias=bp)
        om, _ = oracle_mod.forward(p, q, k, v, bias=bm)
        fd[idx] = float(np.sum((op - om) * do)) / (2 * h)
    np.testing.assert_allclose(db, fd, rtol=0, atol=2e-7 * max(1.0, float(np.abs(fd).max())))


@pytest.mark.parametrize("name,batch1", [("causal_br_long_kv", False), ("padded", True), ("gqa", False)])
def test_bias_backward_matches_central_differences(oracle_mod, name, batch1):
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=23)
    bias = _bias(p, 24, 1 if batch1 else p.B)
    o, lse = oracle_mod.forward(p, q, k, v, bias=bias)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse, bias=bias)
    h = 1e-6
    for tensor, grad, which in ((q, dq, "q"), (k, dk, "k"), (v, dv, "v")):
        fd = np.zeros_like(tensor)
        it = np.nditer(tensor, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            args = {"q": q, "k": k, "v": v}
            for sgn in (1, -1):
                t = tensor.copy()
                t[idx] += sgn * h
                args[which] = t
                o2, _ = oracle_mod.forward(p, args["q"], args["k"], args["v"], bias=bias)
                fd[idx] += sgn * float(np.sum(o2 * do)) / (2 * h)
        np.testing.assert_allclose(grad, fd, rtol=0, atol=2e-7 * max(1.0, float(np.abs(fd).max())),
                                   err_msg=f"d{which}")


@pytest.mark.parametrize("batch1", [False, True])
@pytest.mark.parametrize("name", ["dense", "causal_tl", "window_only", "padded", "gqa", "mqa_scale"])
def test_bias_matches_torch_sdpa_float64(oracle_mod, name, batch1):
    """torch SDPA adds a float attn_mask to the scaled scores; under float64
    autograd it returns dQ/dK/dV and the mask's gradient (summed over the batch
    when the mask broadcasts), on rows that see at least one key."""
    p = FD_CASES[name]
    q, k, v, do = _inputs(p, seed=25)
    bias = _bias(p, 26, 1 if batch1 else p.B)
    G = p.Hq // p.Hkv
    mask = _torch_mask(p)
    rows = mask.any(-1)
    live = rows.expand(-1, p.Hq, -1)
    do = do * live[..., None].numpy()  # dO on empty rows is irrelevant to the oracle
    o, lse = oracle_mod.forward(p, q, k, v, bias=bias)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse, bias=bias)
    db = oracle_mod.dbias(p, q, k, v, o, do, lse, bias)
    tq = torch.tensor(q, requires_grad=True)
    tk = torch.tensor(k, requires_grad=True)
    tv = torch.tensor(v, requires_grad=True)
    tb = torch.tensor(bias, requires_grad=True)
    add = tb.masked_fill(~mask, float("-inf")) if batch1 is False else \
        tb.expand(p.B, -1, -1, -1).masked_fill(~mask, float("-inf"))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(G, 1), tv.repeat_interleave(G, 1), attn_mask=add,
        scale=p.resolved_scale)
    out = torch.where(live[..., None], out, torch.zeros_like(out))
    (out * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(o, out.detach().numpy(), atol=1e-12)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)
    tgrad = torch.nan_to_num(tb.grad, nan=0.0).numpy()
    np.testing.assert_allclose(db, tgrad, atol=1e-11)


def test_minus_infinity_bias_equals_the_causal_mask(oracle_mod):
    """A bias of -inf above the diagonal reproduces causal=True: the bias is
    indexed (query, key), not transposed."""
    pc = Problem(2, 2, 1, 6, 9, 4, 3, causal=True, bottom_right=True)
    pn = Problem(2, 2, 1, 6, 9, 4, 3)
    q, k, v, do = _inputs(pc, seed=27)
    diag = 9 - 6
    qi, ki = np.meshgrid(np.arange(6), np.arange(9), indexing="ij")
    bias = np.where(ki > qi + diag, -np.inf, 0.0)[None, None].repeat(2, 0).repeat(2, 1)
    o0, lse0 = oracle_mod.forward(pc, q, k, v)
    o1, lse1 = oracle_mod.forward(pn, q, k, v, bias=bias)
    np.testing.assert_allclose(o1, o0, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0, atol=1e-14)
    g0 = oracle_mod.backward(pc, q, k, v, o0, do, lse0)
    g1 = oracle_mod.backward(pn, q, k, v, o1, do, lse1, bias=bias)
    for a, b in zip(g1, g0):
        np.testing.assert_allclose(a, b, atol=1e-13)
    db = oracle_mod.dbias(pn, q, k, v, o1, do, lse1, bias)
    assert np.all(db[..., ki > qi + diag] == 0.0)


def test_row_constant_bias_only_shifts_lse(oracle_mod):
    """bias[q, k] = c_q: softmax is shift invariant, so O and dQ/dK/dV are
    unchanged, LSE moves by c_q, and every dBias row sums to zero."""
    p = FD_CASES["window_causal"]
    q, k, v, do = _inputs(p, seed=28)
    c = np.random.default_rng(29).standard_normal((p.B, p.Hq, p.Sq))
    bias = np.repeat(c[..., None], p.Skv, -1)
    o0, lse0 = oracle_mod.forward(p, q, k, v)
    o1, lse1 = oracle_mod.forward(p, q, k, v, bias=bias)
    np.testing.assert_allclose(o1, o0, atol=1e-14)
    np.testing.assert_allclose(lse1, lse0 + c, atol=1e-13)
    for a, b in zip(oracle_mod.backward(p, q, k, v, o1, do, lse1, bias=bias),
                    oracle_mod.backward(p, q, k, v, o0, do, lse0)):
        np.testing.assert_allclose(a, b, atol=1e-13)
    db = oracle_mod.dbias(p, q, k, v, o1, do, lse1, bias)
    np.testing.assert_allclose(db.sum(-1), 0.0, atol=1e-13)


def test_rank_one_bias_equals_one_more_head_dim(oracle_mod):
    """bias[q, k] = u_q w_k is one more head dimension with Q' = [Q, u / scale]
    and K' = [K, w]: O and LSE agree, dQ and dK agree on the first D_qk columns,
    and sum_k dBias[q, k] w_k = dQ'[q, D_qk] / scale."""
    p = Problem(1, 2, 2, 5, 7, 3, 4, causal=True, bottom_right=True)
    pa = Problem(1, 2, 2, 5, 7, 4, 4, causal=True, bottom_right=True, scale=p.resolved_scale)
    q, k, v, do = _inputs(p, seed=30)
    rng = np.random.default_rng(31)
    u = rng.standard_normal((1, 2, 5))
    w = rng.standard_normal((1, 2, 7))
    bias = u[..., :, None] * w[..., None, :]
    qa = np.concatenate([q, (u / p.resolved_scale)[..., None]], -1)
    ka = np.concatenate([k, w[..., None]], -1)
    o, lse = oracle_mod.forward(p, q, k, v, bias=bias)
    oa, lsea = oracle_mod.forward(pa, qa, ka, v)
    np.testing.assert_allclose(o, oa, atol=1e-14)
    np.testing.assert_allclose(lse, lsea, atol=1e-14)
    dq, dk, dv = oracle_mod.backward(p, q, k, v, o, do, lse, bias=bias)
    dqa, dka, dva = oracle_mod.backward(pa, qa, ka, v, oa, do, lsea)
    np.testing.assert_allclose(dq, dqa[..., :3], atol=1e-13)
    np.testing.assert_allclose(dk, dka[..., :3], atol=1e-13)
    np.testing.assert_allclose(dv, dva, atol=1e-13)
    db = oracle_mod.dbias(p, q, k, v, o, do, lse, bias)
    np.testing.assert_allclose((db * w[..., None, :]).sum(-1), dqa[..., 3] / p.resolved_scale,
                               atol=1e-13)


def test_dbias_rows_equal_full_dbias(oracle_mod):
    for batch1 in (False, True):
        p = FD_CASES["padded"]
        q, k, v, do = _inputs(p, seed=32)
        bias = _bias(p, 33, 1 if batch1 else p.B)
        o, lse = oracle_mod.forward(p, q, k, v, bias=bias)
        full = oracle_mod.dbias(p, q, k, v, o, do, lse, bias).reshape(-1, p.Skv)
        rows = [0, 3, 5, full.shape[0] - 1]
        np.testing.assert_array_equal(oracle_mod.dbias_rows(p, q, k, v, o, do, lse, bias, rows),
                                      full[rows])


# ---- NVFP4 QAT ("NVFP4 Attention QAT Backward" page, Overview). The pins fix the
# oracle's E4M3 / E2M1 rounding to brute force over every code of each format
# (decoded from its bit fields here) and to torch's float8_e4m3fn cast, its
# block fake quantization to a block worked by hand, and its QAT backward to
# the plain (pinned) backward on the quantized operands for dQ/dK and to a
# fake-quantized P built here, independently, for dV and the QAT forward.
def _e4m3_values():
    vals = []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue  # NaN
            vals.append((m / 8 * 2.0 ** -6) if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals), np.array([m for e in range(16) for m in range(8) if not (e == 15 and m == 7)])


def _e2m1_values():
    vals, mant = [], []
    for e in range(4):
        for m in range(2):
            vals.append(m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1))
            mant.append(m)
    return np.array(vals), np.array(mant)


def _nearest(x, vals, mant, top):
    a = min(abs(x), top)
    d = np.abs(vals - a)
    best = np.flatnonzero(d == d.min())
    if len(best) > 1:  # a tie: the even mantissa
        best = [b for b in best if mant[b] % 2 == 0]
    q = vals[best[0]]
    return -q if x < 0 else q


def _probe_points(vals, rng):
    v = np.unique(vals)
    mids = (v[1:] + v[:-1]) / 2
    pts = np.concatenate([v, mids, mids * (1 + 1e-9), mids * (1 - 1e-9), v * 1.3,
                          rng.uniform(0, v.max() * 1.2, 400)])
    return np.concatenate([pts, -pts])


def test_e4m3_rounding_matches_brute_force_and_torch(oracle_mod):
    vals, mant = _e4m3_values()
    rng = np.random.default_rng(40)
    pts = _probe_points(vals, rng)
    for x in pts:
        assert oracle_mod.round_e4m3(x) == _nearest(x, vals, mant, 448.0), x
    # torch casts through fp32, so compare on fp32 inputs (no double rounding)
    inr = pts[np.abs(pts) <= 448.0].astype(np.float32).astype(np.float64)
    t = torch.tensor(inr, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.array([oracle_mod.round_e4m3(x) for x in inr]), t)


def test_e2m1_rounding_matches_brute_force(oracle_mod):
    vals, mant = _e2m1_values()
    rng = np.random.default_rng(41)
    for x in _probe_points(vals, rng):
        assert oracle_mod.round_e2m1(x) == _nearest(x, vals, mant, 6.0), x


def test_fake_nvfp4_block_worked_by_hand(oracle_mod):
    """amax 1.25: scale = E4M3(1.25/6 = 0.2083) = 0.203125 (13/64; the E4M3
    neighbours are 0.203125 and 0.21875); 0.1 -> 0.1/0.203125 = 0.49 -> 0.5 ->
    0.1015625; -0.5 -> -2.46 -> -2 -> -0.40625; 1.25 -> 6.15 -> 6 -> 1.21875."""
    x = np.zeros((2, 32))
    x[0, :4] = [1.25, 0.1, -0.5, 0.3]
    x[0, 16:20] = [6.0, -3.0, 1.5, 0.5]        # scale 1: E2M1 values are kept
    x[1, :2] = [1e4, 100.0]                     # scale saturates at 448
    y = oracle_mod.fake_nvfp4(x)
    np.testing.assert_array_equal(y[0, :4], [1.21875, 0.1015625, -0.40625, 0.3046875])
    np.testing.assert_array_equal(y[0, 16:20], [6.0, -3.0, 1.5, 0.5])
    assert np.all(y[0, 4:16] == 0) and np.all(y[0, 20:] == 0)
    # 1e4/448 = 22.3 saturates to 6; 100/448 = 0.223 rounds to 0
    np.testing.assert_array_equal(y[1, :2], [6 * 448.0, 0.0])
    assert np.all(y[1, 16:] == 0)  # an all-zero block stays zero


def test_fake_nvfp4_invariants(oracle_mod):
    rng = np.random.default_rng(42)
    x = rng.standard_normal((64, 48)) * rng.uniform(0.01, 50, (64, 1))
    y = oracle_mod.fake_nvfp4(x)
    np.testing.assert_array_equal(oracle_mod.fake_nvfp4(y), y)       # idempotent
    np.testing.assert_array_equal(oracle_mod.fake_nvfp4(-x), -y)     # odd
    np.testing.assert_array_equal(oracle_mod.fake_nvfp4(4 * x), 4 * y)  # power-of-two scaling
    x2 = x.copy()
    x2[:, 16:32] *= 3.0
    np.testing.assert_array_equal(oracle_mod.fake_nvfp4(x2)[:, :16], y[:, :16])  # blocks independent
    assert np.all(np.abs(y - x) <= np.abs(x).reshape(64, 3, 16).max(-1).repeat(16, -1) / 6 * 1.07 + 1e-12)


def _fq_independent(x):
    """Fake quantization written here from the brute-force format tables."""
    ev, em = _e4m3_values()
    fv, fm = _e2m1_values()
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    flat, oflat = x.reshape(-1, x.shape[-1]), out.reshape(-1, x.shape[-1])
    for r in range(flat.shape[0]):
        for c0 in range(0, flat.shape[1], 16):
            blk = flat[r, c0:c0 + 16].astype(np.float32)
            amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
            s = np.float32(_nearest(float(amax / np.float32(6.0)), ev, em, 448.0))
            if s == 0:
                continue
            oflat[r, c0:c0 + 16] = [_nearest(float(v / s), fv, fm, 6.0) * float(s) for v in blk]
    return out


def test_qat_oracle_against_independent_pieces(oracle_mod):
    p = Problem(1, 2, 2, 9, 21, 32, 16, causal=True, bottom_right=True)
    q, k, v, do = _inputs(p, seed=43)
    o_hp, lse, o_user = oracle_mod.qat_forward(p, q, k, v)
    qh, kh, vh = _fq_independent(q), _fq_independent(k), _fq_independent(v)
    np.testing.assert_array_equal(oracle_mod.fake_nvfp4(q), qh)
    # O_hp / LSE: the plain forward of the quantized operands
    o2, lse2 = oracle_mod.forward(p, qh, kh, vh)
    np.testing.assert_array_equal(o_hp, o2)
    np.testing.assert_array_equal(lse, lse2)
    # P from the quantized scores (torch mask helper), fake-quantized along keys
    mask = _torch_mask(p).numpy()[:, 0]
    s = np.einsum("bhqd,bhkd->bhqk", qh, kh) * p.resolved_scale
    P = np.where(mask[:, None], np.exp(s - lse[..., None]), 0.0)
    Ph = _fq_independent(P)
    np.testing.assert_allclose(o_user, np.einsum("bhqk,bhkd->bhqd", Ph, vh), atol=1e-12)
    dq, dk, dv = oracle_mod.qat_backward(p, q, k, v, o_hp, do, lse)
    rq, rk, rv = oracle_mod.backward(p, qh, kh, vh, o_hp, do, lse)  # straight-through dQ, dK
    np.testing.assert_allclose(dq, rq, atol=1e-13)
    np.testing.assert_allclose(dk, rk, atol=1e-13)
    np.testing.assert_allclose(dv, np.einsum("bhqk,bhqd->bhkd", Ph, do), atol=1e-12)
    assert np.abs(dv - rv).max() > 1e-6  # the quantized P really differs from P


def test_qat_backward_gqa_sums_group_heads(oracle_mod):
    """dK/dV of a KV head equal the sums of an explicit MHA problem over its group."""
    p = Problem(1, 4, 2, 7, 18, 32, 32, causal=True)
    q, k, v, do = _inputs(p, seed=44)
    o, lse, _ = oracle_mod.qat_forward(p, q, k, v)
    dq, dk, dv = oracle_mod.qat_backward(p, q, k, v, o, do, lse)
    pm = Problem(1, 4, 4, 7, 18, 32, 32, causal=True)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    dq2, dk2, dv2 = oracle_mod.qat_backward(pm, q, kr, vr, o, do, lse)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(1, 2, 2, 18, 32).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(1, 2, 2, 18, 32).sum(2), atol=1e-13)


@pytest.mark.parametrize("name", ["padded", "window_causal", "window_only"])
def test_qat_oracle_under_masks(oracle_mod, name):
    """The QAT backward under padding and windows: dQ/dK are the plain backward
    of the quantized operands, dV uses the independently quantized P (masked
    entries 0 inside their 16-key blocks); D 16/32 so that blocks are whole."""
    base = FD_CASES[name]
    p = Problem(base.B, base.Hq, base.Hkv, base.Sq, base.Skv, 32, 16, causal=base.causal,
                bottom_right=base.bottom_right, window_left=base.window_left,
                window_right=base.window_right, seq_q_lens=base.seq_q_lens,
                seq_kv_lens=base.seq_kv_lens)
    q, k, v, do = _inputs(p, seed=45)
    o_hp, lse, _ = oracle_mod.qat_forward(p, q, k, v)
    qh, kh, vh = _fq_independent(q), _fq_independent(k), _fq_independent(v)
    dq, dk, dv = oracle_mod.qat_backward(p, q, k, v, o_hp, do, lse)
    rq, rk, _ = oracle_mod.backward(p, qh, kh, vh, o_hp, do, lse)
    np.testing.assert_allclose(dq, rq, atol=1e-13)
    np.testing.assert_allclose(dk, rk, atol=1e-13)
    mask = _torch_mask(p).numpy()[:, 0]
    s = np.einsum("bhqd,bhkd->bhqk", qh, np.repeat(kh, p.Hq // p.Hkv, axis=1)) * p.resolved_scale
    with np.errstate(invalid="ignore", over="ignore"):
        P = np.where(mask[:, None], np.exp(s - lse[..., None]), 0.0)
    P = np.nan_to_num(P, nan=0.0, posinf=0.0)
    Ph = _fq_independent(P)
    dv_ref = np.einsum("bhqk,bhqd->bhkd", Ph, do)
    dv_ref = dv_ref.reshape(p.B, p.Hkv, p.Hq // p.Hkv, p.Skv, p.Dv).sum(2)
    np.testing.assert_allclose(dv, dv_ref, atol=1e-12)
