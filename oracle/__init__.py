"""fp64 CPU oracle for the SDPA backward (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The GPU library never does, and this package
imports nothing from it: the two share no code.

The arithmetic lives in ``sdpa_oracle.c`` (plain definitions in double
precision, see its header for the page sections it follows). This module only
marshals numpy float64 arrays into it through ctypes.

Layout of every tensor: contiguous (B, H, S, D); LSE and delta are (B, H, S).
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))


class _Cfg(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("Sq", ctypes.c_int), ("Skv", ctypes.c_int), ("Dqk", ctypes.c_int), ("Dv", ctypes.c_int),
        ("scale", ctypes.c_double),
        ("causal", ctypes.c_int), ("bottom_right", ctypes.c_int),
        ("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
        ("seq_q_lens", ctypes.POINTER(ctypes.c_int32)),
        ("seq_kv_lens", ctypes.POINTER(ctypes.c_int32)),
        ("bias", ctypes.POINTER(ctypes.c_double)),
        ("bias_batch", ctypes.c_int),
    ]


@dataclass
class Problem:
    """Shape and mask of one attention problem (mirrors the C struct)."""
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    Dqk: int
    Dv: int
    scale: Optional[float] = None   # None -> 1/sqrt(Dqk)
    causal: bool = False
    bottom_right: bool = False
    window_left: int = -1
    window_right: int = -1
    seq_q_lens: Optional[np.ndarray] = None
    seq_kv_lens: Optional[np.ndarray] = None

    @property
    def resolved_scale(self) -> float:
        return 1.0 / math.sqrt(self.Dqk) if self.scale is None else float(self.scale)

    def _struct(self, bias=None):
        keep = []

        def lens(a):
            if a is None:
                return ctypes.POINTER(ctypes.c_int32)()
            arr = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
            keep.append(arr)
            return arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))

        s = _Cfg(self.B, self.Hq, self.Hkv, self.Sq, self.Skv, self.Dqk, self.Dv,
                 self.resolved_scale, int(self.causal), int(self.bottom_right),
                 int(self.window_left), int(self.window_right),
                 lens(self.seq_q_lens), lens(self.seq_kv_lens),
                 ctypes.POINTER(ctypes.c_double)(), 0)
        if bias is not None:
            arr = self.check_bias(bias)
            keep.append(arr)
            s.bias = _p(arr)
            s.bias_batch = arr.shape[0]
        return s, keep

    def check_bias(self, bias):
        """The bias as a contiguous float64 (1|B, Hq, Sq, Skv) array."""
        arr = np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
        if arr.ndim != 4 or arr.shape[0] not in (1, self.B) or \
                tuple(arr.shape[1:]) != (self.Hq, self.Sq, self.Skv):
            raise ValueError(f"bias must be (1|B, Hq, Sq, Skv), got {arr.shape}")
        return arr


_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.library_path()
        if not os.path.exists(path) or _build.is_stale():
            _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.POINTER(ctypes.c_double)
        C = ctypes.POINTER(_Cfg)
        I64 = ctypes.POINTER(ctypes.c_int64)
        lib.oracle_forward.argtypes = [C, P, P, P, P, P]
        lib.oracle_forward_sink.argtypes = [C, P, P, P, P, P, P]
        lib.oracle_dsink.argtypes = [C, P, P, P, P]
        lib.oracle_delta.argtypes = [C, P, P, P]
        lib.oracle_backward.argtypes = [C, P, P, P, P, P, P, P, P, P]
        lib.oracle_backward_sampled.argtypes = [C, P, P, P, P, P, P, ctypes.c_long, I64, P,
                                                ctypes.c_long, I64, P, P]
        lib.oracle_dbias.argtypes = [C, P, P, P, P, P, P, P]
        lib.oracle_dbias_rows.argtypes = [C, P, P, P, P, P, P, ctypes.c_long, I64, P]
        lib.oracle_round_e4m3.argtypes = [ctypes.c_double]
        lib.oracle_round_e4m3.restype = ctypes.c_double
        lib.oracle_round_e2m1.argtypes = [ctypes.c_double]
        lib.oracle_round_e2m1.restype = ctypes.c_double
        lib.oracle_fake_nvfp4.argtypes = [P, P, ctypes.c_long, ctypes.c_int]
        lib.oracle_qat_forward.argtypes = [C, P, P, P, P, P, P]
        lib.oracle_qat_backward.argtypes = [C, P, P, P, P, P, P, P, P, P]
        lib.oracle_count_visible.argtypes = [C]
        lib.oracle_count_visible.restype = ctypes.c_longlong
        lib.oracle_max_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        _lib = lib
    return _lib


def _f64(a, shape=None):
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and tuple(arr.shape) != tuple(shape):
        raise ValueError(f"expected shape {tuple(shape)}, got {tuple(arr.shape)}")
    return arr


def _p(a):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _check_heads(p: Problem):
    if p.Hkv <= 0 or p.Hq % p.Hkv != 0:
        raise ValueError("H_kv must divide H_q")


def forward(p: Problem, q, k, v, sink=None, bias=None):
    """Returns (O, LSE) in float64; LSE is the natural-log row log-sum-exp.
    ``sink`` (H_q,) adds a per-head sink logit to every row's denominator;
    ``bias`` (1|B, H_q, S_q, S_kv) is added to the scaled scores."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = np.zeros((p.B, p.Hq, p.Sq, p.Dv))
    lse = np.zeros((p.B, p.Hq, p.Sq))
    s, keep = p._struct(bias)
    if sink is None:
        lib.oracle_forward(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(lse))
    else:
        sk = _f64(sink, (p.Hq,))
        lib.oracle_forward_sink(ctypes.byref(s), _p(q), _p(k), _p(v), _p(sk), _p(o), _p(lse))
    return o, lse


def dsink(p: Problem, sink, lse, delta_):
    """dsink[h] = -sum_{b, q < L_q} exp(sink[h] - LSE[b,h,q]) * delta[b,h,q], shape (H_q,)."""
    lib = _load()
    sk = _f64(sink, (p.Hq,))
    lse = _f64(lse, (p.B, p.Hq, p.Sq))
    dl = _f64(delta_, (p.B, p.Hq, p.Sq))
    out = np.zeros(p.Hq)
    s, keep = p._struct()
    lib.oracle_dsink(ctypes.byref(s), _p(sk), _p(lse), _p(dl), _p(out))
    return out


def delta(p: Problem, o, do):
    """delta = rowsum(O * dO), shape (B, Hq, Sq)."""
    lib = _load()
    o = _f64(o, (p.B, p.Hq, p.Sq, p.Dv))
    do = _f64(do, (p.B, p.Hq, p.Sq, p.Dv))
    out = np.zeros((p.B, p.Hq, p.Sq))
    s, keep = p._struct()
    lib.oracle_delta(ctypes.byref(s), _p(o), _p(do), _p(out))
    return out


def backward(p: Problem, q, k, v, o, do, lse, bias=None):
    """Returns (dQ, dK, dV) in float64 from the given forward tensors (``bias``
    as in forward(): the replayed P includes it)."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = _f64(o, (p.B, p.Hq, p.Sq, p.Dv))
    do = _f64(do, (p.B, p.Hq, p.Sq, p.Dv))
    lse = _f64(lse, (p.B, p.Hq, p.Sq))
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    s, keep = p._struct(bias)
    lib.oracle_backward(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse),
                        _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


def backward_sampled(p: Problem, q, k, v, o, do, lse, q_rows, kv_rows, bias=None):
    """dQ at the flat query rows ``q_rows`` ((b*Hq + h)*Sq + q) and dK/dV at the
    flat key rows ``kv_rows`` ((b*Hkv + hk)*Skv + k). Returns three 2-D arrays."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = _f64(o, (p.B, p.Hq, p.Sq, p.Dv))
    do = _f64(do, (p.B, p.Hq, p.Sq, p.Dv))
    lse = _f64(lse, (p.B, p.Hq, p.Sq))
    qi = np.ascontiguousarray(np.asarray(q_rows, dtype=np.int64))
    ki = np.ascontiguousarray(np.asarray(kv_rows, dtype=np.int64))
    dq = np.zeros((len(qi), p.Dqk))
    dk = np.zeros((len(ki), p.Dqk))
    dv = np.zeros((len(ki), p.Dv))
    s, keep = p._struct(bias)
    I64 = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_backward_sampled(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse),
                                len(qi), qi.ctypes.data_as(I64), _p(dq),
                                len(ki), ki.ctypes.data_as(I64), _p(dk), _p(dv))
    return dq, dk, dv


def dbias(p: Problem, q, k, v, o, do, lse, bias):
    """Gradient of the additive bias: dS = P * (dP - delta) at visible pairs,
    shaped like ``bias``; a one-batch bias gets the sum over the batch rows."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = _f64(o, (p.B, p.Hq, p.Sq, p.Dv))
    do = _f64(do, (p.B, p.Hq, p.Sq, p.Dv))
    lse = _f64(lse, (p.B, p.Hq, p.Sq))
    s, keep = p._struct(bias)
    out = np.zeros((s.bias_batch, p.Hq, p.Sq, p.Skv))
    lib.oracle_dbias(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(out))
    return out


def dbias_rows(p: Problem, q, k, v, o, do, lse, bias, rows):
    """dbias() at the flat bias rows ``rows`` ((bb * Hq + h) * Sq + q), (len(rows), Skv)."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = _f64(o, (p.B, p.Hq, p.Sq, p.Dv))
    do = _f64(do, (p.B, p.Hq, p.Sq, p.Dv))
    lse = _f64(lse, (p.B, p.Hq, p.Sq))
    s, keep = p._struct(bias)
    ri = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if ri.size and (ri.min() < 0 or ri.max() >= s.bias_batch * p.Hq * p.Sq):
        raise ValueError("bias row out of range")
    out = np.zeros((len(ri), p.Skv))
    lib.oracle_dbias_rows(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), len(ri),
                          ri.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _p(out))
    return out


def round_e4m3(x: float) -> float:
    """Nearest E4M3 value (ties to even, saturating at 448)."""
    return float(_load().oracle_round_e4m3(float(x)))


def round_e2m1(x: float) -> float:
    """Nearest E2M1 value (ties to even, saturating at 6)."""
    return float(_load().oracle_round_e2m1(float(x)))


def fake_nvfp4(x):
    """NVFP4 fake quantization along the last axis, blocks of 16 values: E4M3
    local scale amax/6, values rounded to E2M1 multiples of it (float64 out)."""
    arr = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.zeros_like(arr)
    cols = arr.shape[-1] if arr.ndim else 1
    rows = arr.size // cols if cols else 0
    _load().oracle_fake_nvfp4(_p(arr), _p(out), rows, cols)
    return out


def qat_forward(p: Problem, q, k, v):
    """NVFP4 QAT forward: (O_hp, LSE, O_user). O_hp and LSE are the forward of
    the fake-quantized Q, K, V; O_user = fake_nvfp4(P) V_hat."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = np.zeros((p.B, p.Hq, p.Sq, p.Dv))
    lse = np.zeros((p.B, p.Hq, p.Sq))
    ou = np.zeros_like(o)
    s, keep = p._struct()
    lib.oracle_qat_forward(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(lse), _p(ou))
    return o, lse, ou


def qat_backward(p: Problem, q, k, v, o_hp, do, lse):
    """NVFP4 QAT backward: (dQ, dK, dV) from the unquantized Q, K, V, the
    high-precision forward output O_hp and its LSE."""
    _check_heads(p)
    lib = _load()
    q = _f64(q, (p.B, p.Hq, p.Sq, p.Dqk))
    k = _f64(k, (p.B, p.Hkv, p.Skv, p.Dqk))
    v = _f64(v, (p.B, p.Hkv, p.Skv, p.Dv))
    o = _f64(o_hp, (p.B, p.Hq, p.Sq, p.Dv))
    do = _f64(do, (p.B, p.Hq, p.Sq, p.Dv))
    lse = _f64(lse, (p.B, p.Hq, p.Sq))
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    s, keep = p._struct()
    lib.oracle_qat_backward(ctypes.byref(s), _p(q), _p(k), _p(v), _p(o), _p(do), _p(lse),
                            _p(dq), _p(dk), _p(dv))
    return dq, dk, dv


def count_visible(p: Problem) -> int:
    """Visible (q, k) pairs summed over batches and query heads."""
    lib = _load()
    s, keep = p._struct()
    return int(lib.oracle_count_visible(ctypes.byref(s)))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))
