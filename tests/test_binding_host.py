"""The Python binding's argument marshalling, without a GPU: CPU tensors stand in
for device tensors (``is_cuda`` patched to True) and a recording stand-in
replaces the shared library, so each call's route (which C entry point), its
argument count against the real library's declared signature, and the returned
tuple are checked. Nothing here launches a kernel."""
import ctypes

import pytest
import torch

import attention_backward_sdpa_gb300 as pkg


class _Recorder:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def fn(*args):
            self.calls.append((name, args))
            return 0
        return fn


@pytest.fixture
def fake(monkeypatch):
    real = pkg.load(build_if_missing=True)
    rec = _Recorder()
    monkeypatch.setattr(pkg, "load", lambda build_if_missing=False: rec)
    monkeypatch.setattr(pkg, "_stream_handle", lambda stream=None: None)
    monkeypatch.setattr(pkg, "_check_launch_device", lambda ref: None)
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    rec.real = real
    return rec


def _last(rec, name):
    called, args = rec.calls[-1]
    assert called == name
    assert len(args) == len(getattr(rec.real, name).argtypes), name
    return args


def _qkv(io=torch.bfloat16, B=2, Hq=4, Hkv=2, S=96, D=64):
    q = torch.zeros(B, Hq, S, D, dtype=io)
    k = torch.zeros(B, Hkv, S, D, dtype=io)
    v = torch.zeros(B, Hkv, S, D, dtype=io)
    lse = torch.zeros(B, Hq, S)
    return q, k, v, q.clone(), q.clone(), lse


def test_backward_routes(fake):
    q, k, v, o, do, lse = _qkv()
    dq, dk, dv = pkg.sdpa_bwd(q, k, v, o, do, lse, causal=True)
    args = _last(fake, "sdpa_bwd")
    assert args[9:16] == (2, 4, 2, 96, 96, 64, 64) and args[17] == 1
    assert dq.shape == q.shape and dk.shape == k.shape and dv.shape == v.shape

    sink = torch.zeros(4)
    out = pkg.sdpa_bwd(q, k, v, o, do, lse, sink=sink)
    _last(fake, "sdpa_bwd_sink")
    assert len(out) == 4 and out[3].shape == (4,)

    bias = torch.zeros(1, 4, 96, 96)
    out = pkg.sdpa_bwd(q, k, v, o, do, lse, bias=bias)
    args = _last(fake, "sdpa_bwd_bias")
    assert len(out) == 4 and out[3].dtype == torch.float32 and out[3].shape == bias.shape
    assert args[-4:-2] == (pkg.DTYPE_F32, 1)

    out = pkg.sdpa_bwd(q, k, v, o, do, lse, bias=bias.to(torch.bfloat16), bias_grad=False)
    args = _last(fake, "sdpa_bwd_bias")
    assert len(out) == 3 and args[-2] is None

    out = pkg.sdpa_bwd(q, k, v, o, do, lse, bias=bias, dbias_dtype=torch.bfloat16, sink=sink)
    args = _last(fake, "sdpa_bwd_typed")
    assert args[0] == 0 and args[-2] == pkg.DTYPE_BF16 and len(out) == 5
    assert out[4].dtype == torch.bfloat16


def test_backward_fp16_io(fake):
    q, k, v, o, do, lse = _qkv(torch.float16)
    dq, dk, dv = pkg.sdpa_bwd(q, k, v, o, do, lse)
    args = _last(fake, "sdpa_bwd_typed")
    assert args[0] == 2 and dq.dtype == torch.float16
    with pytest.raises(ValueError):  # one element type for every tensor
        pkg.sdpa_bwd(q, k, v, o.to(torch.bfloat16), do, lse)


def test_backward_rejects_bad_sink_on_every_route(fake):
    q, k, v, o, do, lse = _qkv(torch.float16)
    with pytest.raises(ValueError, match="sink"):
        pkg.sdpa_bwd(q, k, v, o, do, lse, sink=torch.zeros(3))
    q, k, v, o, do, lse = _qkv()
    with pytest.raises(ValueError, match="sink"):
        pkg.sdpa_bwd(q, k, v, o, do, lse, sink=torch.zeros(4, dtype=torch.float16))


def test_forward_routes(fake):
    q, k, v, _, _, _ = _qkv()
    o, lse = pkg.sdpa_fwd(q, k, v, causal=True)
    _last(fake, "sdpa_fwd")
    assert o.shape == q.shape and lse.shape == (2, 4, 96)
    pkg.sdpa_fwd(q, k, v, bias=torch.zeros(2, 4, 96, 96, dtype=torch.float16))
    args = _last(fake, "sdpa_fwd_bias")
    assert args[-3:-1] == (pkg.DTYPE_F16, 2)
    q, k, v, _, _, _ = _qkv(torch.float16)
    o, _ = pkg.sdpa_fwd(q, k, v)
    assert _last(fake, "sdpa_fwd_typed")[0] == 2 and o.dtype == torch.float16


def test_qat_routes(fake):
    q, k, v, o, do, lse = _qkv(D=128)
    dq, dk, dv = pkg.sdpa_bwd_nvfp4_qat(q, k, v, o, do, lse, causal=True)
    _last(fake, "sdpa_bwd_nvfp4_qat")
    y = pkg.nvfp4_fake_quant(q)
    args = _last(fake, "sdpa_nvfp4_fake_quant")
    assert args[2] == q.numel() and y.shape == q.shape
    with pytest.raises(ValueError):
        pkg.sdpa_bwd_nvfp4_qat(q, k, v, o, do, lse, dq=torch.zeros(1))


def test_pointers_are_the_tensors(fake):
    q, k, v, o, do, lse = _qkv()
    ws = torch.zeros(1024, dtype=torch.uint8)
    dq, dk, dv = pkg.sdpa_bwd(q, k, v, o, do, lse, workspace=ws)
    args = _last(fake, "sdpa_bwd")
    ptrs = [a.value if isinstance(a, ctypes.c_void_p) else a for a in args[:9]]
    assert ptrs == [t.data_ptr() for t in (q, k, v, o, do, lse, dq, dk, dv)]
    assert args[-3].value == ws.data_ptr() and args[-2] == 1024
