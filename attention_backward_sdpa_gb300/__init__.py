"""GB300 (sm_103a) scaled-dot-product-attention backward.

A thin ctypes binding over ``libsdpa_bwd.so`` (C ABI in ``include/sdpa_bwd.h``).
Every step of the backward runs in the library's CUDA kernels; this module
only checks tensor properties and passes pointers, sizes and the current CUDA
stream. PyTorch is used for device memory and streams.

There is no fallback: if the library cannot be loaded, or the device is not
an sm_103 GPU, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

from . import _build

__all__ = ["sdpa_bwd", "sdpa_fwd", "workspace_size", "nvfp4_fake_quant", "sdpa_fwd_nvfp4_qat",
           "sdpa_bwd_nvfp4_qat", "nvfp4_qat_workspace_size", "check_device_status", "debug_relay",
           "profile_enable", "profile_read", "library_path", "load", "SdpaError", "KERNEL_NAMES"]

KERNEL_NAMES = ("preprocess", "main", "dq")

_STATUS = {0: "SDPA_OK", 1: "SDPA_ERR_INVALID", 2: "SDPA_ERR_UNSUPPORTED", 3: "SDPA_ERR_ALIGN",
           4: "SDPA_ERR_WORKSPACE", 5: "SDPA_ERR_CUDA", 6: "SDPA_ERR_TIMEOUT", 7: "SDPA_ERR_BOUNDS"}


class SdpaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_STATUS.get(code, code)} ({_lib_status_string(code)})")


_lib = None


def library_path() -> str:
    """The library this process loads: libsdpa_bwd.so, or the build named by the
    SDPA_BWD_LIBRARY environment variable (for example the debug-bounds build,
    libsdpa_bwd_debug.so, whose kernels check their global accesses)."""
    return os.environ.get("SDPA_BWD_LIBRARY") or _build.LIB


def load(build_if_missing: bool = False):
    """Loads libsdpa_bwd.so (optionally building it first) and declares its ABI."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if build_if_missing and (not os.path.exists(path) or _build.is_stale()):
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m attention_backward_sdpa_gb300._build`"
                           " (or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.sdpa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, ctypes.c_float,
                             i, i, i, i, i, vp, vp, vp, sz, vp]
    lib.sdpa_bwd.restype = i
    lib.sdpa_bwd_sink.argtypes = list(lib.sdpa_bwd.argtypes[:-1]) + [vp, vp, vp]
    lib.sdpa_bwd_sink.restype = i
    lib.sdpa_bwd_bias.argtypes = list(lib.sdpa_bwd.argtypes[:-1]) + [vp, vp, vp, i, i, vp, vp]
    lib.sdpa_bwd_bias.restype = i
    lib.sdpa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, ctypes.c_float, i, i, i, i,
                             vp, vp, vp, vp]
    lib.sdpa_fwd.restype = i
    lib.sdpa_fwd_bias.argtypes = list(lib.sdpa_fwd.argtypes[:-1]) + [vp, i, i, vp]
    lib.sdpa_fwd_bias.restype = i
    lib.sdpa_bwd_typed.argtypes = [i] + list(lib.sdpa_bwd.argtypes[:-1]) + [vp, vp, vp, i, i, vp, i, vp]
    lib.sdpa_bwd_typed.restype = i
    lib.sdpa_fwd_typed.argtypes = [i] + list(lib.sdpa_fwd.argtypes[:-1]) + [vp, i, i, vp]
    lib.sdpa_fwd_typed.restype = i
    lib.sdpa_nvfp4_fake_quant.argtypes = [vp, vp, ctypes.c_longlong, vp]
    lib.sdpa_nvfp4_fake_quant.restype = i
    lib.sdpa_bwd_nvfp4_qat_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.sdpa_bwd_nvfp4_qat_workspace_size.restype = sz
    lib.sdpa_bwd_nvfp4_qat.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i,
                                       ctypes.c_float, i, i, i, i, vp, vp, vp, sz, vp]
    lib.sdpa_bwd_nvfp4_qat.restype = i
    lib.sdpa_bwd_workspace_size.argtypes = [i] * 13
    lib.sdpa_bwd_workspace_size.restype = sz
    lib.sdpa_status_string.argtypes = [i]
    lib.sdpa_status_string.restype = ctypes.c_char_p
    lib.sdpa_bwd_debug_relay.argtypes = [ctypes.c_ulonglong, i]
    lib.sdpa_bwd_debug_relay.restype = i
    lib.sdpa_bwd_check_device_status.argtypes = [vp]
    lib.sdpa_bwd_check_device_status.restype = i
    lib.sdpa_bwd_profile_enable.argtypes = [i]
    lib.sdpa_bwd_profile_enable.restype = i
    lib.sdpa_bwd_profile_read.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), i]
    lib.sdpa_bwd_profile_read.restype = i
    lib.sdpa_bwd_version.restype = i
    _lib = lib
    return lib


def _lib_status_string(code: int) -> str:
    try:
        return load().sdpa_status_string(code).decode()
    except Exception:  # pragma: no cover - only used while formatting an error
        return "?"


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def workspace_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv, deterministic=False, *, causal=False,
                   bottom_right=False, window_left=-1, window_right=-1, padded=False) -> int:
    """Workspace bytes of sdpa_bwd for this shape and mask (``padded``: length
    arrays will be passed). The defaults (no mask) give the largest size for the
    shape, which serves every mask."""
    return int(load().sdpa_bwd_workspace_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv, int(causal),
                                              int(bottom_right), int(window_left),
                                              int(window_right), int(deterministic), int(padded)))


def _check_bf16(name, t, shape, dtype=torch.bfloat16):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check_lens(B, seq_q_lens, seq_kv_lens):
    for name, lens in (("seq_q_lens", seq_q_lens), ("seq_kv_lens", seq_kv_lens)):
        if lens is not None and (lens.dtype != torch.int32 or not lens.is_cuda or lens.numel() != B
                                 or not lens.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor of B elements")


def _check_lse(lse, B, Hq, Sq):
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous() \
            or lse.numel() != B * Hq * Sq:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor with B*Hq*Sq elements")


def _check_workspace(workspace) -> int:
    if workspace is None:
        return 0
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return workspace.numel() * workspace.element_size()


def _check_sink(sink, dsink, Hq):
    """Validates the fp32 (Hq,) sink logits; returns dsink (allocated when None)."""
    if sink.dtype != torch.float32 or not sink.is_cuda or not sink.is_contiguous() \
            or sink.numel() != Hq:
        raise ValueError("sink must be a contiguous fp32 CUDA tensor of Hq elements")
    dsink = torch.empty_like(sink) if dsink is None else dsink
    if dsink.dtype != torch.float32 or not dsink.is_cuda or not dsink.is_contiguous() \
            or dsink.numel() != Hq:
        raise ValueError("dsink must be a contiguous fp32 CUDA tensor of Hq elements")
    return dsink


def _check_same_device(ref: torch.Tensor, **tensors) -> None:
    """Every tensor argument lives on ref's device (the library takes raw pointers
    and launches on one device)."""
    for name, t in tensors.items():
        if t is not None and t.device != ref.device:
            raise ValueError(f"{name} is on {t.device} but q is on {ref.device}: "
                             "all tensors must be on one device")


def _check_launch_device(ref: torch.Tensor) -> None:
    """The library launches on the current CUDA device: it must be the tensors' one."""
    if ref.device.index != torch.cuda.current_device():
        raise ValueError(f"the tensors are on {ref.device} but the current device is "
                         f"cuda:{torch.cuda.current_device()}: call under torch.cuda.device({ref.device})")


# io element types of the C ABI (sdpa_dtype) for the typed entry points.
_IO_CODES = {torch.bfloat16: 0, torch.float16: 2}


def _io_dtype(q):
    if not isinstance(q, torch.Tensor) or q.dtype not in _IO_CODES:
        raise ValueError("q must be a bf16 or fp16 tensor")
    return q.dtype


def sdpa_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, do: torch.Tensor,
             lse: torch.Tensor, *, scale: Optional[float] = None, causal: bool = False,
             bottom_right: bool = False, window_left: int = -1, window_right: int = -1,
             deterministic: bool = False, seq_q_lens: Optional[torch.Tensor] = None,
             seq_kv_lens: Optional[torch.Tensor] = None, dq: Optional[torch.Tensor] = None,
             dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, sink: Optional[torch.Tensor] = None,
             dsink: Optional[torch.Tensor] = None, bias: Optional[torch.Tensor] = None,
             dbias: Optional[torch.Tensor] = None, bias_grad: bool = True,
             dbias_dtype: torch.dtype = torch.float32,
             stream: Optional[torch.cuda.Stream] = None):
    """dQ, dK, dV of scaled-dot-product attention (see include/sdpa_bwd.h).

    q (B,Hq,Sq,Dqk), k (B,Hkv,Skv,Dqk), v (B,Hkv,Skv,Dv), o/do (B,Hq,Sq,Dv): bf16 or fp16
    (one type for all) CUDA tensors on the current device, contiguous. lse (B,Hq,Sq) fp32 natural-log forward statistic. Lengths: int32 (B,) CUDA.
    Outputs are allocated when not given. Runs on ``stream`` (default: current stream).
    With ``sink`` (fp32 (Hq,) CUDA sink logits, already folded into ``lse`` by the
    forward) the call goes through sdpa_bwd_sink and returns (dq, dk, dv, dsink).
    With ``bias`` ((1|B, Hq, Sq, Skv) bf16, fp16 or fp32 CUDA, contiguous: the additive
    bias that ``lse`` was computed with) the call goes through sdpa_bwd_bias and,
    unless ``bias_grad`` is False, appends the fp32 dBias (shaped like ``bias``) to
    the returned tuple (``dbias_dtype`` float32, or bfloat16 / float16 for the
    io-type dBias of the general entry point).
    """
    lib = load()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be (B, H, S, D)")
    io = _io_dtype(q)
    B, Hq, Sq, Dqk = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    _check_bf16("q", q, (B, Hq, Sq, Dqk), io)
    _check_bf16("k", k, (B, Hkv, Skv, Dqk), io)
    _check_bf16("v", v, (B, Hkv, Skv, Dv), io)
    _check_bf16("o", o, (B, Hq, Sq, Dv), io)
    _check_bf16("do", do, (B, Hq, Sq, Dv), io)
    _check_lse(lse, B, Hq, Sq)
    _check_lens(B, seq_q_lens, seq_kv_lens)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_bf16("dq", dq, q.shape, io)
    _check_bf16("dk", dk, k.shape, io)
    _check_bf16("dv", dv, v.shape, io)
    ws_bytes = _check_workspace(workspace)
    if sink is not None:
        dsink = _check_sink(sink, dsink, Hq)
    _check_same_device(q, k=k, v=v, o=o, do=do, lse=lse, seq_q_lens=seq_q_lens,
                       seq_kv_lens=seq_kv_lens, dq=dq, dk=dk, dv=dv, workspace=workspace,
                       sink=sink, dsink=dsink if sink is not None else None, bias=bias,
                       dbias=dbias if bias is not None and bias_grad else None)
    _check_launch_device(q)
    sc = 0.0 if scale is None else float(scale)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
            _ptr(dv), B, Hq, Hkv, Sq, Skv, Dqk, Dv, sc, int(causal), int(bottom_right),
            int(window_left), int(window_right), int(deterministic), _ptr(seq_q_lens),
            _ptr(seq_kv_lens), _ptr(workspace), ws_bytes)
    if io == torch.float16 or (bias is not None and bias_grad and dbias_dtype != torch.float32):
        # the general typed entry: fp16 io, or an io-type dBias (sink and bias optional)
        bias_dtype, bias_batch = 0, 0
        if bias is not None:
            bias_dtype = _check_bias(bias, B, Hq, Sq, Skv)
            bias_batch = int(bias.shape[0])
            if bias_grad:
                if dbias_dtype not in (torch.float32, torch.bfloat16, torch.float16):
                    raise ValueError("dbias_dtype must be float32, bfloat16 or float16")
                dbias = torch.empty(bias.shape, dtype=dbias_dtype, device=bias.device) \
                    if dbias is None else dbias
                if dbias.dtype != dbias_dtype or not dbias.is_cuda or not dbias.is_contiguous() \
                        or tuple(dbias.shape) != tuple(bias.shape):
                    raise ValueError("dbias must be a contiguous CUDA tensor shaped like bias, of dbias_dtype")
            else:
                dbias = None
        else:
            dbias = None
        dbias_code = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16,
                      torch.float16: DTYPE_F16}[dbias.dtype] if dbias is not None else DTYPE_F32
        rc = lib.sdpa_bwd_typed(_IO_CODES[io], *args, _ptr(sink), _ptr(dsink if sink is not None else None),
                                _ptr(bias), bias_dtype, bias_batch, _ptr(dbias), dbias_code,
                                _stream_handle(stream))
        if rc != 0:
            raise SdpaError(rc, "sdpa_bwd_typed")
        out = (dq, dk, dv) + ((dsink,) if sink is not None else ())
        return out + ((dbias,) if bias is not None and bias_grad else ())
    if sink is None and bias is None:
        rc = lib.sdpa_bwd(*args, _stream_handle(stream))
        if rc != 0:
            raise SdpaError(rc, "sdpa_bwd")
        return dq, dk, dv
    if bias is None:
        rc = lib.sdpa_bwd_sink(*args, _ptr(sink), _ptr(dsink), _stream_handle(stream))
        if rc != 0:
            raise SdpaError(rc, "sdpa_bwd_sink")
        return dq, dk, dv, dsink
    bias_dtype = _check_bias(bias, B, Hq, Sq, Skv)
    if bias_grad:
        dbias = torch.empty(bias.shape, dtype=torch.float32, device=bias.device) if dbias is None else dbias
        if dbias.dtype != torch.float32 or not dbias.is_cuda or not dbias.is_contiguous() \
                or tuple(dbias.shape) != tuple(bias.shape):
            raise ValueError("dbias must be a contiguous fp32 CUDA tensor shaped like bias")
    else:
        dbias = None
    rc = lib.sdpa_bwd_bias(*args, _ptr(sink), _ptr(dsink if sink is not None else None), _ptr(bias),
                           bias_dtype, int(bias.shape[0]), _ptr(dbias), _stream_handle(stream))
    if rc != 0:
        raise SdpaError(rc, "sdpa_bwd_bias")
    out = (dq, dk, dv) + ((dsink,) if sink is not None else ())
    return out + ((dbias,) if bias_grad else ())


# Element-type codes of the C ABI (sdpa_dtype).
DTYPE_BF16, DTYPE_F32, DTYPE_F16 = 0, 1, 2


def _check_bias(bias, B, Hq, Sq, Skv) -> int:
    if not isinstance(bias, torch.Tensor) or not bias.is_cuda or not bias.is_contiguous():
        raise ValueError("bias must be a contiguous CUDA tensor")
    if bias.dtype not in (torch.bfloat16, torch.float16, torch.float32):
        raise ValueError("bias must be bf16, fp16 or fp32")
    if bias.dim() != 4 or bias.shape[0] not in (1, B) or tuple(bias.shape[1:]) != (Hq, Sq, Skv):
        raise ValueError(f"bias must be (1|B, Hq, Sq, Skv), got {tuple(bias.shape)}")
    return {torch.float32: DTYPE_F32, torch.float16: DTYPE_F16}.get(bias.dtype, DTYPE_BF16)


def sdpa_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: Optional[float] = None,
             causal: bool = False, bottom_right: bool = False, window_left: int = -1,
             window_right: int = -1, seq_q_lens: Optional[torch.Tensor] = None,
             seq_kv_lens: Optional[torch.Tensor] = None, sink: Optional[torch.Tensor] = None,
             bias: Optional[torch.Tensor] = None,
             o: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
             stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O (bf16, (B,Hq,Sq,Dv)) and natural-log LSE (fp32, (B,Hq,Sq)) of the masked
    softmax attention (see include/sdpa_bwd.h); the inputs of sdpa_bwd. ``bias``
    ((1|B, Hq, Sq, Skv) bf16, fp16 or fp32 CUDA, contiguous) is added to the scaled
    scores (sdpa_fwd_bias)."""
    lib = load()
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be (B, H, S, D)")
    io = _io_dtype(q)
    B, Hq, Sq, Dqk = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    Dv = v.shape[3]
    _check_bf16("q", q, (B, Hq, Sq, Dqk), io)
    _check_bf16("k", k, (B, Hkv, Skv, Dqk), io)
    _check_bf16("v", v, (B, Hkv, Skv, Dv), io)
    _check_lens(B, seq_q_lens, seq_kv_lens)
    if sink is not None and (sink.dtype != torch.float32 or not sink.is_cuda
                             or not sink.is_contiguous() or sink.numel() != Hq):
        raise ValueError("sink must be a contiguous fp32 CUDA tensor of Hq elements")
    o = torch.empty((B, Hq, Sq, Dv), dtype=io, device=q.device) if o is None else o
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_bf16("o", o, (B, Hq, Sq, Dv), io)
    _check_lse(lse, B, Hq, Sq)
    _check_same_device(q, k=k, v=v, o=o, lse=lse, seq_q_lens=seq_q_lens, seq_kv_lens=seq_kv_lens,
                       sink=sink, bias=bias)
    _check_launch_device(q)
    sc = 0.0 if scale is None else float(scale)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, Dqk, Dv, sc,
            int(causal), int(bottom_right), int(window_left), int(window_right),
            _ptr(seq_q_lens), _ptr(seq_kv_lens), _ptr(sink))
    if io == torch.float16:
        bias_dtype = _check_bias(bias, B, Hq, Sq, Skv) if bias is not None else 0
        rc = lib.sdpa_fwd_typed(_IO_CODES[io], *args, _ptr(bias), bias_dtype,
                                0 if bias is None else int(bias.shape[0]), _stream_handle(stream))
    elif bias is None:
        rc = lib.sdpa_fwd(*args, _stream_handle(stream))
    else:
        dt = _check_bias(bias, B, Hq, Sq, Skv)
        rc = lib.sdpa_fwd_bias(*args, _ptr(bias), dt, int(bias.shape[0]), _stream_handle(stream))
    if rc != 0:
        raise SdpaError(rc, "sdpa_fwd_bias" if bias is not None else "sdpa_fwd")
    return o, lse


def nvfp4_fake_quant(x: torch.Tensor, out: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """NVFP4 fake quantization of a contiguous bf16 CUDA tensor in blocks of 16
    consecutive values (sdpa_nvfp4_fake_quant); numel must be a multiple of 16."""
    lib = load()
    if not isinstance(x, torch.Tensor) or x.dtype != torch.bfloat16 or not x.is_cuda \
            or not x.is_contiguous():
        raise ValueError("x must be a contiguous bf16 CUDA tensor")
    out = torch.empty_like(x) if out is None else out
    _check_bf16("out", out, x.shape)
    _check_same_device(x, out=out)
    _check_launch_device(x)
    rc = lib.sdpa_nvfp4_fake_quant(_ptr(x), _ptr(out), x.numel(), _stream_handle(stream))
    if rc != 0:
        raise SdpaError(rc, "sdpa_nvfp4_fake_quant")
    return out


def sdpa_fwd_nvfp4_qat(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, **kw):
    """The QAT forward statistics the QAT backward takes: sdpa_fwd() of the
    fake-quantized q, k, v, i.e. (O_hp, LSE) with O_hp = softmax(scale q^ k^^T) v^."""
    stream = kw.get("stream")
    return sdpa_fwd(nvfp4_fake_quant(q, stream=stream), nvfp4_fake_quant(k, stream=stream),
                    nvfp4_fake_quant(v, stream=stream), **kw)


def sdpa_bwd_nvfp4_qat(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o_hp: torch.Tensor,
                       do: torch.Tensor, lse: torch.Tensor, *, scale: Optional[float] = None,
                       causal: bool = False, bottom_right: bool = False, window_left: int = -1,
                       window_right: int = -1, seq_q_lens: Optional[torch.Tensor] = None,
                       seq_kv_lens: Optional[torch.Tensor] = None, dq: Optional[torch.Tensor] = None,
                       dk: Optional[torch.Tensor] = None, dv: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None):
    """dQ, dK, dV of NVFP4 QAT attention (sdpa_bwd_nvfp4_qat): q, k, v unquantized,
    o_hp / lse from sdpa_fwd_nvfp4_qat. D = 128."""
    lib = load()
    if not isinstance(q, torch.Tensor) or q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be (B, H, S, D) tensors")
    B, Hq, Sq, Dqk = q.shape
    Hkv, Skv, Dv = k.shape[1], k.shape[2], v.shape[3]
    for name, t, shape in (("q", q, (B, Hq, Sq, Dqk)), ("k", k, (B, Hkv, Skv, Dqk)),
                           ("v", v, (B, Hkv, Skv, Dv)), ("o_hp", o_hp, (B, Hq, Sq, Dv)),
                           ("do", do, (B, Hq, Sq, Dv))):
        _check_bf16(name, t, shape)
    _check_lse(lse, B, Hq, Sq)
    _check_lens(B, seq_q_lens, seq_kv_lens)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check_bf16("dq", dq, q.shape)
    _check_bf16("dk", dk, k.shape)
    _check_bf16("dv", dv, v.shape)
    ws_bytes = _check_workspace(workspace)
    _check_same_device(q, k=k, v=v, o_hp=o_hp, do=do, lse=lse, seq_q_lens=seq_q_lens,
                       seq_kv_lens=seq_kv_lens, dq=dq, dk=dk, dv=dv, workspace=workspace)
    _check_launch_device(q)
    rc = lib.sdpa_bwd_nvfp4_qat(_ptr(q), _ptr(k), _ptr(v), _ptr(o_hp), _ptr(do), _ptr(lse), _ptr(dq),
                                _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, Dqk, Dv,
                                0.0 if scale is None else float(scale), int(causal),
                                int(bottom_right), int(window_left), int(window_right),
                                _ptr(seq_q_lens), _ptr(seq_kv_lens), _ptr(workspace), ws_bytes,
                                _stream_handle(stream))
    if rc != 0:
        raise SdpaError(rc, "sdpa_bwd_nvfp4_qat")
    return dq, dk, dv


def nvfp4_qat_workspace_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv) -> int:
    return int(load().sdpa_bwd_nvfp4_qat_workspace_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv))


def debug_relay(wait_limit_ns: int = 0, turn_skew: int = 0) -> None:
    """Sets the ordered relay's wait limit (0: the 4 s default) and turn skew (0:
    normal use) for later calls; see sdpa_bwd_debug_relay in the header."""
    load().sdpa_bwd_debug_relay(int(wait_limit_ns), int(turn_skew))


def check_device_status(stream: Optional[torch.cuda.Stream] = None) -> None:
    """Synchronizes the stream and raises if a kernel reported a timed-out wait."""
    rc = load().sdpa_bwd_check_device_status(_stream_handle(stream))
    if rc != 0:
        raise SdpaError(rc, "device status")


def profile_enable(on: bool = True) -> None:
    load().sdpa_bwd_profile_enable(int(on))


def profile_read():
    """{kernel name: (total ms, launches)} accumulated since profile_enable()."""
    ms = (ctypes.c_float * len(KERNEL_NAMES))()
    n = (ctypes.c_int * len(KERNEL_NAMES))()
    load().sdpa_bwd_profile_read(ms, n, len(KERNEL_NAMES))
    return {name: (float(ms[i]), int(n[i])) for i, name in enumerate(KERNEL_NAMES)}
