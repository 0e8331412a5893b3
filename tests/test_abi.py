"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, sizes its workspace as documented, and rejects bad arguments
with the documented status codes before launching anything."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa_bwd.h")

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE, CUDA, TIMEOUT = range(7)


@pytest.fixture(scope="module")
def lib():
    import attention_backward_sdpa_gb300 as pkg
    return pkg.load(build_if_missing=True)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(sdpa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for expected in ("sdpa_bwd", "sdpa_bwd_workspace_size", "sdpa_status_string",
                     "sdpa_bwd_check_device_status", "sdpa_bwd_profile_enable",
                     "sdpa_bwd_profile_read", "sdpa_bwd_version"):
        assert expected in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in sdpa_bwd.h but not exported"


def test_version_and_status_strings(lib):
    assert lib.sdpa_bwd_version() == 200
    assert lib.sdpa_status_string(OK) == b"ok"
    for code in range(1, 8):
        assert lib.sdpa_status_string(code) not in (b"ok", b"unknown status")
    assert lib.sdpa_status_string(99) == b"unknown status"


def _a256(x):
    return (x + 255) // 256 * 256


def visited_query_tiles(kt, Lq, Lk, causal, br, wl, wr):
    """64-row query tiles that 128-key tile kt visits (the kernels' loop bounds),
    restated from the mask definitions: keys k <= q + diag + max(wr, 0) when causal,
    k >= q + diag - wl with a left window, diag = Lk - Lq when bottom-right."""
    k0 = kt * 128
    if k0 >= Lk or Lq <= 0:
        return 0, -1
    diag = Lk - Lq if br else 0
    k_last = min(k0 + 127, Lk - 1)
    q_min, q_max = 0, Lq - 1
    if causal:
        q_min = max(0, k0 - diag - max(wr, 0))
    if wl >= 0:
        q_max = min(q_max, k_last - diag + wl)
    if q_min > q_max:
        return 0, -1
    return q_min // 64, q_max // 64


def band_tiles(Sq, Skv, causal, br, wl, wr, padded):
    """dS tiles stored per (batch, query head): the query tiles each key tile visits at
    the full lengths, or every query tile when a bottom-right mask meets per-batch lengths."""
    n_qt, n_kt = -(-Sq // 64), -(-Skv // 128)
    if br and padded:
        return n_kt * n_qt
    tot = 0
    for kt in range(n_kt):
        lo, hi = visited_query_tiles(kt, Sq, Skv, causal, br, wl, wr if causal else -1)
        tot += max(0, hi - lo + 1)
    return tot


def route(det, Dqk):
    return "two" if Dqk > 128 or (det and Dqk == 128) else "reduce"


def carve_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv, rt, causal=0, br=0, wl=-1, wr=-1, padded=0):
    """Documented layout: per-query-tile row statistics (2 x 64 fp32 per 64-row tile);
    then either the fp32 dQ accumulator over whole 64-row tiles (rows of max(D_qk, 64)
    columns) or, on the routes that store dS, one 16 KiB dS^T tile per (128-key tile,
    64-query tile of its band) plus one zero tile; one int per query tile plus a ticket;
    one fp32 sink-token partial per query tile; and for GQA on the routes that split a
    group, the bf16 dK/dV partials with H_q heads. Every region 256-byte aligned."""
    n_qt = -(-Sq // 64)
    total = _a256(B * Hq * n_qt * 128 * 4)
    if rt != "reduce":
        total += _a256(B * Hq * band_tiles(Sq, Skv, causal, br, wl, wr, padded) * 16384) + _a256(16384)
    else:
        total += _a256(B * Hq * n_qt * 64 * (64 if Dqk <= 64 else 128) * 4)
    total += _a256((B * Hq * n_qt + 1) * 4)
    total += _a256(B * Hq * n_qt * 4)
    if Hkv < Hq:
        total += _a256(B * Hq * Skv * Dqk * 2) + _a256(B * Hq * Skv * Dv * 2)
    return total


def expected_workspace(B, Hq, Hkv, Sq, Skv, Dqk, Dv, det=0, causal=0, br=0, wl=-1, wr=-1, padded=0):
    return carve_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv, route(det, Dqk), causal=causal, br=br, wl=wl,
                      wr=wr, padded=padded)


def ws(lib, B, Hq, Hkv, Sq, Skv, Dqk, Dv, det=0, causal=0, br=0, wl=-1, wr=-1, padded=0):
    return lib.sdpa_bwd_workspace_size(B, Hq, Hkv, Sq, Skv, Dqk, Dv, causal, br, wl, wr, det, padded)


SHAPES = [(1, 2, 2, 128, 128, 64, 64), (2, 16, 16, 2048, 2048, 128, 128),
          (1, 32, 8, 4096, 4096, 128, 128), (3, 4, 1, 300, 177, 128, 128),
          (1, 1, 1, 1, 1, 64, 64), (1, 16, 16, 4096, 4096, 192, 128),
          (2, 4, 2, 300, 177, 192, 128), (2, 4, 2, 300, 177, 32, 32),
          (2, 4, 2, 300, 177, 256, 256), (1, 8, 8, 4096, 4096, 256, 256),
          (1, 3, 1, 200, 130, 96, 96), (2, 2, 2, 65, 70, 8, 8)]
MASKS = [dict(), dict(causal=1), dict(causal=1, br=1), dict(causal=1, wl=1024),
         dict(causal=1, wr=100, wl=50), dict(wl=70), dict(causal=1, padded=1),
         dict(causal=1, br=1, padded=1)]


@pytest.mark.parametrize("shape", SHAPES)
def test_workspace_size_matches_layout(lib, shape):
    for det in (0, 1):
        for m in MASKS:
            assert ws(lib, *shape, det=det, **m) == expected_workspace(*shape, det=det, **m), (det, m)


def test_workspace_band_halves_causal_and_shrinks_windows(lib):
    # causal: about half of the rectangle of dS tiles; a 1024-key window far less
    full = ws(lib, 1, 32, 32, 4096, 4096, 128, 128, det=1)
    causal = ws(lib, 1, 32, 32, 4096, 4096, 128, 128, det=1, causal=1)
    assert 0.5 < causal / full < 0.53
    assert ws(lib, 4, 16, 16, 4096, 4096, 128, 128, det=1, causal=1, wl=1024, padded=1) < \
        0.3 * ws(lib, 4, 16, 16, 4096, 4096, 128, 128, det=1, padded=1)
    # a bottom-right mask with per-batch lengths keeps the whole rectangle
    assert ws(lib, 1, 2, 2, 512, 512, 128, 128, det=1, causal=1, br=1, padded=1) == \
        ws(lib, 1, 2, 2, 512, 512, 128, 128, det=1)


def test_band_model_against_brute_force():
    """The band restated above against a brute-force scan of (query, key) pairs."""
    for (Sq, Skv, causal, br, wl, wr) in [(300, 177, 1, 0, -1, -1), (177, 300, 1, 1, -1, -1),
                                           (500, 500, 1, 0, 100, -1), (260, 380, 1, 1, 90, 30),
                                           (200, 200, 0, 0, 33, -1)]:
        diag = Skv - Sq if br else 0
        for kt in range(-(-Skv // 128)):
            tiles = set()
            for q in range(Sq):
                for k in range(kt * 128, min(kt * 128 + 128, Skv)):
                    ok = (not causal or k <= q + diag + max(wr, 0)) and (wl < 0 or k >= q + diag - wl)
                    if ok:
                        tiles.add(q // 64)
            lo, hi = visited_query_tiles(kt, Sq, Skv, causal, br, wl, wr)
            if tiles:
                assert (lo, hi) == (min(tiles), max(tiles))
            else:
                assert hi < lo


def test_band_contains_every_shorter_batch_row():
    """With per-batch lengths and a top-left mask (or no lengths at all) the stored band,
    taken at the full lengths, contains the query tiles that each key tile visits for
    any shorter batch row: the kernels index a stored tile by its offset inside the band."""
    rng = np.random.default_rng(7)
    for _ in range(60):
        Sq, Skv = int(rng.integers(1, 700)), int(rng.integers(1, 700))
        causal = int(rng.integers(0, 2))
        wl = int(rng.integers(0, 300)) if rng.random() < 0.5 else -1
        wr = int(rng.integers(0, 100)) if causal and rng.random() < 0.3 else -1
        for kt in range(-(-Skv // 128)):
            lo, hi = visited_query_tiles(kt, Sq, Skv, causal, 0, wl, wr)
            for _ in range(8):
                Lq, Lk = int(rng.integers(0, Sq + 1)), int(rng.integers(0, Skv + 1))
                a, b = visited_query_tiles(kt, Lq, Lk, causal, 0, wl, wr)
                if a <= b:
                    assert lo <= a and b <= hi, (Sq, Skv, causal, wl, wr, kt, Lq, Lk)
    # A bottom-right mask moves the visited range with the lengths, so the host stores
    # the whole rectangle there: shorter rows leave the full-length band.
    outside = 0
    for kt in range(4):
        lo, hi = visited_query_tiles(kt, 512, 512, 1, 1, -1, -1)
        a, b = visited_query_tiles(kt, 200, 512, 1, 1, -1, -1)
        outside += a <= b and not (lo <= a and b <= hi)
    assert outside > 0


def test_workspace_size_rejects(lib):
    assert ws(lib, 1, 3, 2, 128, 128, 128, 128) == 0  # Hkv does not divide
    assert ws(lib, 1, 2, 2, 128, 128, 100, 100) == 0  # head dim not served
    assert ws(lib, 0, 2, 2, 128, 128, 128, 128) == 0
    assert ws(lib, 1, 2, 2, 0, 128, 128, 128) == 0    # nothing to stage


FAKE = 0x10000  # never dereferenced: every call below fails validation first


def call(lib, ptrs=None, B=1, Hq=2, Hkv=2, Sq=128, Skv=128, Dqk=128, Dv=128, scale=0.0, causal=0,
         br=0, wl=-1, wr=-1, det=0, ws=None, ws_bytes=0):
    ptrs = ptrs or [FAKE] * 9
    vp = [ctypes.c_void_p(p) if p is not None else None for p in ptrs]
    return lib.sdpa_bwd(*vp, B, Hq, Hkv, Sq, Skv, Dqk, Dv, ctypes.c_float(scale), causal, br, wl,
                        wr, det, None, None, ws, ws_bytes, None)


def test_argument_validation(lib):
    assert call(lib, Hq=3, Hkv=2) == INVALID
    assert call(lib, B=0) == INVALID
    assert call(lib, Sq=-1) == INVALID
    assert call(lib, Dqk=100, Dv=100) == UNSUPPORTED   # not a multiple of 8
    assert call(lib, Dqk=136, Dv=136) == UNSUPPORTED   # past 128 (other than 192/128)
    assert call(lib, Dqk=128, Dv=64) == UNSUPPORTED
    assert call(lib, Dqk=32, Dv=64) == UNSUPPORTED
    assert call(lib, Dqk=256, Dv=128) == UNSUPPORTED
    assert call(lib, Dqk=192, Dv=192) == UNSUPPORTED
    assert call(lib, Dqk=264, Dv=264) == UNSUPPORTED
    # 256/256 is served: these pointer checks fail only after the head dims pass
    assert call(lib, Dqk=256, Dv=256, ptrs=[FAKE] * 8 + [None]) == INVALID
    for i in range(9):
        ptrs = [FAKE] * 9
        ptrs[i] = None
        assert call(lib, ptrs) == INVALID
    for i in (0, 1, 2, 3, 4, 6, 7, 8):  # bf16 tensors need 16-byte alignment
        ptrs = [FAKE] * 9
        ptrs[i] = FAKE + 8
        assert call(lib, ptrs) == ALIGN
    ptrs = [FAKE] * 9
    ptrs[5] = FAKE + 2  # lse needs 4-byte alignment
    assert call(lib, ptrs) == ALIGN
    assert call(lib, wr=3, causal=0) == UNSUPPORTED  # a right band only widens a causal mask


def call_sink(lib, sink, dsink, ptrs=None):
    ptrs = ptrs or [FAKE] * 9
    vp = [ctypes.c_void_p(p) for p in ptrs]
    return lib.sdpa_bwd_sink(*vp, 1, 2, 2, 128, 128, 128, 128, ctypes.c_float(0.0), 0, 0, -1, -1, 0,
                             None, None, None, 0,
                             None if sink is None else ctypes.c_void_p(sink),
                             None if dsink is None else ctypes.c_void_p(dsink), None)


def test_sink_argument_validation(lib):
    lib.sdpa_bwd_sink.restype = ctypes.c_int
    assert call_sink(lib, None, FAKE) == INVALID
    assert call_sink(lib, FAKE, None) == INVALID
    assert call_sink(lib, FAKE + 2, FAKE) == ALIGN  # fp32 vectors need 4-byte alignment
    assert call_sink(lib, FAKE, FAKE + 1) == ALIGN
    ptrs = [FAKE] * 9
    ptrs[0] = FAKE + 8
    assert call_sink(lib, FAKE, FAKE, ptrs) == ALIGN


def test_python_binding_rejects_cpu_tensors():
    import torch
    import attention_backward_sdpa_gb300 as pkg
    x = torch.zeros(1, 2, 128, 128, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 128)
    with pytest.raises(ValueError):
        pkg.sdpa_bwd(x, x, x, x, x, lse)


def test_python_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    """No fallback: with the shared library absent, loading raises instead of
    routing anywhere else."""
    import attention_backward_sdpa_gb300 as pkg
    monkeypatch.setattr(pkg, "_lib", None)
    monkeypatch.setattr(pkg._build, "LIB", str(tmp_path / "libsdpa_bwd.so"))
    with pytest.raises(RuntimeError, match="missing"):
        pkg.load()


def test_python_binding_checks_one_device():
    """Tensors on different devices are refused before any pointer is passed."""
    import torch
    import attention_backward_sdpa_gb300 as pkg
    a = torch.zeros(4)
    pkg._check_same_device(a, b=torch.zeros(4), c=None)
    with pytest.raises(ValueError, match="one device"):
        pkg._check_same_device(a, b=torch.zeros(4, device="meta"))


def test_python_binding_rejects_cpu_inputs_everywhere():
    import torch
    import attention_backward_sdpa_gb300 as pkg
    x = torch.zeros(1, 2, 128, 128, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 128)
    with pytest.raises(ValueError):
        pkg.sdpa_bwd_nvfp4_qat(x, x, x, x, x, lse)
    with pytest.raises(ValueError):
        pkg.sdpa_fwd(x, x, x)
    with pytest.raises(ValueError):
        pkg.nvfp4_fake_quant(x)
    with pytest.raises(ValueError):
        pkg._check_sink(torch.zeros(2), None, 2)


def test_public_names_exist():
    import attention_backward_sdpa_gb300 as pkg
    assert [n for n in pkg.__all__ if not hasattr(pkg, n)] == []


def call_fwd(lib, ptrs=None, B=1, Hq=2, Hkv=2, Sq=128, Skv=128, Dqk=128, Dv=128, causal=0, wr=-1,
             sink=None):
    ptrs = ptrs or [FAKE] * 5
    vp = [ctypes.c_void_p(p) if p is not None else None for p in ptrs]
    return lib.sdpa_fwd(*vp, B, Hq, Hkv, Sq, Skv, Dqk, Dv, ctypes.c_float(0.0), causal, 0, -1, wr,
                        None, None, None if sink is None else ctypes.c_void_p(sink), None)


def test_forward_argument_validation(lib):
    lib.sdpa_fwd.restype = ctypes.c_int
    assert call_fwd(lib, Hq=3, Hkv=2) == INVALID
    assert call_fwd(lib, B=0) == INVALID
    assert call_fwd(lib, Dqk=100, Dv=100) == UNSUPPORTED
    assert call_fwd(lib, Dqk=192, Dv=192) == UNSUPPORTED
    assert call_fwd(lib, Dqk=256, Dv=128) == UNSUPPORTED
    # 256/256 is served: the null LSE pointer fails only after the head dims pass
    assert call_fwd(lib, Dqk=256, Dv=256, ptrs=[FAKE] * 4 + [None]) == INVALID
    for i in range(5):
        ptrs = [FAKE] * 5
        ptrs[i] = None
        assert call_fwd(lib, ptrs) == INVALID
    for i in range(4):  # q, k, v, o: 16-byte alignment
        ptrs = [FAKE] * 5
        ptrs[i] = FAKE + 8
        assert call_fwd(lib, ptrs) == ALIGN
    ptrs = [FAKE] * 5
    ptrs[4] = FAKE + 2  # lse: 4-byte alignment
    assert call_fwd(lib, ptrs) == ALIGN
    assert call_fwd(lib, sink=FAKE + 1) == ALIGN
    assert call_fwd(lib, wr=3, causal=0) == UNSUPPORTED


def call_bias(lib, bias, dtype=0, batch=1, dbias=FAKE, B=1, det=0, Dqk=128, Dv=128, sink=None,
              dsink=None):
    vp = [ctypes.c_void_p(FAKE)] * 9
    return lib.sdpa_bwd_bias(*vp, B, 2, 2, 128, 128, Dqk, Dv, ctypes.c_float(0.0), 0, 0, -1, -1, det,
                             None, None, None, 0,
                             None if sink is None else ctypes.c_void_p(sink),
                             None if dsink is None else ctypes.c_void_p(dsink),
                             None if bias is None else ctypes.c_void_p(bias), dtype, batch,
                             None if dbias is None else ctypes.c_void_p(dbias), None)


def test_bias_argument_validation(lib):
    lib.sdpa_bwd_bias.restype = ctypes.c_int
    assert call_bias(lib, None) == INVALID
    assert call_bias(lib, FAKE, dtype=3) == INVALID          # unknown element type
    assert call_bias(lib, FAKE, batch=3, B=2) == INVALID     # bias batch is 1 or B
    assert call_bias(lib, FAKE, batch=0) == INVALID
    # a one-batch dBias summed over B > 1 batch rows is atomic: not in deterministic mode
    assert call_bias(lib, FAKE, batch=1, B=2, det=1) == INVALID
    assert call_bias(lib, FAKE, dsink=FAKE) == INVALID        # dsink needs the sink logits
    assert call_bias(lib, FAKE + 1, dtype=0) == ALIGN         # bf16 bias: 2-byte alignment
    assert call_bias(lib, FAKE + 2, dtype=1) == ALIGN         # fp32 bias: 4-byte alignment
    assert call_bias(lib, FAKE, dbias=FAKE + 2) == ALIGN      # fp32 dBias: 4-byte alignment
    assert call_bias(lib, FAKE, Dqk=100, Dv=100) == UNSUPPORTED


def test_forward_bias_argument_validation(lib):
    lib.sdpa_fwd_bias.restype = ctypes.c_int
    vp = [ctypes.c_void_p(FAKE)] * 5

    def call(bias, dtype=0, batch=1, B=1):
        return lib.sdpa_fwd_bias(*vp, B, 2, 2, 128, 128, 128, 128, ctypes.c_float(0.0), 0, 0, -1, -1,
                                 None, None, None, None if bias is None else ctypes.c_void_p(bias),
                                 dtype, batch, None)
    assert call(None) == INVALID
    assert call(FAKE, dtype=5) == INVALID
    assert call(FAKE, batch=2, B=3) == INVALID
    assert call(FAKE + 1, dtype=0) == ALIGN
    assert call(FAKE + 2, dtype=1) == ALIGN


def test_nvfp4_qat_argument_validation(lib):
    lib.sdpa_bwd_nvfp4_qat.restype = ctypes.c_int
    lib.sdpa_nvfp4_fake_quant.restype = ctypes.c_int
    lib.sdpa_bwd_nvfp4_qat_workspace_size.restype = ctypes.c_size_t
    vp = [ctypes.c_void_p(FAKE)] * 9

    def call(Dqk=128, Dv=128, Hq=2, Hkv=2):
        return lib.sdpa_bwd_nvfp4_qat(*vp, 1, Hq, Hkv, 128, 128, Dqk, Dv, ctypes.c_float(0.0), 1, 0,
                                      -1, -1, None, None, None, ctypes.c_size_t(0), None)
    assert call(Dqk=64, Dv=64) == UNSUPPORTED       # D = 128 only
    assert call(Dqk=192, Dv=128) == UNSUPPORTED
    assert call(Hq=3, Hkv=2) == INVALID
    fq = lib.sdpa_nvfp4_fake_quant
    assert fq(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_longlong(17), None) == INVALID
    assert fq(None, ctypes.c_void_p(FAKE), ctypes.c_longlong(16), None) == INVALID
    assert fq(ctypes.c_void_p(FAKE + 8), ctypes.c_void_p(FAKE), ctypes.c_longlong(16), None) == ALIGN
    assert fq(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), ctypes.c_longlong(0), None) == OK
    # workspace: the plain chain's regions plus bf16 copies of Q, K and V
    qws = lib.sdpa_bwd_nvfp4_qat_workspace_size(1, 2, 2, 128, 128, 128, 128)
    base = ws(lib, 1, 2, 2, 128, 128, 128, 128)
    assert qws == base + 3 * 2 * 128 * 128 * 2
    assert lib.sdpa_bwd_nvfp4_qat_workspace_size(1, 2, 2, 128, 128, 64, 64) == 0


def test_typed_entry_validation(lib):
    lib.sdpa_bwd_typed.restype = ctypes.c_int
    lib.sdpa_fwd_typed.restype = ctypes.c_int
    vp = [ctypes.c_void_p(FAKE)] * 9

    def bwd(io, sink=None, dsink=None, bias=None, bias_dtype=0, dbias=None, dbias_dtype=1):
        return lib.sdpa_bwd_typed(io, *vp, 1, 2, 2, 128, 128, 128, 128, ctypes.c_float(0.0), 0, 0, -1,
                                  -1, 0, None, None, None, ctypes.c_size_t(0),
                                  None if sink is None else ctypes.c_void_p(sink),
                                  None if dsink is None else ctypes.c_void_p(dsink),
                                  None if bias is None else ctypes.c_void_p(bias), bias_dtype, 1,
                                  None if dbias is None else ctypes.c_void_p(dbias), dbias_dtype, None)
    assert bwd(1) == INVALID          # fp32 io is not an io type
    assert bwd(7) == INVALID
    assert bwd(2, dsink=FAKE) == INVALID
    assert bwd(2, sink=FAKE + 1, dsink=FAKE) == ALIGN
    assert bwd(2, dbias=FAKE) == INVALID                     # dbias without a bias
    assert bwd(2, bias=FAKE, bias_dtype=5) == INVALID
    assert bwd(2, bias=FAKE + 1, bias_dtype=2) == ALIGN      # fp16 bias: 2-byte alignment
    assert bwd(2, bias=FAKE, dbias=FAKE, dbias_dtype=7) == INVALID
    assert bwd(2, bias=FAKE, dbias=FAKE + 2, dbias_dtype=1) == ALIGN   # fp32 dBias: 4-byte
    assert bwd(2, bias=FAKE, dbias=FAKE + 1, dbias_dtype=0) == ALIGN   # bf16 dBias: 2-byte
    fv = [ctypes.c_void_p(FAKE)] * 5
    assert lib.sdpa_fwd_typed(3, *fv, 1, 2, 2, 128, 128, 128, 128, ctypes.c_float(0.0), 0, 0, -1, -1,
                              None, None, None, None, 0, 0, None) == INVALID
