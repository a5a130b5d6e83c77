"""Host-side checks of the C ABI: the library builds, loads without a GPU, exports every
function include/fa.h declares, and rejects bad arguments before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_02_gb300.build import build
    path = build()
    import exact_attention_02_gb300 as fa
    assert os.path.samefile(path, fa.LIB_PATH)
    return fa.lib()


def _declared():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            names += re.findall(r"^FA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)
    return names


def test_header_declares_the_boundary():
    assert set(_declared()) >= {"fa_fwd", "fa_bwd_preprocess", "fa_bwd", "fa_bwd_workspace_size",
                                "fa_get_error_string", "fa_get_last_device_status", "fa_fwd_splitkv",
                                "fa_fwd_splitkv_workspace_size", "fa_fwd_fp8", "fa_fwd_masked", "fa_bwd_masked",
                                "fa_fwd_dropout", "fa_bwd_dropout", "fa_fwd_bitmask", "fa_bwd_bitmask"}


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_error_strings(lib):
    import exact_attention_02_gb300 as fa
    for code in range(6):
        assert fa.error_string(code).startswith("FA_")
    assert "unknown" in fa.error_string(99)


def test_workspace_size(lib):
    import exact_attention_02_gb300 as fa
    assert fa.fa_bwd_workspace_size(2, 16, 8192, 128, fa.FA_DTYPE_BF16) == 2 * 16 * 8192 * 128 * 4
    assert fa.fa_bwd_workspace_size(1, 1, 128, 64, fa.FA_DTYPE_FP32) == 0
    assert fa.fa_bwd_workspace_size(1, 1, 100, 64, fa.FA_DTYPE_BF16) == 100 * 64 * 4  # any N
    assert fa.fa_bwd_workspace_size(1, 1, 128, 96, fa.FA_DTYPE_BF16) == 0  # rejected head dim
    assert fa.fa_bwd_workspace_size(0, 1, 128, 64, fa.FA_DTYPE_BF16) == 0


P = 0x10000  # a 16-byte-aligned dummy address: never dereferenced, calls fail validation first
GOOD = dict(B=1, H=1, N=128, d=64, scale=0.125, causal=0, dtype=0)


def _fwd(lib, ptrs=(P, P, P, P, P), **kw):
    a = dict(GOOD, **kw)
    return lib.fa_fwd(*[ctypes.c_void_p(p) for p in ptrs], a["B"], a["H"], a["N"], a["d"],
                      ctypes.c_float(a["scale"]), a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(B=0), 1), (dict(H=-1), 1), (dict(N=0), 1), (dict(d=0), 1),
    (dict(d=96), 2), (dict(d=256), 2), (dict(d=32), 2),
    (dict(dtype=1, N=8192), 2), (dict(dtype=7), 1),
    (dict(scale=0.0), 1), (dict(scale=-1.0), 1), (dict(scale=float("nan")), 1),
    (dict(scale=float("inf")), 1), (dict(causal=2), 1),
    (dict(B=1 << 16, H=1 << 15), 1),
])
def test_fwd_rejects(lib, kw, code):
    assert _fwd(lib, **kw) == code


@pytest.mark.parametrize("ptrs", [(0, P, P, P, P), (P, P, P, P, 0), (P + 2, P, P, P, P),
                                  (P, P, P + 8, P, P)])
def test_fwd_rejects_pointers(lib, ptrs):
    assert _fwd(lib, ptrs=ptrs) == 1


def test_preprocess_rejects(lib):
    vp = ctypes.c_void_p
    assert lib.fa_bwd_preprocess(vp(0), vp(P), vp(P), 1, 1, 128, 64, 0, None) == 1
    assert lib.fa_bwd_preprocess(vp(P), vp(P), vp(P), 1, 1, 128, 80, 0, None) == 2


def _bwd(lib, D=P, ws=P, wsb=1 << 30, **kw):
    a = dict(GOOD, **kw)
    vp = ctypes.c_void_p
    return lib.fa_bwd(vp(P), vp(P), vp(P), vp(P), vp(P), vp(P), vp(D), vp(P), vp(P), vp(P), vp(ws),
                      ctypes.c_size_t(wsb), a["B"], a["H"], a["N"], a["d"], ctypes.c_float(a["scale"]),
                      a["causal"], a["dtype"], None)


def test_bwd_rejects(lib):
    assert _bwd(lib, d=96) == 2
    assert _bwd(lib, scale=0.0) == 1
    assert _bwd(lib, D=P + 4) == 1
    assert _bwd(lib, ws=0) == 5                          # bf16 needs the dQ accumulator
    assert _bwd(lib, wsb=128 * 64 * 4 - 16) == 5         # one row short
    assert _bwd(lib, D=0, wsb=128 * 64 * 4) == 5         # no room for D
    assert _bwd(lib, ws=P + 8) == 1


def test_binding_refuses_to_run_without_library(monkeypatch):
    import exact_attention_02_gb300 as fa
    monkeypatch.setattr(fa, "_lib", None)
    monkeypatch.setattr(fa, "LIB_PATH", os.path.join(ROOT, "does_not_exist.so"))
    with pytest.raises(RuntimeError, match="not built"):
        fa.lib()


def _splitkv(lib, ws=P, wsb=1 << 30, **kw):
    a = dict(B=1, H=2, Nq=1, Nk=1000, d=128, scale=0.088, causal=1, dtype=0)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.fa_fwd_splitkv(vp(P), vp(P), vp(P), vp(P), vp(P), a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                              ctypes.c_float(a["scale"]), a["causal"], a["dtype"], vp(ws), ctypes.c_size_t(wsb), None)


def test_splitkv_workspace_and_rejects(lib):
    import exact_attention_02_gb300 as fa
    n = fa.lib().fa_fwd_splitkv_workspace_size(1, 2, 1, 1000, 128, 0)
    assert n > 0 and n % 4 == 0
    assert fa.lib().fa_fwd_splitkv_workspace_size(1, 2, 65, 1000, 128, 0) == 0
    assert fa.lib().fa_fwd_splitkv_workspace_size(1, 2, 65, 1000, 64, 0) == 0
    assert fa.lib().fa_fwd_splitkv_workspace_size(1, 2, 64, 1000, 64, 0) > 0
    assert _splitkv(lib, Nq=65) == 2            # more queries than the split-KV path takes
    assert _splitkv(lib, Nq=65, d=64) == 2
    assert _splitkv(lib, d=96) == 2
    assert _splitkv(lib, dtype=1) == 2          # fp32 goes through fa_fwd
    assert _splitkv(lib, Nq=8, Nk=4) == 1       # causal needs N_q <= N_k
    assert _splitkv(lib, Nk=0) == 1
    assert _splitkv(lib, scale=-1.0) == 1
    assert _splitkv(lib, ws=0) == 5
    assert _splitkv(lib, wsb=16) == 5


def test_fp8_rejects_before_launch(lib):
    """Host-side checks of fa_fwd_fp8 (dummy pointers; nothing is launched)."""
    import exact_attention_02_gb300 as fa
    vp, f = ctypes.c_void_p, ctypes.c_float
    L = fa.lib()

    def call(B=1, H=1, N=128, d=128, scale=0.088, causal=0, qd=1.0, kd=1.0, vd=1.0, ptr=P):
        return L.fa_fwd_fp8(vp(ptr), vp(P), vp(P), vp(P), vp(P), B, H, N, d, f(scale), causal, f(qd), f(kd), f(vd),
                            None)
    assert call(d=64) == fa.FA_ERR_UNSUPPORTED        # e4m3 path is d = 128 only
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED
    assert call(qd=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(vd=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(kd=-1.0) == fa.FA_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FA_ERR_INVALID_ARG
    assert call(causal=2) == fa.FA_ERR_INVALID_ARG
    assert call(N=0) == fa.FA_ERR_INVALID_ARG
    assert call(ptr=P + 8) == fa.FA_ERR_INVALID_ARG    # misaligned


def test_masked_rejects_before_launch(lib):
    """Host-side checks of the mask arguments (dummy pointers; nothing is launched)."""
    import exact_attention_02_gb300 as fa
    vp, f, ll = ctypes.c_void_p, ctypes.c_float, ctypes.c_longlong
    L = fa.lib()
    L.fa_fwd_masked.argtypes = [vp] * 6 + [ll, ll, ll] + [ctypes.c_int] * 4 + [f, ctypes.c_int, ctypes.c_int, vp]

    def call(mask=P, sb=0, sh=0, srow=128, N=128, dtype=0, d=64):
        return L.fa_fwd_masked(vp(P), vp(P), vp(P), vp(P), vp(P), vp(mask), ll(sb), ll(sh), ll(srow), 1, 1, N, d,
                               f(0.125), 0, dtype, None)
    assert call(mask=0) == fa.FA_ERR_INVALID_ARG            # no mask
    assert call(mask=P + 8) == fa.FA_ERR_INVALID_ARG        # misaligned
    assert call(srow=120) == fa.FA_ERR_INVALID_ARG          # row shorter than N
    assert call(N=100, srow=100) == fa.FA_ERR_INVALID_ARG   # rows not padded to a multiple of 8
    assert call(sb=-8) == fa.FA_ERR_INVALID_ARG
    assert call(sh=4) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=1) == fa.FA_ERR_UNSUPPORTED           # the fp32 path has no mask
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED


def test_bitmask_rejects_before_launch(lib):
    """Host-side checks of the packed mask arguments (dummy pointers; nothing is launched)."""
    import exact_attention_02_gb300 as fa
    vp, f, ll = ctypes.c_void_p, ctypes.c_float, ctypes.c_longlong
    L = fa.lib()

    def call(bits=P, sb=0, sh=0, srow=4, N=128, dtype=0, d=64):
        return L.fa_fwd_bitmask(vp(P), vp(P), vp(P), vp(P), vp(P), vp(bits), ll(sb), ll(sh), ll(srow), 1, 1, N, d,
                                f(0.125), 0, dtype, None)
    assert call(bits=0) == fa.FA_ERR_INVALID_ARG            # no words
    assert call(bits=P + 4) == fa.FA_ERR_INVALID_ARG        # misaligned
    assert call(N=129, srow=4) == fa.FA_ERR_INVALID_ARG     # 2 key tiles need 8 words per row
    assert call(srow=6) == fa.FA_ERR_INVALID_ARG            # not a multiple of 4 words
    assert call(sb=-4) == fa.FA_ERR_INVALID_ARG
    assert call(sh=2) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=1) == fa.FA_ERR_UNSUPPORTED           # the fp32 path has no mask
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED


def test_pack_mask_bits_layout():
    """pack_mask_bits puts key j of a row at bit j % 32 of word j / 32, rows padded to 4
    words per 128 keys, written out here bit by bit with numpy."""
    import numpy as np
    torch = pytest.importorskip("torch")
    import exact_attention_02_gb300 as fa
    rng = np.random.default_rng(5)
    vis = rng.random((2, 3, 200, 200)) < 0.4
    got = fa.pack_mask_bits(torch.from_numpy(vis)).numpy().astype(np.int64) & 0xFFFFFFFF
    assert got.shape == (2, 3, 200, 8)
    want = np.zeros((2, 3, 200, 8), np.int64)
    for j in range(200):
        want[..., j // 32] |= vis[..., j].astype(np.int64) << (j % 32)
    assert np.array_equal(got, want)


def test_binding_checks_mask_bits_before_calling(lib):
    """The binding refuses packed bits of the wrong dtype, shape or row length before it
    calls into the library (CPU tensors: nothing reaches a device)."""
    torch = pytest.importorskip("torch")
    import exact_attention_02_gb300 as fa
    q = torch.zeros(2, 3, 200, 64, dtype=torch.bfloat16)
    good = fa.pack_mask_bits(torch.ones(1, 1, 200, 200, dtype=torch.bool))
    bad = [good.to(torch.int64),                              # not int32
           good[..., :4].contiguous(),                       # 4 words cannot hold 200 keys' tiles
           torch.zeros(1, 2, 200, 8, dtype=torch.int32),     # 2 heads for H = 3
           torch.zeros(1, 1, 199, 8, dtype=torch.int32),     # rows for the wrong N
           torch.zeros(1, 1, 200, 10, dtype=torch.int32)[..., :8],  # row stride not a multiple of 4
           good[0]]                                          # not 4-D
    for bits in bad:
        with pytest.raises(ValueError):
            fa.fa_fwd(q, q, q, False, mask_bits=bits)
        with pytest.raises(ValueError):
            fa.fa_bwd(q, q, q, q, q, torch.zeros(2, 3, 200), False, mask_bits=bits,
                      workspace=torch.zeros(16, dtype=torch.uint8))
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, False, mask_bits=good, dropout=(0.1, 1))


def test_dropout_rejects_before_launch(lib):
    """Host-side checks of the dropout rate (dummy pointers; nothing is launched)."""
    import exact_attention_02_gb300 as fa
    vp, f, i = ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    L = fa.lib()

    def call(p=0.1, dtype=0, d=64):
        return L.fa_fwd_dropout(vp(P), vp(P), vp(P), vp(P), vp(P), 1, 1, 128, d, f(0.125), 0, f(p),
                                ctypes.c_ulonglong(1), dtype, None)
    assert call(p=1.0) == fa.FA_ERR_INVALID_ARG
    assert call(p=-0.1) == fa.FA_ERR_INVALID_ARG
    assert call(p=float("nan")) == fa.FA_ERR_INVALID_ARG
    assert call(dtype=1) == fa.FA_ERR_UNSUPPORTED
    assert call(d=96) == fa.FA_ERR_UNSUPPORTED


def _fwd_rect(lib, ptrs=(P, P, P, P, P), Nq=128, Nk=256, **kw):
    a = dict(GOOD, **kw)
    return lib.fa_fwd_rect(*[ctypes.c_void_p(p) for p in ptrs], a["B"], a["H"], Nq, Nk, a["d"],
                           ctypes.c_float(a["scale"]), a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(Nq=0), 1), (dict(Nk=0), 1), (dict(Nk=-5), 1), (dict(d=96), 2),
    (dict(dtype=1, Nk=5000), 2), (dict(dtype=1, Nq=5000), 2), (dict(causal=3), 1),
    (dict(scale=0.0), 1), (dict(B=1 << 16, H=1 << 15), 1),
    # bf16 rows: the longer length counts against the 32-bit row limit
    (dict(B=1 << 10, H=1 << 10, Nq=1, Nk=1 << 12), 2),
])
def test_fwd_rect_rejects(lib, kw, code):
    assert _fwd_rect(lib, **kw) == code


@pytest.mark.parametrize("ptrs", [(0, P, P, P, P), (P, P, P, P, 0), (P + 8, P, P, P, P)])
def test_fwd_rect_rejects_pointers(lib, ptrs):
    assert _fwd_rect(lib, ptrs=ptrs) == 1


def test_bwd_rect_workspace_and_rejects(lib):
    assert lib.fa_bwd_rect_workspace_size(2, 4, 1000, 8192, 128, 0) == 2 * 4 * 1000 * 128 * 4  # dQ rows only
    assert lib.fa_bwd_rect_workspace_size(1, 1, 100, 300, 64, 1) == 0  # fp32: none
    assert lib.fa_bwd_rect_workspace_size(1, 1, 100, 0, 64, 0) == 0  # rejected
    v = [ctypes.c_void_p(P)] * 10
    ws = ctypes.c_void_p(P)
    need = lib.fa_bwd_rect_workspace_size(1, 1, 128, 256, 64, 0)
    # too small a workspace, and a zero key length
    assert lib.fa_bwd_rect(*v, ws, need - 16, 1, 1, 128, 256, 64, ctypes.c_float(0.125), 0, 0, None) == 5
    assert lib.fa_bwd_rect(*v, ws, need, 1, 1, 128, 0, 64, ctypes.c_float(0.125), 0, 0, None) == 1
