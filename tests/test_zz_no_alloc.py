"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Such callers (code inside a framework that owns all device memory, or latency-critical
paths that cannot take cudaMalloc's implicit synchronisation) get their scratch from a
static array inside the library instead of a caller-provided workspace. These tests
call the entry point through the C ABI and compare it with fa_bwd on the same inputs.
This file is collected last so that a run stopping at its first failure has already run
every other test.
"""
import ctypes
import math

import numpy as np
import pytest

import exact_attention_02_gb300 as fa
from exact_attention_02_gb300.workloads import Workload, make_inputs

GRAD_REL_TOL = 2e-2  # the bf16 gradient tolerance used by every GPU parity test
P = 0x10000          # dummy aligned address for host-only argument checks


def _noalloc(L):
    f = L.fa_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [vp] * 10 + [i, i, i, i, ctypes.c_float, i, i, vp]
    f.restype = i
    return f


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Host-side check, no GPU needed: too large a problem is refused before any launch."""
    from exact_attention_02_gb300.build import build
    build()
    f = _noalloc(fa.lib())
    vp = ctypes.c_void_p
    ptrs = [vp(P)] * 10
    # 2 x 16 x 8192 x 128 = 33.5 M elements > FA_NOALLOC_MAX_ELEMS (8 M)
    assert f(*ptrs, 2, 16, 8192, 128, 0.088, 1, fa.FA_DTYPE_BF16, None) == fa.FA_ERR_WORKSPACE
    # argument errors are reported as fa_bwd reports them
    assert f(*ptrs, 1, 1, 128, 96, 0.088, 1, fa.FA_DTYPE_BF16, None) == fa.FA_ERR_UNSUPPORTED
    assert f(*ptrs, 0, 1, 128, 128, 0.088, 1, fa.FA_DTYPE_BF16, None) == fa.FA_ERR_INVALID_ARG


NOALLOC_SHAPES = [  # the last two have more (key tile, head) items than a GB300 has SMs
    Workload("noalloc_b1h4_n1024_d128_bf16_causal", 1, 4, 1024, 128, "bf16", True, seed=21),
    Workload("noalloc_b1h8_n8192_d128_bf16_causal", 1, 8, 8192, 128, "bf16", True, seed=22),
    Workload("noalloc_b2h16_n2048_d64_bf16", 2, 16, 2048, 64, "bf16", False, seed=23),
]


@pytest.mark.gpu
@pytest.mark.parametrize("w", NOALLOC_SHAPES, ids=lambda w: w.name)
def test_noalloc_matches_fa_bwd_on_consecutive_calls(w):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    f = _noalloc(fa.lib())
    assert w.B * w.H * w.N * w.d <= 8 * 1024 * 1024
    x = make_inputs(w)
    q, k, v, do = (torch.from_numpy(x[n]).cuda().to(torch.bfloat16) for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, w.causal, w.scale)
    D = fa.fa_bwd_preprocess(o, do)
    ref = fa.fa_bwd(q, k, v, o, do, lse, w.causal, w.scale, D=D)  # the existing entry point
    torch.cuda.synchronize()

    def p(t):
        return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, Darg in enumerate((D, None)):  # second call also rebuilds D inside the scratch
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        st = f(p(q), p(k), p(v), p(o), p(do), p(lse), p(Darg), p(dq), p(dk), p(dv),
               w.B, w.H, w.N, w.d, ctypes.c_float(w.scale), int(w.causal), fa.FA_DTYPE_BF16, stream)
        assert st == fa.FA_OK, fa.error_string(st)
        torch.cuda.synchronize()
        assert fa.fa_get_last_device_status() == fa.FA_OK
        for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
            g, r = got.float(), want.float()
            assert torch.isfinite(g).all(), (call, name)
            rel = ((g - r).norm() / r.norm()).item()
            assert rel <= GRAD_REL_TOL, (call, name, rel)
        # dK and dV come from the same deterministic kernel: identical bits expected
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
