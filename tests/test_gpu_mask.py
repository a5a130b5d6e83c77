"""Additive mask (fa_fwd_masked / fa_bwd_masked) through the C ABI against the fp64 oracle.

The mask is added to the scaled scores before the softmax; -inf entries hide keys. Inputs
are N(0, 1) rounded to bf16 (the mask too: both sides read the same bf16 values), with
the bf16 tolerances of every other parity test: O max-abs 2e-2, LSE max-abs 1e-3 (and
-inf exactly where the oracle has no visible key), dQ/dK/dV relative Frobenius 2e-2.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import round_to_bf16  # noqa: E402
from oracle import attention as ora  # noqa: E402

pytestmark = pytest.mark.gpu
O_TOL, LSE_TOL, GRAD_TOL = 2e-2, 1e-3, 2e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


def _make_mask(kind, B, H, N, rng):
    """float32 mask of shape [mb, mh, N, N] (bf16 values) for one of the test patterns."""
    if kind == "bias":          # per-head dense bias with scattered -inf entries
        M = rng.standard_normal((B, H, N, N)).astype(np.float32) * 2
        M[rng.random((B, H, N, N)) < 0.1] = -np.inf
    elif kind == "broadcast":   # one [N, N] bias for every batch and head
        M = rng.standard_normal((1, 1, N, N)).astype(np.float32)
    elif kind == "padding":     # per-batch key length, shared by the heads
        M = np.zeros((B, 1, N, N), np.float32)
        for b in range(B):
            M[b, 0, :, max(1, N - 37 * (b + 1)):] = -np.inf
    elif kind == "hidden_rows":  # some queries see no key at all
        M = rng.standard_normal((B, H, N, N)).astype(np.float32)
        M[:, :, 3] = -np.inf
        M[:, :, N // 2:N // 2 + 5] = -np.inf
    else:
        raise ValueError(kind)
    return round_to_bf16(M)


CASES = [  # B, H, N, d, causal, kind
    (1, 2, 256, 128, False, "bias"),
    (2, 2, 384, 64, True, "broadcast"),
    (2, 3, 200, 128, False, "padding"),
    (1, 2, 256, 128, True, "hidden_rows"),
    (1, 2, 100, 64, False, "bias"),          # rows padded to 104 by padded_mask
    (1, 4, 1024, 128, True, "bias"),
    (2, 2, 640, 128, False, "broadcast"),
    # more items than SMs: each persistent backward CTA runs two or three (key tile, head) items
    (1, 40, 1024, 128, True, "bias"),
    (1, 48, 700, 64, False, "broadcast"),
]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}d{}{}-{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_masked_fwd_bwd_match_oracle(case):
    B, H, N, d, causal, kind = case
    rng = np.random.default_rng(N + 11 * d)
    q, k, v, do = (round_to_bf16(rng.standard_normal((B, H, N, d), dtype=np.float32)) for _ in range(4))
    M = _make_mask(kind, B, H, N, rng)
    dev = [torch.from_numpy(a).cuda().to(torch.bfloat16) for a in (q, k, v, do)]
    mask = fa.padded_mask(torch.from_numpy(M).cuda().to(torch.bfloat16))
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(*dev[:3], causal, scale, mask=mask)
    dq, dk, dv = fa.fa_bwd(*dev[:3], o, dev[3], lse, causal, scale, mask=mask)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    got = {n: t.float().cpu().numpy() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    for n in got:
        assert not np.isnan(got[n]).any(), n
    ref = ora.backward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), do.astype(np.float64),
                       scale, causal, mask=M.astype(np.float64))
    assert np.abs(got["o"] - ref["o"]).max() <= O_TOL
    hidden = np.isneginf(ref["lse"])
    assert np.array_equal(np.isneginf(got["lse"]), hidden)
    assert np.abs(got["lse"][~hidden] - ref["lse"][~hidden]).max() <= LSE_TOL
    if hidden.any():
        assert np.all(got["o"][hidden] == 0) and np.all(got["dq"][hidden] == 0)
    for n in ("dq", "dk", "dv"):
        assert _rel(got[n], ref[n]) <= GRAD_TOL, (n, _rel(got[n], ref[n]))


def test_zero_mask_equals_unmasked():
    """A zero mask reproduces the unmasked kernels' outputs to their rounding."""
    B, H, N, d = 1, 4, 512, 128
    g = torch.Generator().manual_seed(3)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g).cuda().to(torch.bfloat16) for _ in range(4))
    mask = torch.zeros(1, 1, N, N, dtype=torch.bfloat16, device="cuda")
    o0, l0 = fa.fa_fwd(q, k, v, True)
    o1, l1 = fa.fa_fwd(q, k, v, True, mask=mask)
    g0 = fa.fa_bwd(q, k, v, o0, do, l0, True)
    g1 = fa.fa_bwd(q, k, v, o1, do, l1, True, mask=mask)
    torch.cuda.synchronize()
    assert (o0.float() - o1.float()).abs().max().item() <= 1e-2
    assert (l0 - l1).abs().max().item() <= 1e-5
    for a, b in zip(g0, g1):
        assert ((a.float() - b.float()).norm() / b.float().norm()).item() <= 1e-2
