"""Dropout (fa_fwd_dropout / fa_bwd_dropout) through the C ABI against the fp64 oracle.

The keep bits are Philox-4x32-10 on both sides (oracle/philox.py and the kernels'
philox.cuh, written separately from the same published definition), so the dropped
attention is the same function of the inputs, and the tolerances are those of every bf16
test: O max-abs 2e-2, LSE 1e-3 (the undropped softmax's), dQ/dK/dV relative Frobenius
2e-2. Kept weights are multiplied by c = 256 / (256 - t), which scales O and its rounding
errors (the bf16 weights, the bf16 output) by c, up to 2 at p = 0.5; the bound on O is
nonetheless not widened by c, and the test records how the error moves with c. Two tests read the keep
bits of each kernel back exactly: with Q = 0 every visible weight is 1/N, and one-hot V
(or dO) rows weighted 1 for keys (queries) below 128 and 2 above turn each output element
into (K1 + 2 K2) c / N, from which both keep bits follow.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import round_to_bf16  # noqa: E402
from oracle import attention as ora  # noqa: E402
from oracle import philox  # noqa: E402

pytestmark = pytest.mark.gpu
SEED = 0x0123_4567_89AB_CDEF


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


CASES = [  # B, H, N, d, causal, p, seed
    (1, 2, 256, 128, False, 0.1, SEED),
    (2, 2, 384, 64, True, 0.3, 7),
    (1, 3, 200, 128, True, 0.5, 2 ** 40 + 3),
    (2, 2, 1024, 128, True, 0.2, 11),
    (1, 2, 640, 64, False, 0.05, 12345),
    # more items than SMs: each persistent backward CTA runs two or three (key tile, head) items
    (1, 40, 1024, 128, True, 0.2, 13),
    (1, 48, 700, 64, False, 0.1, 14),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}d{}{}-p{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_dropout_matches_oracle(case):
    B, H, N, d, causal, p, seed = case
    rng = np.random.default_rng(N + d)
    q, k, v, do = (round_to_bf16(rng.standard_normal((B, H, N, d), dtype=np.float32)) for _ in range(4))
    dev = [torch.from_numpy(a).cuda().to(torch.bfloat16) for a in (q, k, v, do)]
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(*dev[:3], causal, scale, dropout=(p, seed))
    dq, dk, dv = fa.fa_bwd(*dev[:3], o, dev[3], lse, causal, scale, dropout=(p, seed))
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    got = {n: t.float().cpu().numpy() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    c = philox.keep_scale(philox.threshold(p))
    for b in range(B):
        for h in range(H):
            K = philox.keep_matrix(seed, b * H + h, N, N, p)
            ref = ora.head_backward(*(x[b, h].astype(np.float64) for x in (q, k, v, do)), scale, causal,
                                    keep=K, keep_scale=c)
            # O grows by c with the kept weights, and so does its bf16 rounding; the bound
            # stays the fixed one of every bf16 test
            e_o = np.abs(got["o"][b, h] - ref["o"]).max()
            assert e_o <= 2e-2, (b, h, "o", e_o, "c", c)
            assert np.abs(got["lse"][b, h] - ref["lse"]).max() <= 1e-3, (b, h)
            for n in ("dq", "dk", "dv"):
                assert _rel(got[n][b, h], ref[n]) <= 2e-2, (b, h, n, _rel(got[n][b, h], ref[n]))


def _decode(x, unit):
    """(bit for index < 128, bit for index >= 128) from values (K1 + 2 K2) * unit."""
    k = np.rint(x / unit).astype(int)
    assert np.all((k >= 0) & (k <= 3)) and np.allclose(x, k * unit, rtol=2e-2, atol=0), "not a keep code"
    return k & 1, k >> 1


@pytest.mark.parametrize("p,seed", [(0.3, SEED), (0.5, 99)])
def test_forward_keep_bits_exact(p, seed):
    B, H, N, d = 1, 3, 256, 128
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(B, H, N, d, device="cuda").to(torch.bfloat16)
    v = torch.zeros(B, H, N, d, device="cuda")
    for j in range(N):
        v[:, :, j, j % 128] = 1.0 if j < 128 else 2.0
    o, _ = fa.fa_fwd(q, k, v.to(torch.bfloat16), False, dropout=(p, seed))
    torch.cuda.synchronize()
    unit = philox.keep_scale(philox.threshold(p)) / N
    o = o.float().cpu().numpy()
    for h in range(H):
        K = philox.keep_matrix(seed, h, N, N, p)
        lo, hi = _decode(o[0, h], unit)
        assert np.array_equal(lo, K[:, :128]) and np.array_equal(hi, K[:, 128:]), h


@pytest.mark.parametrize("p,seed", [(0.3, SEED), (0.5, 99)])
def test_backward_keep_bits_exact(p, seed):
    """dV_j = sum_i P_ij K_ij c dO_i: with uniform P and one-hot dO rows, dV reveals K^T."""
    B, H, N, d = 1, 2, 256, 128
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(B, H, N, d, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, H, N, d, device="cuda").to(torch.bfloat16)
    do = torch.zeros(B, H, N, d, device="cuda")
    for i in range(N):
        do[:, :, i, i % 128] = 1.0 if i < 128 else 2.0
    do = do.to(torch.bfloat16)
    o, lse = fa.fa_fwd(q, k, v, False, dropout=(p, seed))
    _, _, dv = fa.fa_bwd(q, k, v, o, do, lse, False, dropout=(p, seed))
    torch.cuda.synchronize()
    unit = philox.keep_scale(philox.threshold(p)) / N
    dv = dv.float().cpu().numpy()
    for h in range(H):
        K = philox.keep_matrix(seed, h, N, N, p)
        lo, hi = _decode(dv[0, h], unit)          # [key j, column c]: queries c and c + 128
        assert np.array_equal(lo, K[:128, :].T) and np.array_equal(hi, K[128:, :].T), h


def test_zero_rate_equals_no_dropout():
    B, H, N, d = 1, 2, 512, 128
    g = torch.Generator().manual_seed(4)
    q, k, v, do = (torch.randn(B, H, N, d, generator=g).cuda().to(torch.bfloat16) for _ in range(4))
    o0, l0 = fa.fa_fwd(q, k, v, True)
    o1, l1 = fa.fa_fwd(q, k, v, True, dropout=(0.0, 5))
    g0 = fa.fa_bwd(q, k, v, o0, do, l0, True)
    g1 = fa.fa_bwd(q, k, v, o1, do, l1, True, dropout=(0.0, 5))
    torch.cuda.synchronize()
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    for a, b in zip(g0, g1):
        assert ((a.float() - b.float()).norm() / b.float().norm()).item() <= 1e-2
