"""fa_fwd_rect / fa_bwd_rect (Nq query rows against Nk key rows) against the fp64 oracle,
through the C ABI.

Causal attention is bottom-right aligned: query i hides keys j > i + Nk - Nq, and with
Nq > Nk the first Nq - Nk queries see no key (O = 0, LSE = -inf, dQ = 0). Tolerances are
those of the square path: bf16 O max-abs 2e-2, LSE max-abs 1e-3, dQ/dK/dV relative
Frobenius 2e-2; fp32 max-abs 1e-4 on everything. Inputs are N(0, 1) from
default_rng(seed), rounded to bf16 for the bf16 cases.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import round_to_bf16  # noqa: E402
from oracle import attention as ora  # noqa: E402

from test_gpu_parity import check_d  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


def _inputs(B, H, Nq, Nk, d, dtype, seed, gain=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, Nq, d), dtype=np.float32) * np.float32(gain)
    k = rng.standard_normal((B, H, Nk, d), dtype=np.float32) * np.float32(gain)
    v = rng.standard_normal((B, H, Nk, d), dtype=np.float32)
    do = rng.standard_normal((B, H, Nq, d), dtype=np.float32)
    if dtype == "bf16":
        q, k, v, do = (round_to_bf16(a) for a in (q, k, v, do))
    return dict(q=q, k=k, v=v, do=do)


def _dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def run_rect(x, dtype, causal, scale):
    q, k, v, do = (_dev(x[n], dtype) for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd_rect(q, k, v, causal, scale)
    D = fa.fa_bwd_preprocess(o, do)
    dq, dk, dv = fa.fa_bwd_rect(q, k, v, o, do, lse, causal, scale, D=D)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    out = dict(o=o, lse=lse, d=D, dq=dq, dk=dk, dv=dv)
    return {n: t.float().cpu().numpy().astype(np.float64) for n, t in out.items()}


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def check_head(got, ref, dtype, do, where):
    """One head: rows that see no key must be exactly O = 0, LSE = -inf, dQ = 0; the rest
    within the square path's tolerances (D against its derived bound)."""
    hidden = ~np.isfinite(ref["lse"])
    assert np.array_equal(np.isfinite(got["lse"]), ~hidden), (where, "hidden rows")
    assert np.all(got["o"][hidden] == 0) and np.all(got["dq"][hidden] == 0), (where, "hidden rows not zero")
    vis = ~hidden
    for n in ("o", "dq", "dk", "dv"):
        assert np.isfinite(got[n]).all(), (where, n, "non-finite")
    if dtype == "fp32":
        for n in ("o", "dq", "dk", "dv"):
            err = np.abs(got[n] - ref[n]).max()
            assert err <= 1e-4, (where, n, err)
        assert np.abs(got["lse"][vis] - ref["lse"][vis]).max(initial=0) <= 1e-4, where
    else:
        e_o = np.abs(got["o"] - ref["o"]).max()
        assert e_o <= 2e-2, (where, "o", e_o)
        e_l = np.abs(got["lse"][vis] - ref["lse"][vis]).max(initial=0)
        assert e_l <= 1e-3, (where, "lse", e_l)
        for n in ("dq", "dk", "dv"):
            if np.linalg.norm(ref[n]) == 0:
                assert np.all(got[n] == 0), (where, n)
                continue
            r = _rel(got[n], ref[n])
            assert r <= 2e-2, (where, n, r)
    check_d(got, ref, do, where)


def _compare(B, H, Nq, Nk, d, causal, dtype="bf16", seed=0, gain=1.0, heads=None):
    x = _inputs(B, H, Nq, Nk, d, dtype, seed, gain)
    scale = 1.0 / math.sqrt(d)
    got = run_rect(x, dtype, causal, scale)
    pick = heads if heads is not None else [(b, h) for b in range(B) for h in range(H)]
    for b, h in pick:
        ref = ora.head_backward(*(x[n][b, h].astype(np.float64) for n in ("q", "k", "v", "do")), scale, causal)
        check_head({n: got[n][b, h] for n in got}, ref, dtype, x["do"][b, h], f"Nq={Nq} Nk={Nk} ({b},{h})")
    return x, got


CASES = [  # B, H, Nq, Nk, d, causal, gain
    # fewer queries than keys: a prefill continuing a cache, or cross-attention
    (1, 2, 65, 32768, 128, True, 1.0),
    (1, 1, 65, 32768, 64, False, 1.0),
    (1, 2, 1000, 8192, 128, True, 2.0),
    (1, 1, 1000, 32768, 64, True, 1.0),
    (2, 1, 1000, 4096, 128, False, 1.0),
    (1, 1, 4096, 8192, 64, True, 1.0),
    (1, 2, 4096, 8192, 128, False, 1.0),
    (1, 2, 4096, 32768, 128, True, 1.0),
    (1, 2, 384, 640, 64, True, 4.0),
    (2, 2, 1, 300, 128, True, 1.0),
    (1, 3, 129, 1000, 64, False, 1.0),
    # more queries than keys: the first Nq - Nk queries see no key when causal
    (1, 2, 300, 200, 128, True, 1.0),
    (1, 1, 1000, 129, 64, True, 1.0),
    (2, 1, 777, 65, 128, False, 1.0),
    (1, 2, 8192, 1000, 128, True, 1.0),
    (1, 2, 129, 1, 64, True, 1.0),
    (1, 1, 1, 1, 128, True, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else ""))
def test_rect_matches_oracle(case):
    B, H, Nq, Nk, d, causal, gain = case
    # one whole head per batch for the long key sequences keeps the oracle to seconds
    heads = [(b, 0) for b in range(B)] if Nq * Nk > 8192 * 8192 else None
    _compare(B, H, Nq, Nk, d, causal, seed=Nq * 7 + Nk, gain=gain, heads=heads)


@pytest.mark.parametrize("case", [(1, 2, 100, 300, 64, True), (1, 1, 300, 100, 128, True),
                                  (1, 2, 77, 200, 128, False), (2, 1, 33, 5, 64, True)],
                         ids=lambda c: "q{}k{}d{}{}".format(*c[2:5], "c" if c[5] else ""))
def test_rect_fp32_matches_oracle(case):
    B, H, Nq, Nk, d, causal = case
    _compare(B, H, Nq, Nk, d, causal, dtype="fp32", seed=Nq + 3 * Nk)


@pytest.mark.parametrize("d", [64, 128])
def test_square_rect_equals_fa_fwd_bwd(d):
    """Nq = Nk through fa_fwd_rect / fa_bwd_rect is fa_fwd / fa_bwd, bit for bit (dQ up to
    the order of its fp32 atomic adds)."""
    x = _inputs(2, 2, 700, 700, d, "bf16", 90 + d)
    q, k, v, do = (_dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    o1, l1 = fa.fa_fwd(q, k, v, True)
    o2, l2 = fa.fa_fwd_rect(q, k, v, True)
    D = fa.fa_bwd_preprocess(o1, do)
    g1 = fa.fa_bwd(q, k, v, o1, do, l1, True, D=D)
    g2 = fa.fa_bwd_rect(q, k, v, o1, do, l1, True, D=D)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert _rel(g2[0].float().cpu().numpy(), g1[0].float().cpu().numpy()) < 1e-3


@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (128, 8192), (1000, 1001)])
def test_causal_rect_rows_equal_square_rows(Nq, Nk):
    """Bottom-right causal: the Nq queries are the last Nq positions, so fa_fwd_rect gives
    the last Nq rows of the square causal forward on the full sequence, bit for bit (each
    row sees the same keys through the same K tiles)."""
    x = _inputs(1, 2, Nk, Nk, 128, "bf16", Nq + Nk)
    q, k, v = (_dev(x[n], "bf16") for n in ("q", "k", "v"))
    o_sq, l_sq = fa.fa_fwd(q, k, v, True)
    o_r, l_r = fa.fa_fwd_rect(q[:, :, Nk - Nq:].contiguous(), k, v, True)
    torch.cuda.synchronize()
    assert torch.equal(o_r, o_sq[:, :, Nk - Nq:]) and torch.equal(l_r, l_sq[:, :, Nk - Nq:])


def test_rect_rejects_mismatched_shapes():
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd_rect(q, k, k[:, :, :100], True)
    with pytest.raises(ValueError):
        fa.fa_fwd_rect(q, k[..., :32].contiguous(), k[..., :32].contiguous(), True)


@pytest.mark.parametrize("case", [(1, 1, 1000, 32768, 64, True), (1, 2, 1000, 8192, 128, True),
                                  (2, 4, 2048, 2048, 64, False), (1, 4, 4096, 4096, 128, True)],
                         ids=lambda c: "q{}k{}d{}{}".format(*c[2:5], "c" if c[5] else ""))
def test_dk_dv_identical_across_runs(case):
    """dK and dV take no atomic additions: four calls on the same inputs must agree bit for bit.
    A product that read a shared-memory stage before its copy landed would show up here as a
    run-to-run difference (dQ sums fp32 partials atomically, so only it may differ)."""
    B, H, Nq, Nk, d, causal = case
    x = _inputs(B, H, Nq, Nk, d, "bf16", seed=Nq + Nk + d)
    q, k, v, do = (_dev(x[n], "bf16") for n in ("q", "k", "v", "do"))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fa_fwd_rect(q, k, v, causal, scale)
    D = fa.fa_bwd_preprocess(o, do)
    first = fa.fa_bwd_rect(q, k, v, o, do, lse, causal, scale, D=D)
    for _ in range(3):
        again = fa.fa_bwd_rect(q, k, v, o, do, lse, causal, scale, D=D)
        torch.cuda.synchronize()
        assert torch.equal(first[1], again[1]) and torch.equal(first[2], again[2])
    assert fa.fa_get_last_device_status() == fa.FA_OK
