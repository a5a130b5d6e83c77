"""The two ways fa_bwd computes dQ (fa_set_bwd_dq_mode), each against the fp64 oracle.

FA_BWD_DQ_SEPARATE runs the 128-key-tile kernel for dK and dV alone and a second kernel over
128-query tiles for dQ; FA_BWD_DQ_ATOMIC adds fp32 dQ partials into the workspace. Both are
held to the parity bars of the square path (bf16: O max-abs 2e-2, LSE max-abs 1e-3,
dQ/dK/dV relative Frobenius 2e-2), on square, ragged and N_q != N_k shapes, causal and not,
at both head dimensions. dK and dV come from the same products in the same order in both
modes, so they agree bit for bit; dQ agrees to bf16 rounding.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import WORKLOADS, Workload, make_inputs, round_to_bf16  # noqa: E402
from oracle import attention as ora  # noqa: E402

from test_gpu_parity import check, run_gpu  # noqa: E402
from test_gpu_rect import check_head  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()
    yield
    fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_AUTO)


@pytest.fixture
def separate():
    fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_SEPARATE)
    yield
    fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_AUTO)


def test_mode_setting_round_trips_and_rejects_others():
    for m in (fa.FA_BWD_DQ_ATOMIC, fa.FA_BWD_DQ_SEPARATE, fa.FA_BWD_DQ_AUTO):
        fa.fa_set_bwd_dq_mode(m)
        assert fa.fa_get_bwd_dq_mode() == m
    with pytest.raises(fa.FAError):
        fa.fa_set_bwd_dq_mode(3)
    assert fa.fa_get_bwd_dq_mode() == fa.FA_BWD_DQ_AUTO


SQUARE = [
    Workload("sep_n128_d64", 1, 1, 128, 64, "bf16", False, seed=40),
    Workload("sep_n128_d128_causal", 1, 2, 128, 128, "bf16", True, seed=41),
    Workload("sep_n1_d64_causal", 1, 2, 1, 64, "bf16", True, seed=42),
    Workload("sep_n65_d128", 2, 1, 65, 128, "bf16", False, seed=43),
    Workload("sep_n333_d128_causal", 2, 1, 333, 128, "bf16", True, seed=44),
    Workload("sep_n640_d64_causal_qk2", 1, 2, 640, 64, "bf16", True, qk_gain=2.0, seed=45),
    Workload("sep_n777_d128_qk2", 1, 2, 777, 128, "bf16", False, qk_gain=2.0, seed=46),
    Workload("sep_n1024_d64", 2, 2, 1024, 64, "bf16", False, seed=47),
    Workload("sep_n2000_d128_causal", 1, 2, 2000, 128, "bf16", True, seed=48),
]


@pytest.mark.parametrize("w", SQUARE, ids=lambda w: w.name)
def test_separate_matches_oracle(w, separate):
    x = make_inputs(w)
    got = run_gpu(w, x)
    ref = ora.backward(*(x[n].astype(np.float64) for n in ("q", "k", "v", "do")), w.scale, w.causal)
    if w.N == 1:
        # One key: P = 1 and dS = P (dP - D) is exactly 0, so the oracle's dQ and dK are 0
        # and a relative error is undefined. The kernels' dP (tensor core) and D (the
        # preprocess pass) are fp32 sums of the same d products in different orders, so dQ
        # and dK sit at the rounding level of those sums: held to an absolute bound instead.
        for n in ("dq", "dk"):
            assert np.abs(ref[n]).max() == 0.0
            assert np.abs(got[n]).max() <= 1e-5, (n, np.abs(got[n]).max())
        got = dict(got, dq=ref["dq"], dk=ref["dk"])
    check(w, got, ref, w.name, do=x["do"])


RECT = [  # B, H, Nq, Nk, d, causal
    (1, 2, 300, 1000, 128, True),
    (1, 1, 65, 4096, 64, False),
    (1, 2, 1000, 129, 64, True),  # the first 871 queries see no key
    (2, 1, 777, 65, 128, False),
    (1, 1, 129, 1, 128, True),
]


@pytest.mark.parametrize("case", RECT, ids=lambda c: "B{}H{}q{}k{}d{}{}".format(*c[:5], "c" if c[5] else ""))
def test_separate_rect_matches_oracle(case, separate):
    B, H, Nq, Nk, d, causal = case
    rng = np.random.default_rng(Nq * 3 + Nk)
    x = {n: round_to_bf16(rng.standard_normal((B, H, Nq if n in ("q", "do") else Nk, d), dtype=np.float32))
         for n in ("q", "k", "v", "do")}
    scale = 1.0 / math.sqrt(d)
    q, k, v, do = (torch.from_numpy(x[n]).cuda().to(torch.bfloat16) for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd_rect(q, k, v, causal, scale)
    D = fa.fa_bwd_preprocess(o, do)
    dq, dk, dv = fa.fa_bwd_rect(q, k, v, o, do, lse, causal, scale, D=D)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    got = {n: t.float().cpu().numpy().astype(np.float64) for n, t in dict(o=o, lse=lse, d=D, dq=dq, dk=dk, dv=dv).items()}
    for b in range(B):
        for h in range(H):
            ref = ora.head_backward(*(x[n][b, h].astype(np.float64) for n in ("q", "k", "v", "do")), scale, causal)
            g = {n: got[n][b, h] for n in got}
            if Nk == 1:  # one key: dQ and dK are exactly 0 (see test_separate_matches_oracle)
                for n in ("dq", "dk"):
                    assert np.abs(ref[n]).max() == 0.0
                    assert np.abs(g[n]).max() <= 1e-5, (n, np.abs(g[n]).max())
                g = dict(g, dq=ref["dq"], dk=ref["dk"])
            check_head(g, ref, "bf16", x["do"][b, h], f"q{Nq} k{Nk} ({b},{h})")


@pytest.mark.parametrize("shape", [(2, 4, 1536, 128, True), (2, 4, 1000, 64, False)], ids=["d128c", "d64"])
def test_modes_agree(shape):
    """dK and dV bit for bit; dQ to bf16 rounding (relative Frobenius difference well under
    the oracle bar)."""
    B, H, N, d, causal = shape
    w = Workload("agree", B, H, N, d, "bf16", causal, seed=N + d)
    x = make_inputs(w)
    q, k, v, do = (torch.from_numpy(x[n]).cuda().to(torch.bfloat16) for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, causal, w.scale)
    out = {}
    try:
        for m in (fa.FA_BWD_DQ_ATOMIC, fa.FA_BWD_DQ_SEPARATE):
            fa.fa_set_bwd_dq_mode(m)
            out[m] = fa.fa_bwd(q, k, v, o, do, lse, causal, w.scale)
            torch.cuda.synchronize()
            assert fa.fa_get_last_device_status() == fa.FA_OK
    finally:
        fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_AUTO)
    a, s = out[fa.FA_BWD_DQ_ATOMIC], out[fa.FA_BWD_DQ_SEPARATE]
    assert torch.equal(a[1], s[1]) and torch.equal(a[2], s[2])
    dqa, dqs = a[0].double(), s[0].double()
    assert float((dqa - dqs).norm() / dqa.norm()) < 5e-3


def test_separate_is_deterministic(separate):
    """No atomic additions: repeated calls give the same dQ bit for bit."""
    w = Workload("det", 1, 4, 2048, 128, "bf16", True, seed=77)
    x = make_inputs(w)
    q, k, v, do = (torch.from_numpy(x[n]).cuda().to(torch.bfloat16) for n in ("q", "k", "v", "do"))
    o, lse = fa.fa_fwd(q, k, v, True, w.scale)
    g1 = fa.fa_bwd(q, k, v, o, do, lse, True, w.scale)
    g2 = fa.fa_bwd(q, k, v, o, do, lse, True, w.scale)
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(g1, g2))


@pytest.mark.parametrize("name", ["b2h16_n8192_d128_bf16_causal", "b16h32_n1024_d128_bf16", "b4h16_n2048_d64_bf16"])
def test_separate_full_size(name, separate):
    """The bench's workloads in the separate mode: three whole heads against the oracle."""
    w = WORKLOADS[name]
    x = make_inputs(w)
    got = run_gpu(w, x)
    bh = w.B * w.H
    for i in sorted({0, bh // 2, bh - 1}):
        b, h = i // w.H, i % w.H
        ref = ora.head_backward(*(x[n][b, h].astype(np.float64) for n in ("q", "k", "v", "do")), w.scale, w.causal)
        check(w, {n: got[n][b, h] for n in got}, ref, f"{name} ({b},{h})", do=x["do"][b, h])
