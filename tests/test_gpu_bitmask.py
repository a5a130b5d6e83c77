"""Boolean mask packed one bit per key (fa_fwd_bitmask / fa_bwd_bitmask) through the C ABI.

A boolean mask is the additive mask of "知识点13 FlashAttention深度攻略" section 7 with
entries 0 (visible) and -inf (hidden), so the oracle is the fp64 oracle's additive-mask
path with that M. Inputs are N(0, 1) rounded to bf16; the bf16 tolerances of every other
parity test apply: O max-abs 2e-2, LSE max-abs 1e-3 (and -inf exactly where the oracle has
no visible key), dQ/dK/dV relative Frobenius 2e-2. The packed path must also agree with
the bf16 additive-mask kernels given the same 0 / -inf mask, and with the unmasked
kernels when every bit is set.
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


def _visible(kind, B, H, N, rng):
    """Boolean [mb, mh, N, N] visibility pattern (True: the key is visible)."""
    if kind == "random":        # per head, about 30% of the keys hidden
        return rng.random((B, H, N, N)) >= 0.3
    if kind == "broadcast":     # one pattern for every batch and head
        return rng.random((1, 1, N, N)) >= 0.5
    if kind == "padding":       # per-batch key length, shared by the heads
        vis = np.ones((B, 1, N, N), bool)
        for b in range(B):
            vis[b, 0, :, max(1, N - 37 * (b + 1)):] = False
        return vis
    if kind == "hidden_rows":   # some queries see no key at all
        vis = rng.random((B, H, N, N)) >= 0.3
        vis[:, :, 3] = False
        vis[:, :, N // 2:N // 2 + 5] = False
        return vis
    if kind == "band":          # a sliding window |i - j| <= 64, shared by all heads
        i = np.arange(N)
        return (np.abs(i[:, None] - i[None, :]) <= 64)[None, None]
    raise ValueError(kind)


CASES = [  # B, H, N, d, causal, kind
    (1, 2, 256, 128, False, "random"),
    (2, 2, 384, 64, True, "broadcast"),
    (2, 3, 200, 128, False, "padding"),
    (1, 2, 256, 128, True, "hidden_rows"),
    (1, 2, 100, 64, False, "random"),
    (1, 4, 1024, 128, True, "random"),
    (2, 2, 640, 128, False, "band"),
    (1, 3, 333, 64, True, "hidden_rows"),
    # more items than SMs: each persistent backward CTA runs two or three (key tile, head) items
    (1, 40, 1024, 128, True, "random"),
    (1, 48, 700, 64, False, "band"),
]


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _inputs(B, H, N, d, seed):
    rng = np.random.default_rng(seed)
    host = [round_to_bf16(rng.standard_normal((B, H, N, d), dtype=np.float32)) for _ in range(4)]
    return rng, host, [torch.from_numpy(a).cuda().to(torch.bfloat16) for a in host]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}d{}{}-{}".format(*c[:4], "c" if c[4] else "", c[5]))
def test_bitmask_fwd_bwd_match_oracle(case):
    B, H, N, d, causal, kind = case
    rng, (q, k, v, do), dev = _inputs(B, H, N, d, 7 * N + d)
    vis = _visible(kind, B, H, N, rng)
    bits = fa.pack_mask_bits(torch.from_numpy(vis).cuda())
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd(*dev[:3], causal, scale, mask_bits=bits)
    dq, dk, dv = fa.fa_bwd(*dev[:3], o, dev[3], lse, causal, scale, mask_bits=bits)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    got = {n: t.float().cpu().numpy() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv))}
    for n in got:
        assert not np.isnan(got[n]).any(), n
    M = np.where(vis, 0.0, -np.inf)
    ref = ora.backward(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64), do.astype(np.float64),
                       scale, causal, mask=M)
    assert np.abs(got["o"] - ref["o"]).max() <= O_TOL
    hidden = np.isneginf(ref["lse"])
    assert np.array_equal(np.isneginf(got["lse"]), hidden)
    assert np.abs(got["lse"][~hidden] - ref["lse"][~hidden]).max() <= LSE_TOL
    if hidden.any():
        assert np.all(got["o"][hidden] == 0) and np.all(got["dq"][hidden] == 0)
    for n in ("dq", "dk", "dv"):
        assert _rel(got[n], ref[n]) <= GRAD_TOL, (n, _rel(got[n], ref[n]))


@pytest.mark.parametrize("causal", [False, True])
def test_bitmask_equals_additive_mask(causal):
    """The packed path and the bf16 additive-mask path compute the same thing for a 0 / -inf
    mask: identical scores reach identical softmax code, so O, LSE, dK and dV agree to
    rounding and dQ to the order of its atomic additions."""
    B, H, N, d = 2, 2, 384, 128
    rng, _, dev = _inputs(B, H, N, d, 17)
    vis = rng.random((B, H, N, N)) >= 0.4
    bits = fa.pack_mask_bits(torch.from_numpy(vis).cuda())
    mask = fa.padded_mask(torch.from_numpy(np.where(vis, 0.0, -np.inf).astype(np.float32)).cuda().to(torch.bfloat16))
    o0, l0 = fa.fa_fwd(*dev[:3], causal, mask=mask)
    o1, l1 = fa.fa_fwd(*dev[:3], causal, mask_bits=bits)
    g0 = fa.fa_bwd(*dev[:3], o0, dev[3], l0, causal, mask=mask)
    g1 = fa.fa_bwd(*dev[:3], o1, dev[3], l1, causal, mask_bits=bits)
    torch.cuda.synchronize()
    assert (o0.float() - o1.float()).abs().max().item() <= 1e-2
    fin = torch.isfinite(l0)
    assert torch.equal(fin, torch.isfinite(l1))
    assert (l0[fin] - l1[fin]).abs().max().item() <= 1e-5
    for a, b in zip(g0, g1):
        assert ((a.float() - b.float()).norm() / b.float().norm()).item() <= 1e-3


def test_all_visible_bits_equal_unmasked():
    B, H, N, d = 1, 4, 512, 128
    _, _, dev = _inputs(B, H, N, d, 23)
    bits = fa.pack_mask_bits(torch.ones(1, 1, N, N, dtype=torch.bool, device="cuda"))
    o0, l0 = fa.fa_fwd(*dev[:3], True)
    o1, l1 = fa.fa_fwd(*dev[:3], True, mask_bits=bits)
    g0 = fa.fa_bwd(*dev[:3], o0, dev[3], l0, True)
    g1 = fa.fa_bwd(*dev[:3], o1, dev[3], l1, True, mask_bits=bits)
    torch.cuda.synchronize()
    assert (o0.float() - o1.float()).abs().max().item() <= 1e-2
    assert (l0 - l1).abs().max().item() <= 1e-5
    for a, b in zip(g0, g1):
        assert ((a.float() - b.float()).norm() / b.float().norm()).item() <= 1e-2
