"""FP8 (e4m3) forward through the C ABI against the fp64 oracle of oracle/fp8.py.

The oracle is the exact attention of the dequantised inputs. The kernel rounds the
attention weights to e4m3 before they multiply V; every other step is fp32. Two checks
follow from that arithmetic, written per element of O (row i, column c), with P the
oracle's weights, w_j = P_ij / max_j P_ij and V the dequantised values:

1. A hard bound. A weight with w_j >= 2^-10 is stored in e4m3's normal range, so its
   rounding error is at most 2^-4 of itself; a smaller one is off by at most its whole
   value. O is also rounded once to bf16 (half an ulp, 2^-8 relative), and LSE-level
   fp32 effects add a tiny absolute term:
       |O_gpu - O| <= 2^-4 sum_{w>=2^-10} P|V| + sum_{w<2^-10} P|V| + 2^-8 |O| + 1e-4 sum P|V| + 1e-6
2. A noise check. Round-to-nearest errors are unbiased, with a standard deviation of at
   most 2^-4/sqrt(3) of each weight, so O's error has a standard deviation of at most
   sigma = 2^-4/sqrt(3) sqrt(sum_j P^2 V^2) (plus the bf16 and small-weight terms). The
   root mean square of (O_gpu - O) / sigma over a head must stay below 1.5: a wrong
   tile or a dropped term gives values far above it, while the hard bound alone is loose
   for rows whose weights are all small.
LSE is fp32 throughout: max-abs <= 1e-3 (the bf16 forward's bar).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import make_fp8_inputs  # noqa: E402
from oracle import attention as ora  # noqa: E402
from oracle import fp8 as ofp8  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


def _bounds(q, k, v, scale, causal, O):
    """(hard bound, sigma) per element of O for one head of dequantised inputs."""
    N = q.shape[0]
    s = ora.scores(q, k, scale, causal, np.arange(N))
    P, _, _ = ora.softmax_rows(s)
    w = P / P.max(axis=1, keepdims=True)
    big = w >= 2.0 ** -10
    av = np.abs(v)
    a_big = (P * big) @ av
    a_small = (P * ~big) @ av
    a_all = P @ av
    hard = 2.0 ** -4 * a_big + a_small + 2.0 ** -8 * np.abs(O) + 1e-4 * a_all + 1e-6
    sigma = 2.0 ** -4 / np.sqrt(3) * np.sqrt((P * P) @ (v * v)) + a_small + 2.0 ** -9 * np.abs(O) + 1e-6
    return hard, sigma


CASES = [  # B, H, N, causal, qk_gain
    (1, 2, 256, False, 1.0),
    (1, 2, 384, True, 1.0),
    (1, 1, 1, True, 1.0),
    (2, 3, 1000, True, 1.0),
    (1, 2, 129, False, 2.0),
    (1, 4, 2048, True, 2.0),
    (1, 2, 4096, False, 1.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}N{}{}g{}".format(c[0], c[1], c[2], "c" if c[3] else "", c[4]))
def test_fp8_forward_matches_oracle(case):
    B, H, N, causal, gain = case
    d = 128
    (q8, k8, v8), desc = make_fp8_inputs(B, H, N, d, seed=N + 7 * H, qk_gain=gain)
    dev = [torch.from_numpy(x).cuda() for x in (q8, k8, v8)]
    scale = 1 / np.sqrt(d)
    o, lse = fa.fa_fwd_fp8(*dev, desc, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        for h in range(H):
            q, k, v = (ofp8.dequantize(x[b, h], f) for x, f in zip((q8, k8, v8), desc))
            O, L = ora.head_forward(q, k, v, scale, causal)
            assert np.abs(lse[b, h] - L).max() <= 1e-3, (b, h)
            err = np.abs(o[b, h] - O)
            hard, sigma = _bounds(q, k, v, scale, causal, O)
            assert np.all(err <= hard), (b, h, float((err / hard).max()))
            z = float(np.sqrt(np.mean((err / sigma) ** 2)))
            assert z <= 1.5, (b, h, z)


def test_fp8_rejects_unsupported_head_dim():
    x = torch.zeros(1, 1, 128, 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_fp8(x, x, x, (1.0, 1.0, 1.0), False)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED


def test_fp8_matches_bf16_forward_on_exact_values():
    """With power-of-two factors every dequantised value is exactly a bf16 value, so the
    bf16 forward sees the same inputs: the two outputs differ only by the weights'
    rounding (e4m3 against bf16)."""
    B, H, N, d = 1, 4, 1024, 128
    (q8, k8, v8), _ = make_fp8_inputs(B, H, N, d, seed=11)
    desc = (2.0 ** -7, 2.0 ** -7, 2.0 ** -8)
    dev8 = [torch.from_numpy(x).cuda() for x in (q8, k8, v8)]
    o8, l8 = fa.fa_fwd_fp8(*dev8, desc, True)
    deq = [torch.from_numpy(ofp8.dequantize(x, f)).cuda().to(torch.bfloat16) for x, f in zip((q8, k8, v8), desc)]
    assert all(torch.equal(t.double().cpu(), torch.from_numpy(ofp8.dequantize(x, f))) for t, x, f in
               zip(deq, (q8, k8, v8), desc))
    ob, lb = fa.fa_fwd(*deq, True)
    torch.cuda.synchronize()
    assert (l8 - lb).abs().max().item() <= 1e-4
    rel = ((o8.float() - ob.float()).norm() / ob.float().norm()).item()
    assert rel <= 0.05, rel
