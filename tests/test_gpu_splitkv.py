"""Split-KV forward (few queries against a long key/value sequence) against the fp64 oracle.

Tolerances as for the bf16 forward: O max-abs <= 2e-2, LSE max-abs <= 1e-3. Causal cases
place the N_q queries at the last N_q key positions (bottom-right alignment).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import round_to_bf16  # noqa: E402
from oracle import attention as ora  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


CASES = [  # B, H, Nq, Nk, d, causal, qk_gain
    (1, 2, 1, 1, 128, True, 1.0),
    (1, 2, 1, 7, 64, False, 1.0),
    (2, 3, 1, 1000, 128, True, 1.0),
    (1, 4, 3, 4096, 128, True, 2.0),
    (1, 2, 4, 333, 64, False, 1.0),
    (2, 2, 5, 2048, 128, True, 1.0),
    (1, 2, 16, 3000, 64, True, 1.0),
    (1, 1, 16, 16, 128, True, 4.0),
    (1, 2, 9, 40000, 128, False, 1.0),
    # CTA key ranges that end inside a head and cover the next head's start
    (4, 16, 1, 300, 128, True, 1.0),
    (2, 8, 7, 777, 64, True, 1.0),
    # one head spread over ~150 CTAs, merged from ~150 partial states
    (1, 1, 1, 100000, 128, False, 1.0),
    # 1000 heads of 5 keys: dozens of short segments per CTA
    (10, 100, 2, 5, 128, True, 1.0),
    (1, 2, 12, 4096, 128, True, 2.0),
    # more d = 128 cases (the tensor-core partial kernel)
    (1, 4, 32, 4096, 128, True, 1.0),
    (2, 2, 64, 3000, 128, False, 1.0),
    (1, 2, 2, 1000, 128, True, 2.0),
    (1, 1, 40, 257, 128, True, 1.0),
    (4, 8, 8, 600, 128, True, 4.0),      # peaky scores: the running max moves often
    (1, 1, 64, 100000, 128, True, 1.0),  # one head over ~150 CTAs
    (10, 100, 3, 5, 128, True, 1.0),     # dozens of short segments per CTA
    # query groups of C = 8, 16, 32 columns: one query in the second group, then both full
    (1, 3, 9, 5000, 128, True, 2.0),
    (2, 2, 17, 1500, 128, False, 1.0),
    (1, 2, 33, 2048, 128, True, 4.0),
    (3, 5, 16, 700, 128, True, 1.0),
    # d = 64 with more than 16 queries, every query-group width
    (1, 2, 24, 3000, 64, True, 1.0),
    (2, 3, 64, 1000, 64, False, 2.0),
    (1, 1, 40, 100000, 64, True, 1.0),
    (4, 4, 33, 777, 64, True, 4.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}H{}q{}k{}d{}{}g{}".format(*c[:5], "c" if c[5] else "", c[6]))
def test_splitkv_matches_oracle(case):
    B, H, Nq, Nk, d, causal, gain = case
    rng = np.random.default_rng(Nq * 1000 + Nk)
    q = round_to_bf16(rng.standard_normal((B, H, Nq, d), dtype=np.float32) * gain)
    k = round_to_bf16(rng.standard_normal((B, H, Nk, d), dtype=np.float32) * gain)
    v = round_to_bf16(rng.standard_normal((B, H, Nk, d), dtype=np.float32))
    dev = [torch.from_numpy(a).cuda().to(torch.bfloat16) for a in (q, k, v)]
    scale = 1 / math.sqrt(d)
    o, lse = fa.fa_fwd_splitkv(*dev, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    for b in range(B):
        for h in range(H):
            O, L = ora.head_forward(q[b, h].astype(np.float64), k[b, h].astype(np.float64),
                                    v[b, h].astype(np.float64), scale, causal)
            assert np.abs(o[b, h] - O).max() <= 2e-2, (b, h)
            assert np.abs(lse[b, h] - L).max() <= 1e-3, (b, h)


def test_splitkv_agrees_with_square_forward():
    """The last N_q rows of a square causal forward equal the split-KV forward of those queries."""
    B, H, N, d, Nq = 1, 4, 1536, 128, 4
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(B, H, N, d, generator=g).cuda().to(torch.bfloat16) for _ in range(3))
    o_full, lse_full = fa.fa_fwd(q, k, v, True)
    o, lse = fa.fa_fwd_splitkv(q[:, :, -Nq:].contiguous(), k, v, True)
    torch.cuda.synchronize()
    assert (o.float() - o_full[:, :, -Nq:].float()).abs().max().item() <= 1e-2
    assert (lse - lse_full[:, :, -Nq:]).abs().max().item() <= 1e-4
