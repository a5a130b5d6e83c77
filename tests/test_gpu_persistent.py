"""The persistent backward's schedule, against the fp64 oracle.

The backward runs min(items, SMs) CTAs, and each takes (key tile, head) items in rounds of
one item per CTA, every other round in reverse order. These shapes put the item count just
below, at and just above one and two rounds of a 152-SM GB300. They also include a single
long causal head, whose items range from one query tile to 160. Every gradient of every head
is held to the bf16 bars of the square path (O max-abs 2e-2, LSE 1e-3, dQ/dK/dV relative
Frobenius 2e-2, D within its derived bound).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import Workload, make_inputs  # noqa: E402
from oracle import attention as ora  # noqa: E402

from test_gpu_parity import check, run_gpu  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


SHAPES = [  # (B, H, N, d, causal): items = B * H * ceil(N / 128)
    Workload("items151", 1, 151, 128, 128, "bf16", False, seed=60),
    Workload("items152_causal", 2, 76, 128, 64, "bf16", True, seed=61),
    Workload("items153_causal", 1, 51, 384, 128, "bf16", True, seed=62),
    Workload("items304", 1, 76, 512, 64, "bf16", False, seed=63),
    Workload("items308_causal", 1, 77, 512, 128, "bf16", True, seed=64),
    Workload("items460_ragged_causal", 1, 115, 500, 128, "bf16", True, seed=65),
    Workload("one_head_160_items_causal", 1, 1, 128 * 160, 64, "bf16", True, seed=66),
]


@pytest.mark.parametrize("w", SHAPES, ids=lambda w: w.name)
def test_schedule_matches_oracle(w):
    x = make_inputs(w)
    got = run_gpu(w, x)
    for b in range(w.B):
        for h in range(w.H):
            ref = ora.head_backward(*(x[n][b, h].astype(np.float64) for n in ("q", "k", "v", "do")), w.scale, w.causal)
            check(w, {n: got[n][b, h] for n in got}, ref, f"{w.name} ({b},{h})", do=x["do"][b, h])
