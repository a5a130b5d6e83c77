"""The device entry points under CUDA stream capture: fa_fwd, fa_bwd_preprocess and fa_bwd
captured into one CUDA graph and replayed give the results of the same calls made eagerly.

Every call only enqueues kernels (and a clearing of the dQ accumulator) on the given stream,
with arguments fixed at the call, so a captured step replays without the host. O, LSE, D,
dK and dV must agree bit for bit; dQ too in the deterministic dQ mode, and to fp32 summation
order in the default one (its partials are added atomically).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import Workload, make_inputs  # noqa: E402

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


@pytest.mark.parametrize("mode", ["atomic", "separate"])
@pytest.mark.parametrize("shape", [(1, 4, 1000, 128, True), (2, 2, 2048, 64, False)], ids=["d128c", "d64"])
def test_captured_step_replays_like_eager(shape, mode):
    B, H, N, d, causal = shape
    fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_SEPARATE if mode == "separate" else fa.FA_BWD_DQ_ATOMIC)
    w = Workload("graph", B, H, N, d, "bf16", causal, seed=N + d)
    x = make_inputs(w)
    q, k, v, do = (torch.from_numpy(x[n]).cuda().to(torch.bfloat16) for n in ("q", "k", "v", "do"))
    out = dict(o=torch.empty_like(q), lse=torch.empty(B, H, N, device="cuda"), D=torch.empty(B, H, N, device="cuda"),
               dq=torch.empty_like(q), dk=torch.empty_like(q), dv=torch.empty_like(q))
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N, d, torch.bfloat16), dtype=torch.uint8, device="cuda")

    def step():
        fa.fa_fwd(q, k, v, causal, w.scale, o=out["o"], lse=out["lse"])
        fa.fa_bwd_preprocess(out["o"], do, D=out["D"])
        fa.fa_bwd(q, k, v, out["o"], do, out["lse"], causal, w.scale, D=out["D"], dq=out["dq"], dk=out["dk"],
                  dv=out["dv"], workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager warm-up: one-time set-up happens outside the capture
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = {n: t.clone() for n, t in out.items()}
    for t in out.values():
        t.fill_(float("nan"))

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        for t in out.values():
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert fa.fa_get_last_device_status() == fa.FA_OK
        for n in ("o", "lse", "D", "dk", "dv"):
            assert torch.equal(out[n], eager[n]), n
        if mode == "separate":
            assert torch.equal(out["dq"], eager["dq"])
        else:
            a, b = out["dq"].double(), eager["dq"].double()
            assert torch.isfinite(a).all() and float((a - b).norm() / b.norm()) < 1e-3
