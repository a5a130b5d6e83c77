"""fa_fwd_bwd_host (host tensors, copies overlapped with the kernels) against the device
entry points on the same inputs: the same kernels run on the same values, so O, LSE, dK
and dV must be identical and dQ equal up to the order of its fp32 atomic additions."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()


@pytest.mark.parametrize("B,H,N,d,causal,chunks", [(2, 3, 256, 128, True, 4), (1, 5, 384, 64, False, 3),
                                                   (2, 2, 200, 128, True, 1), (1, 7, 512, 128, True, 16),
                                                   (4, 8, 1024, 128, True, 0)])
def test_host_pipeline_matches_device_calls(B, H, N, d, causal, chunks):
    g = torch.Generator().manual_seed(B * 100 + H * 10 + N)
    host = [torch.randn(B, H, N, d, generator=g).to(torch.bfloat16).pin_memory() for _ in range(4)]
    o, lse, dq, dk, dv = fa.fa_fwd_bwd_host(*host, causal, chunks=chunks)
    torch.cuda.current_stream().synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    dev = [t.cuda() for t in host]
    o2, lse2 = fa.fa_fwd(*dev[:3], causal)
    dq2, dk2, dv2 = fa.fa_bwd(*dev[:3], o2, dev[3], lse2, causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2.cpu()) and torch.equal(lse, lse2.cpu())
    assert torch.equal(dk, dk2.cpu()) and torch.equal(dv, dv2.cpu())
    rel = ((dq.float() - dq2.float().cpu()).norm() / dq2.float().norm().cpu()).item()
    assert rel < 1e-3, rel


def test_host_pipeline_follows_the_callers_stream():
    """Work queued on the caller's stream before the call is finished before the call
    reads its inputs, and the caller's stream waits for the call's results."""
    B, H, N, d = 1, 4, 512, 128
    g = torch.Generator().manual_seed(3)
    src = [torch.randn(B, H, N, d, generator=g).to(torch.bfloat16) for _ in range(4)]
    host = [torch.zeros(B, H, N, d, dtype=torch.bfloat16).pin_memory() for _ in range(4)]
    s = torch.cuda.Stream()
    staged = [t.cuda() for t in src]
    with torch.cuda.stream(s):
        torch.cuda._sleep(20_000_000)                      # keep the stream busy a while
        for h, t in zip(host, staged):
            h.copy_(t, non_blocking=True)                  # device -> pinned host, queued on s
        out = fa.fa_fwd_bwd_host(*host, True, chunks=2, stream=s)
    s.synchronize()
    dev = [t.cuda() for t in src]
    o2, _ = fa.fa_fwd(*dev[:3], True)
    torch.cuda.synchronize()
    assert torch.equal(out[0], o2.cpu())
