"""The failure path of the bounded device-side waits, made to run on purpose.

Every mbarrier wait in the tensor-core kernels gives up after a time limit; the kernel then
records FA_ERR_DEVICE_TIMEOUT in the device status word, stops its other roles, waits
(bounded) for its own copies and products in flight, frees its tensor memory and returns,
so the CUDA context stays usable. The test hook fa_test_inject_timeout makes the first CTA
of one kernel never arm one barrier (a phase that nothing completes) and shortens the limit
to 20 ms, at a tiny size. Nothing traps, faults or waits without a bound.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_02_gb300 as fa  # noqa: E402
from exact_attention_02_gb300.workloads import Workload, make_inputs  # noqa: E402
from oracle import attention as ora  # noqa: E402

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000  # 20 ms


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from exact_attention_02_gb300.build import build
    build()
    fa.lib()
    yield
    fa.fa_test_inject_timeout(fa.FA_INJECT_OFF, 0)


def _inputs():
    w = Workload("timeout_b1h1_n512_d128_bf16", 1, 1, 512, 128, "bf16", False, seed=31)
    x = make_inputs(w)
    return w, x, [torch.from_numpy(x[n]).cuda().to(torch.bfloat16) for n in ("q", "k", "v", "do")]


def _parity_after(w, x, dev):
    """A normal forward and backward right after the timeout match the oracle."""
    q, k, v, do = dev
    o, lse = fa.fa_fwd(q, k, v, w.causal, w.scale)
    dq, dk, dv = fa.fa_bwd(q, k, v, o, do, lse, w.causal, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK
    ref = ora.head_backward(*(x[n][0, 0].astype(np.float64) for n in ("q", "k", "v", "do")), w.scale, w.causal)
    got = {n: t[0, 0].float().cpu().numpy() for n, t in dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv).items()}
    assert np.abs(got["o"] - ref["o"]).max() <= 2e-2
    assert np.abs(got["lse"] - ref["lse"]).max() <= 1e-3
    for n in ("dq", "dk", "dv"):
        assert np.linalg.norm(got[n] - ref[n]) / np.linalg.norm(ref[n]) <= 2e-2, n


@pytest.mark.parametrize("which", ["fwd", "bwd", "bwd_separate_dq"])
def test_wait_that_runs_out_reports_timeout_and_the_context_survives(which):
    """bwd_separate_dq: the backward in the separate dQ mode, where both of its kernels (dK/dV
    and dQ) skip their first Q arrival in CTA 0."""
    w, x, dev = _inputs()
    q, k, v, do = dev
    o, lse = fa.fa_fwd(q, k, v, w.causal, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_last_device_status() == fa.FA_OK  # a clean word to start from
    try:
        if which == "bwd_separate_dq":
            fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_SEPARATE)
        fa.fa_test_inject_timeout(fa.FA_INJECT_FWD if which == "fwd" else fa.FA_INJECT_BWD, LIMIT_NS)
        t0 = time.perf_counter()
        if which == "fwd":
            fa.fa_fwd(q, k, v, w.causal, w.scale)
        else:
            fa.fa_bwd(q, k, v, o, do, lse, w.causal, w.scale)
        torch.cuda.synchronize()  # the kernel returns: no CUDA error, no hang
        elapsed = time.perf_counter() - t0
    finally:
        fa.fa_test_inject_timeout(fa.FA_INJECT_OFF, 0)
        fa.fa_set_bwd_dq_mode(fa.FA_BWD_DQ_AUTO)
    # it gave up after the short limit, long before the default of 4 s
    assert elapsed < 1.0, elapsed
    assert fa.fa_get_last_device_status() == fa.FA_ERR_DEVICE_TIMEOUT
    assert fa.fa_get_last_device_status() == fa.FA_OK  # reading clears the word
    _parity_after(w, x, dev)


def test_inject_rejects_unknown_kernel():
    with pytest.raises(fa.FAError):
        fa.fa_test_inject_timeout(7, LIMIT_NS)
