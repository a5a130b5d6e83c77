"""Named attention workloads and their seeded synthetic inputs.

This module only draws numbers: it holds none of the attention arithmetic, so both
the CUDA path and the fp64 CPU oracle can take their inputs from it without sharing
any of the method's code.

Recipe (identical on every machine, since numpy's PCG64 stream and its ziggurat
normal sampler are platform independent):

  1. ``rng = numpy.random.default_rng(seed)``.
  2. Draw Q, K, V, dO in that order, each ``[B, H, N, d]`` float32 i.i.d. N(0, 1).
  3. Multiply Q and K by ``qk_gain`` (2 for the peaky long-context workload).
  4. For bf16 workloads, round every value to the nearest bfloat16 (ties to even);
     the arrays stay float32 but hold bf16-representable values, so the GPU sees the
     same numbers after a lossless cast and the oracle widens them to float64.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str          # "bf16" or "fp32"
    causal: bool
    qk_gain: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def shape(self) -> tuple[int, int, int, int]:
        return (self.B, self.H, self.N, self.d)

    def fwd_flop(self) -> float:
        """Forward FLOPs by the convention 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def bwd_flop(self) -> float:
        """Backward FLOPs: 2.5 x the forward count."""
        return 2.5 * self.fwd_flop()

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads: a tiny fp32 exact check and four bf16 shapes.
WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("b1h1_n128_d64_fp32", 1, 1, 128, 64, "fp32", False),
        Workload("b4h16_n2048_d64_bf16", 4, 16, 2048, 64, "bf16", False),
        Workload("b2h16_n8192_d128_bf16_causal", 2, 16, 8192, 128, "bf16", True),
        Workload("b1h8_n32768_d128_bf16_causal_qk2", 1, 8, 32768, 128, "bf16", True, qk_gain=2.0),
        Workload("b16h32_n1024_d128_bf16", 16, 32, 1024, 128, "bf16", False),
    ]
}

HEADLINE = "b2h16_n8192_d128_bf16_causal"


def quantize_e4m3(x: np.ndarray) -> tuple[np.ndarray, float]:
    """Encode float32 values as e4m3 bytes with one factor for the whole array.

    The factor is amax / 448, so the largest magnitude maps to e4m3's largest finite
    value; each x / factor is rounded to the nearest e4m3 value (ties to even) by
    PyTorch's float8_e4m3fn conversion. Returns (uint8 bytes, factor): the value of byte
    b is factor * e4m3(b). This only encodes inputs; both the CUDA path and the oracle
    read the same bytes.
    """
    import torch
    x = np.ascontiguousarray(x, dtype=np.float32)
    amax = float(np.abs(x).max()) if x.size else 0.0
    factor = amax / 448.0 if amax > 0 else 1.0
    t = torch.from_numpy(x / np.float32(factor)).clamp_(-448.0, 448.0)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy(), factor


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int, qk_gain: float = 1.0):
    """Q, K, V drawn as in the recipe above (N(0, 1) float32, Q and K times qk_gain),
    then each encoded by ``quantize_e4m3``: returns ((q8, k8, v8), (q, k, v factors))."""
    rng = np.random.default_rng(seed)
    xs = [rng.standard_normal((B, H, N, d), dtype=np.float32) for _ in range(3)]
    xs[0] *= np.float32(qk_gain)
    xs[1] *= np.float32(qk_gain)
    enc = [quantize_e4m3(x) for x in xs]
    return tuple(e[0] for e in enc), tuple(e[1] for e in enc)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    # NaN/inf are never produced by the normal draws; keep them untouched anyway.
    bad = ~np.isfinite(x)
    if bad.any():
        out = out.copy()
        out[bad] = x[bad]
    return out


def make_inputs(w: Workload) -> dict[str, np.ndarray]:
    """Q, K, V, dO for workload ``w`` as float32 arrays of shape [B, H, N, d]."""
    rng = np.random.default_rng(w.seed)
    out = {}
    for name in ("q", "k", "v", "do"):
        a = rng.standard_normal(w.shape, dtype=np.float32)
        if name in ("q", "k") and w.qk_gain != 1.0:
            a *= np.float32(w.qk_gain)
        if w.dtype == "bf16":
            a = round_to_bf16(a)
        out[name] = a
    return out
