"""fp64 CPU oracle for the FP8 (e4m3) forward.

TEST INFRASTRUCTURE, like ``oracle.attention``: only the test-suite, ``__graft_entry__``'s
smoke check and the benchmark's CPU legs may import it; it shares no code with the CUDA
path.

What the FP8 forward computes. The pages name FP8 as FlashAttention-3's low-precision
format ("flash-attention" (data.6616ai.com), 参考答案; "知识点13 FlashAttention深度攻略",
前沿研究方向) without fixing an encoding or a scaling rule. Reading taken: the inputs are
OCP FP8 E4M3 bytes (the format FlashAttention-3 uses) with one dequantisation factor per
tensor, and the result is the exact attention of the dequantised values:

    Q = q_descale * e4m3(q8),  K = k_descale * e4m3(k8),  V = v_descale * e4m3(v8),
    O, LSE = attention(Q, K, V)   (``oracle.attention.head_forward``).

The kernel's one approximation, rounding the attention weights to e4m3 before they
multiply V, is not part of this definition; the tests bound it separately.

E4M3 (OCP 8-bit floating point, E4M3 variant): bit 7 sign, bits 6-3 exponent field E
(bias 7), bits 2-0 mantissa M. E = 0: subnormal, value (M / 8) * 2^-6. Otherwise
(1 + M / 8) * 2^(E - 7). There are no infinities; S.1111.111 encodes NaN, so the
largest finite magnitude is 1.75 * 2^8 = 448.

Pins: tests/test_oracle_fp8.py (closed-form codes from the format, every code against
PyTorch's float8_e4m3fn conversion, monotonicity, and attention closed forms).
"""
from __future__ import annotations

import numpy as np

from . import attention


def e4m3_to_float64(b) -> np.ndarray:
    """Decode E4M3 bytes (any integer array of values 0..255) to float64."""
    b = np.asarray(b).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    subnormal = (m / 8.0) * 2.0 ** -6
    v = sign * np.where(e == 0, subnormal, normal)
    return np.where((b & 0x7F) == 0x7F, np.nan, v)


def dequantize(b, descale: float) -> np.ndarray:
    """descale * e4m3(b) in float64."""
    return float(descale) * e4m3_to_float64(b)


def head_forward_fp8(q8, k8, v8, descale, scale, causal, rows=None):
    """O and LSE of one head of e4m3 inputs ([N, d] bytes each) and their factors
    ``descale = (q, k, v)``: the exact attention of the dequantised values."""
    qd, kd, vd = descale
    return attention.head_forward(dequantize(q8, qd), dequantize(k8, kd), dequantize(v8, vd), scale, causal,
                                  rows=rows)
