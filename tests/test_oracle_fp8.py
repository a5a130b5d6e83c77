"""Pins for the FP8 (e4m3) oracle, oracle/fp8.py: checks against things other than itself.

- Codes whose values the E4M3 layout fixes in closed form (1.0, 448, the smallest
  subnormal, NaN, ...).
- Every one of the 256 codes against PyTorch's float8_e4m3fn -> float64 conversion (a
  library routine).
- Invariants: positive codes decode in increasing order; negative codes mirror them.
- Attention closed forms and invariants on dequantised inputs: all-zero Q gives uniform
  weights (O = mean of V, LSE = ln #visible); moving a factor from the scale into Q's
  factor changes nothing; O is linear in V's factor; a tiny head by explicit loops.
- Planted mistakes in copies of the module, each caught by at least one pin.
"""
import math
import types

import numpy as np
import pytest

from oracle import fp8 as oracle_fp8


def pin_format_codes(mod):
    dec = lambda c: float(mod.e4m3_to_float64(np.array([c]))[0])  # noqa: E731
    expect = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x30: 0.5, 0x7E: 448.0, 0xFE: -448.0,
              0x78: 256.0, 0x77: 240.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
              0xB8: -1.0, 0x81: -(2.0 ** -9)}
    for c, v in expect.items():
        assert dec(c) == v, (hex(c), dec(c), v)
    assert math.copysign(1.0, dec(0x80)) == -1.0 and dec(0x80) == 0.0
    assert math.isnan(dec(0x7F)) and math.isnan(dec(0xFF))


def pin_torch_conversion(mod):
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mod.e4m3_to_float64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def pin_monotone(mod):
    pos = mod.e4m3_to_float64(np.arange(0, 127))
    neg = mod.e4m3_to_float64(np.arange(128, 255))
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(neg, -pos)


def _codes(shape, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=shape)
    return np.where((c & 0x7F) == 0x7F, 0x38, c).astype(np.uint8)  # no NaN codes


def pin_uniform_attention(mod):
    N, d = 9, 4
    q8 = np.zeros((N, d), np.uint8)
    k8, v8 = _codes((N, d), 1), _codes((N, d), 2)
    vd = 0.25
    V = vd * mod.e4m3_to_float64(v8)
    for causal in (False, True):
        O, L = mod.head_forward_fp8(q8, k8, v8, (0.5, 0.125, vd), 0.3, causal)
        for i in range(N):
            n = i + 1 if causal else N
            assert np.allclose(O[i], V[:n].mean(axis=0), rtol=0, atol=1e-12)
            assert abs(L[i] - math.log(n)) < 1e-12


def pin_factor_invariances(mod):
    N, d = 7, 5
    q8, k8, v8 = _codes((N, d), 3), _codes((N, d), 4), _codes((N, d), 5)
    O, L = mod.head_forward_fp8(q8, k8, v8, (0.01, 0.02, 0.03), 0.4, True)
    O2, L2 = mod.head_forward_fp8(q8, k8, v8, (0.01 * 4, 0.02, 0.03), 0.4 / 4, True)
    assert np.allclose(O, O2, rtol=1e-12, atol=1e-14) and np.allclose(L, L2, rtol=1e-12, atol=1e-12)
    O3, L3 = mod.head_forward_fp8(q8, k8, v8, (0.01, 0.02, 0.03 * 3), 0.4, True)
    assert np.allclose(O3, 3 * O, rtol=1e-12, atol=1e-14) and np.allclose(L3, L, rtol=1e-12, atol=1e-12)


def pin_tiny_head_by_loops(mod):
    """N = 3, d = 2, non-causal, written out with Python loops on decoded floats."""
    q8 = np.array([[0x38, 0xC0], [0x30, 0x44], [0x00, 0x3C]], np.uint8)   # 1,-2 | .5,3 | 0,1.5
    k8 = np.array([[0x40, 0x38], [0xB8, 0x30], [0x3C, 0x00]], np.uint8)   # 2,1 | -1,.5 | 1.5,0
    v8 = np.array([[0x38, 0x00], [0x00, 0x40], [0xB0, 0x3C]], np.uint8)   # 1,0 | 0,2 | -.5,1.5
    qv = [[1, -2], [0.5, 3], [0, 1.5]]
    kv = [[2, 1], [-1, 0.5], [1.5, 0]]
    vv = [[1, 0], [0, 2], [-0.5, 1.5]]
    qd, kd, vd, scale = 0.5, 2.0, 0.25, 0.7
    O, L = mod.head_forward_fp8(q8, k8, v8, (qd, kd, vd), scale, False)
    for i in range(3):
        s = [scale * sum(qd * qv[i][c] * kd * kv[j][c] for c in range(2)) for j in range(3)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        tot = sum(e)
        for c in range(2):
            want = sum(e[j] / tot * vd * vv[j][c] for j in range(3))
            assert abs(O[i, c] - want) < 1e-12, (i, c)
        assert abs(L[i] - (mx + math.log(tot))) < 1e-12


PINS = [pin_format_codes, pin_torch_conversion, pin_monotone, pin_uniform_attention, pin_factor_invariances,
        pin_tiny_head_by_loops]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle_fp8)


MUTATIONS = [
    ("exponent bias 8", "np.exp2(e.astype(np.float64) - 7.0)", "np.exp2(e.astype(np.float64) - 8.0)"),
    ("subnormal scale 2^-7", "subnormal = (m / 8.0) * 2.0 ** -6", "subnormal = (m / 8.0) * 2.0 ** -7"),
    ("no implicit leading one", "normal = (1.0 + m / 8.0)", "normal = (m / 8.0)"),
    ("mantissa over 16", "normal = (1.0 + m / 8.0)", "normal = (1.0 + m / 16.0)"),
    ("sign ignored", "sign = np.where(b & 0x80, -1.0, 1.0)", "sign = 1.0"),
    ("NaN code not recognised", "(b & 0x7F) == 0x7F", "(b & 0x7F) == 0x100"),
    ("V dequantised with K's factor", "dequantize(v8, vd)", "dequantize(v8, kd)"),
    ("Q's factor dropped", "dequantize(q8, qd)", "dequantize(q8, 1.0)"),
]


def _mutant(old, new):
    src = open(oracle_fp8.__file__).read()
    assert old in src, old
    mod = types.ModuleType("oracle_fp8_mutant")
    mod.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), "oracle_fp8_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(mut):
    mod = _mutant(mut[1], mut[2])
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, FloatingPointError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught: {mut[0]}"
