"""Pins for oracle/philox.py (the dropout bits), checked against things other than itself.

- Philox-4x32-10 against the generator's published known-answer vectors (the Random123
  library's known-answer tests for philox4x32 with 10 rounds, distributed with the paper
  "Parallel random numbers: as easy as 1, 2, 3", SC 2011).
- The keep layout: element (i, j) takes byte j % 4 of word (j % 16) / 4 of the block
  (j // 16, i, head, 0), checked against direct calls of the generator.
- The keep decision's closed forms (p = 0 keeps everything; the threshold of p = 1/2) and
  its statistics (binomial bounds on the kept fraction, the mean of a uniform byte).
- Planted mistakes in copies of the module, each caught.
"""
import math
import types

import numpy as np
import pytest

from oracle import philox

KAT = [  # counter (4 words), key (2 words), output (4 words)
    ((0x00000000, 0x00000000, 0x00000000, 0x00000000), (0x00000000, 0x00000000),
     (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
    ((0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF, 0xFFFFFFFF), (0xFFFFFFFF, 0xFFFFFFFF),
     (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
    ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
     (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)),
]


def pin_known_answers(mod):
    for ctr, key, want in KAT:
        got = mod.philox4x32_10(np.array(ctr, np.uint64), np.array(key, np.uint64))
        assert tuple(int(x) for x in got) == want, ([hex(int(x)) for x in got], [hex(x) for x in want])


def pin_layout(mod):
    seed, head = 0x1234_5678_9ABC_DEF0, 5
    u = mod.uniforms(seed, head, [0, 3, 77], 37)
    key = np.array([seed & 0xFFFFFFFF, seed >> 32], np.uint64)
    for a, i in enumerate((0, 3, 77)):
        for j in range(37):
            w = mod.philox4x32_10(np.array([j // 16, i, head, 0], np.uint64), key)
            octet = (int(w[(j % 16) // 4]) >> (8 * (j % 4))) & 0xFF
            assert u[a, j] == octet, (i, j)


def pin_keep_rule(mod):
    assert mod.threshold(0.0) == 0 and mod.threshold(0.5) == 128 and mod.threshold(0.9999999) == 255
    assert mod.threshold(0.1) == 26   # round(25.6)
    assert mod.keep_scale(0) == 1.0 and mod.keep_scale(128) == 2.0 and mod.keep_scale(192) == 4.0
    assert mod.keep_matrix(7, 0, 16, 40, 0.0).all()
    n_rows, n_cols, p = 256, 2048, 0.25
    K = mod.keep_matrix(99, 3, n_rows, n_cols, p)
    n = K.size
    keep_p = 1 - mod.threshold(p) / 256
    assert abs(K.mean() - keep_p) < 5 * math.sqrt(keep_p * (1 - keep_p) / n)
    u = mod.uniforms(99, 3, np.arange(64), 512).astype(np.float64)
    assert u.max() <= 255 and abs(u.mean() - 127.5) < 5 * 73.9 / math.sqrt(u.size)   # uniform on 0..255
    assert not np.array_equal(K, mod.keep_matrix(99, 4, n_rows, n_cols, p))   # another head
    assert not np.array_equal(K, mod.keep_matrix(100, 3, n_rows, n_cols, p))  # another seed


PINS = [pin_known_answers, pin_layout, pin_keep_rule]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(philox)


MUTATIONS = [
    ("wrong multiplier", "M0, M1 = 0xD2511F53, 0xCD9E8D57", "M0, M1 = 0xD2511F53, 0xCD9E8D55"),
    ("no key bump", "k0 = (k0 + np.uint64(W0)) & _MASK", "k0 = k0"),
    ("hi and lo swapped",
     "c0, c1, c2, c3 = (p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & _MASK, (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & _MASK",
     "c0, c1, c2, c3 = (p1 & _MASK) ^ c1 ^ k0, p1 >> np.uint64(32), (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & _MASK"),
    ("bytes in the wrong order", "np.stack([(words >> (8 * b)) & 0xFF for b in range(4)], axis=-1)",
     "np.stack([(words >> (8 * b)) & 0xFF for b in range(3, -1, -1)], axis=-1)"),
    ("row and head swapped in the counter", "ctr[..., 1] = rows[:, None]\n    ctr[..., 2] = np.uint64(head)",
     "ctr[..., 2] = rows[:, None]\n    ctr[..., 1] = np.uint64(head)"),
]


def _mutant(old, new):
    src = open(philox.__file__).read()
    assert old in src, old
    mod = types.ModuleType("philox_mutant")
    exec(compile(src.replace(old, new), "philox_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(mut):
    mod = _mutant(mut[1], mut[2])
    failed = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught: {mut[0]}"
