"""Counter-based random bits for attention dropout: Philox-4x32-10, written from its
published definition (J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel
random numbers: as easy as 1, 2, 3", SC 2011), and the keep decision built on it.

TEST INFRASTRUCTURE, like the rest of ``oracle/``. The CUDA kernels draw the same bits
from their own implementation of the same published generator; the two share no code.

Philox-4x32-10: a 128-bit counter (4 words) and a 64-bit key (2 words). One round maps
(c0, c1, c2, c3) to (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)) with
M0 = 0xD2511F53, M1 = 0xCD9E8D57 (hi/lo: upper/lower 32 bits of the 64-bit product). The
key is bumped by (0x9E3779B9, 0xBB67AE85) between rounds; 10 rounds.

Dropout layout (the reading this project takes; the pages only name dropout as one of the
steps fused into the softmax, "知识点13 FlashAttention深度攻略" section 7):
  * element (i, j) of head h (h = b * H + head within batch b) takes the 8-bit uniform
    u = bits 8*(j % 4)..+7 of word (j % 16) / 4 of Philox(counter = (j // 16, i, h, 0),
    key = (seed & 0xffffffff, seed >> 32)): one generator call serves 16 keys;
  * the key is kept iff u >= t, where t = min(255, round(p * 256)) for the dropout
    probability p; kept weights are scaled by 256 / (256 - t), so every weight keeps its
    expected value exactly for the quantised probability t / 256.
"""
from __future__ import annotations

import numpy as np

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
_MASK = np.uint64(0xFFFFFFFF)


def philox4x32_10(ctr, key) -> np.ndarray:
    """Philox-4x32-10 of counters ``ctr`` [..., 4] and keys ``key`` [..., 2] (uint32-valued
    arrays that broadcast against each other); returns [..., 4] uint32."""
    ctr = np.asarray(ctr, dtype=np.uint64)
    key = np.asarray(key, dtype=np.uint64)
    c0, c1, c2, c3 = (ctr[..., n] for n in range(4))
    k0, k1 = key[..., 0], key[..., 1]
    for r in range(10):
        if r:
            k0 = (k0 + np.uint64(W0)) & _MASK
            k1 = (k1 + np.uint64(W1)) & _MASK
        p0 = np.uint64(M0) * c0          # exact: both factors are below 2^32
        p1 = np.uint64(M1) * c2
        c0, c1, c2, c3 = (p1 >> np.uint64(32)) ^ c1 ^ k0, p1 & _MASK, (p0 >> np.uint64(32)) ^ c3 ^ k1, p0 & _MASK
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def threshold(p: float) -> int:
    """The 8-bit keep threshold of dropout probability p in [0, 1)."""
    return int(min(255, int(np.floor(float(p) * 256.0 + 0.5))))


def keep_scale(t: int) -> float:
    """Scale of a kept weight: 256 / (256 - t)."""
    return 256.0 / (256.0 - t)


def uniforms(seed: int, head: int, rows, ncols: int) -> np.ndarray:
    """The 8-bit uniforms u of the query rows ``rows`` against keys 0..ncols-1 of one head."""
    rows = np.asarray(rows, dtype=np.uint64)
    nblk = (ncols + 15) // 16
    ctr = np.zeros((rows.size, nblk, 4), dtype=np.uint64)
    ctr[..., 0] = np.arange(nblk, dtype=np.uint64)[None, :]
    ctr[..., 1] = rows[:, None]
    ctr[..., 2] = np.uint64(head)
    key = np.array([seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF], dtype=np.uint64)
    words = philox4x32_10(ctr, key).astype(np.uint32)                  # [rows, nblk, 4]
    octets = np.stack([(words >> (8 * b)) & 0xFF for b in range(4)], axis=-1)  # [rows, nblk, 4, 4]
    return octets.reshape(rows.size, nblk * 16)[:, :ncols].astype(np.uint32)


def keep_matrix(seed: int, head: int, n_rows: int, n_cols: int, p: float) -> np.ndarray:
    """Boolean [n_rows, n_cols] keep decisions of one head for dropout probability p."""
    return uniforms(seed, head, np.arange(n_rows), n_cols) >= threshold(p)
