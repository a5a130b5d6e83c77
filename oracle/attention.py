"""fp64 CPU oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE. Only the test-suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this module. The attention library never
calls it, and it shares no code with the CUDA path: it takes plain arrays and
computes the textbook definitions in float64 with numpy.

Sources (web pages on FlashAttention, cited by title and section):
  [BWD]  aiqz.cc "flash-attention-backpropagation": sections 显存困境 (P =
         softmax(QK^T/sqrt(d))), 前向台账 (row max m_i, row sum l_i), 反向总览
         (P_hat = exp(s - m)/l; dQ = dS K/sqrt(d), dK = dS^T Q/sqrt(d), dV = P^T dO),
         Softmax梯度 (D_i = sum_c dO_ic O_ic, dP = dO V^T, dS = P (dP - D)).
  [FA2]  aiqz.cc "flash-attention-v2-sram-tiling": section 1 (Attention =
         softmax(QK^T/sqrt(d)) V).
  [KP13] blog.xiaohack.org "知识点13 FlashAttention深度攻略": 代码手撕 section
         (causal mask: key j is hidden from query i when j > i).

Readings where the pages leave a choice open:
  * ``scale`` is an argument; the pages always use 1/sqrt(d). dQ and dK are
    multiplied by ``scale`` (the factor the pages write as 1/sqrt(d)).
  * The saved statistic is LSE_i = m_i + ln(l_i) (natural log, scaled scores),
    which packs the pages' two ledger rows (m, l) into one.
  * D_i uses the oracle's own float64 O.
  * An additive mask M (optional; [N_q, N_k] per head, finite or -inf) is added to the
    scaled scores, s_ij = scale * q_i . k_j + M_ij, before the causal rule applies; it is
    the "mask" that "知识点13" section 7 (算子融合优化) fuses into the softmax step. A row
    whose every key is hidden (all -inf) has no softmax: its weights are taken as 0, so
    O_i = 0, LSE_i = -inf and the row contributes nothing to any gradient.
  * Dropout (optional; "知识点13" section 7 lists it with the mask inside the fused
    softmax step) multiplies each weight by keep_ij * c after the softmax: O = (P o K c) V
    with K a 0/1 keep matrix and c = keep_scale. LSE stays the softmax's. The backward
    follows from L(O): dV = (P o K c)^T dO, dP = (dO V^T) o K c, dS = P o (dP - D) with
    D_i = dO_i . O_i of the dropped O. The keep matrix comes from oracle/philox.py.
  * Causal attention hides key j from query i iff j > i (queries and keys share
    the same positions; the diagonal is always visible, so no row is empty). With
    N_q != N_k (a decode or a prefill against a cache; cross-attention) the queries are
    the last N_q positions: query row i sits at position i + N_k - N_q and hides keys
    j > i + N_k - N_q (bottom-right alignment; the pages only show N_q = N_k). With
    N_q > N_k the first N_q - N_k queries see no key: their rows are wholly hidden and
    take the rule above (O = 0, LSE = -inf, no gradient).

Evaluation order: every quantity is computed from its definition, a whole row of
scores at a time. To bound memory the rows of a head are taken in groups; rows
are independent in every definition above, and the only sums that run across
groups (dK_j and dV_j, sums over query rows i) are accumulated group by group in
float64, which changes nothing but rounding order.

Pins: tests/test_oracle_pins.py checks this module against closed forms,
invariants, brute-force finite differences, a high-precision mpmath evaluation,
PyTorch's CPU float64 scaled_dot_product_attention with autograd, and the
block-wise online-softmax recurrences the pages describe.
"""
from __future__ import annotations

import numpy as np

# Rows per group: keeps one [rows, N] float64 score block near 256 MB at most.
_GROUP_ELEMS = 1 << 25


def _group_rows(N: int) -> int:
    return max(1, min(N, _GROUP_ELEMS // max(N, 1)))


def scores(q, k, scale, causal, rows, mask=None):
    """s_ij = scale * q_i . k_j (+ M_ij) for the query rows ``rows``; hidden keys get -inf.

    [BWD] 显存困境 (S_ij = Q_i.K_j / sqrt(d)); [KP13] 代码手撕 (mask j > i) and section 7
    (the mask fused into the softmax step).
    """
    rows = np.asarray(rows)
    s = scale * (q[rows] @ k.T)
    if mask is not None:
        s = s + np.asarray(mask, np.float64)[rows]
    if causal:
        offset = k.shape[0] - q.shape[0]  # query row i sits at key position i + offset
        j = np.arange(k.shape[0])
        s = np.where(j[None, :] > rows[:, None] + offset, -np.inf, s)
    return s


def softmax_rows(s):
    """Row softmax with the row maximum subtracted first: returns (P, m, l).

    [BWD] 前向台账: m_i = max_j s_ij, l_i = sum_j exp(s_ij - m_i),
    P_ij = exp(s_ij - m_i) / l_i; hidden keys (s = -inf) get P = 0. A row with every key
    hidden has m = -inf, l = 0 and P = 0.
    """
    m = s.max(axis=1)
    m_ref = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_ref[:, None])
    l = e.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        P = np.where(l[:, None] > 0, e / l[:, None], 0.0)
    return P, m, l


def head_forward(q, k, v, scale, causal, rows=None, mask=None, keep=None, keep_scale=1.0):
    """O and LSE of one head for query ``rows`` (default: all rows).

    q, k, v: [N, d] float64; mask: optional [N_q, N_k] additive mask; keep: optional
    [N_q, N_k] 0/1 dropout keep matrix with its scale keep_scale. Returns O
    [len(rows), d] and LSE [len(rows)], where O_i = sum_j P_ij v_j ([FA2] section 1) and
    LSE_i = m_i + ln l_i (-inf for a row with no visible key).
    """
    q, k, v = (np.asarray(a, dtype=np.float64) for a in (q, k, v))
    N = q.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    O = np.empty((rows.size, v.shape[1]))
    LSE = np.empty(rows.size)
    g = _group_rows(k.shape[0])
    for a in range(0, rows.size, g):
        r = rows[a:a + g]
        P, m, l = softmax_rows(scores(q, k, scale, causal, r, mask))
        if keep is not None:
            P = P * (np.asarray(keep, np.float64)[r] * keep_scale)
        O[a:a + g] = P @ v
        with np.errstate(divide="ignore"):
            LSE[a:a + g] = m + np.log(l)
    return O, LSE


def row_dot(do, o):
    """D_i = sum_c dO_ic * O_ic ([BWD] Softmax梯度)."""
    return np.einsum("ic,ic->i", np.asarray(do, np.float64), np.asarray(o, np.float64))


def head_backward(q, k, v, do, scale, causal, return_ds=False, mask=None, keep=None, keep_scale=1.0):
    """All outputs of one head: O, LSE, D, dQ, dK, dV (and dS when asked, small N only).

    [BWD] 反向总览 / Softmax梯度 / QKV梯度:
      dV = P^T dO;  dP = dO V^T;  dS = P * (dP - D);
      dQ = scale * dS K;  dK = scale * dS^T Q.
    """
    q, k, v, do = (np.asarray(a, dtype=np.float64) for a in (q, k, v, do))
    N, d = q.shape
    O, LSE = head_forward(q, k, v, scale, causal, mask=mask, keep=keep, keep_scale=keep_scale)
    D = row_dot(do, O)
    dQ = np.empty_like(q)
    dK = np.zeros_like(k)
    dV = np.zeros_like(v)
    dS_all = np.empty((N, k.shape[0])) if return_ds else None
    g = _group_rows(k.shape[0])  # each row of scores holds one value per key
    for a in range(0, N, g):
        r = np.arange(a, min(N, a + g))
        P, _, _ = softmax_rows(scores(q, k, scale, causal, r, mask))
        Kc = 1.0 if keep is None else np.asarray(keep, np.float64)[r] * keep_scale
        dV += (P * Kc).T @ do[r]
        dP = (do[r] @ v.T) * Kc
        dS = P * (dP - D[r, None])
        dQ[r] = scale * (dS @ k)
        dK += scale * (dS.T @ q[r])
        if return_ds:
            dS_all[r] = dS
    out = dict(o=O, lse=LSE, d=D, dq=dQ, dk=dK, dv=dV)
    if return_ds:
        out["ds"] = dS_all
    return out


def _head_mask(mask, b, h):
    """The [N_q, N_k] slice of a mask broadcastable to [B, H, N_q, N_k] (None stays None)."""
    if mask is None:
        return None
    mask = np.asarray(mask)
    return mask[b if mask.shape[0] > 1 else 0, h if mask.shape[1] > 1 else 0]


def forward(q, k, v, scale, causal, mask=None):
    """Whole-tensor forward over [B, H, N, d] inputs: O [B,H,N,d], LSE [B,H,N].
    mask: optional additive mask of shape [B or 1, H or 1, N, N]."""
    B, H, N, d = q.shape
    O = np.empty((B, H, N, v.shape[-1]))
    LSE = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            O[b, h], LSE[b, h] = head_forward(q[b, h], k[b, h], v[b, h], scale, causal,
                                              mask=_head_mask(mask, b, h))
    return O, LSE


def backward(q, k, v, do, scale, causal, mask=None):
    """Whole-tensor forward + backward over [B, H, N, d] inputs (mask as in ``forward``).

    Returns a dict of float64 arrays: o, lse, d, dq, dk, dv.
    """
    B, H = q.shape[:2]
    res = None
    for b in range(B):
        for h in range(H):
            r = head_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, mask=_head_mask(mask, b, h))
            if res is None:
                res = {n: np.empty((B, H) + a.shape) for n, a in r.items()}
            for n, a in r.items():
                res[n][b, h] = a
    return res
