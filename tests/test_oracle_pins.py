"""Pins for the fp64 oracle: it is checked against things other than itself.

Each ``pin_*`` function takes an oracle module and raises AssertionError when the
module disagrees with a closed form, an invariant, a brute-force evaluation or a
library routine. ``test_pins_hold`` runs every pin on the real oracle;
``test_planted_mistakes_are_caught`` plants plausible mistakes in copies of the
oracle's source and checks that some pin fails for each one.
"""
import json
import math
import os
import types

import numpy as np
import pytest

from oracle import attention as oracle_attention

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _visible_count(N, causal):
    return np.arange(1, N + 1) if causal else np.full(N, N)


# ----------------------------------------------------------------------------- pins
def pin_probability_rows(m):
    """Rows of P sum to one; P is in (0, 1] on visible keys and 0 on hidden ones
    ('flash-attention-backpropagation', 显存困境 and 数值稳定)."""
    for causal in (False, True):
        q, k = _rand((9, 5), 1), _rand((9, 5), 2)
        P, mx, l = m.softmax_rows(m.scores(q, k, 0.4, causal, np.arange(9)))
        assert np.allclose(P.sum(1), 1.0, rtol=0, atol=1e-14)
        vis = np.tril(np.ones((9, 9), bool)) if causal else np.ones((9, 9), bool)
        assert (P[vis] > 0).all() and (P[vis] <= 1).all()
        assert (P[~vis] == 0).all()


def pin_zero_query_uniform(m):
    """Q = 0 makes every visible score 0: P is uniform, O_i is the mean of the
    visible V rows (the prefix mean when causal) and LSE_i = ln(#visible)."""
    N, d = 11, 6
    v = _rand((N, d), 3)
    k = _rand((N, d), 4)
    for causal in (False, True):
        O, LSE = m.head_forward(np.zeros((N, d)), k, v, 0.7, causal)
        cnt = _visible_count(N, causal)
        mean = np.cumsum(v, 0) / cnt[:, None] if causal else np.broadcast_to(v.mean(0), v.shape)
        assert np.allclose(O, mean, rtol=0, atol=1e-13)
        assert np.allclose(LSE, np.log(cnt), rtol=0, atol=1e-13)


def pin_single_key(m):
    """N = 1: O = V_0, LSE = scale q.k, dQ = dK = 0, dV = dO."""
    q, k, v, do = (_rand((1, 7), s) for s in (5, 6, 7, 8))
    for causal in (False, True):
        r = m.head_backward(q, k, v, do, 0.3, causal)
        assert np.allclose(r["o"], v, atol=1e-15)
        assert np.allclose(r["lse"], 0.3 * (q @ k.T).ravel(), atol=1e-14)
        assert np.abs(r["dq"]).max() < 1e-15 and np.abs(r["dk"]).max() < 1e-15
        assert np.allclose(r["dv"], do, atol=1e-15)


def pin_constant_values(m):
    """Identical V rows: O equals that row whatever P is, so dQ = dK = 0."""
    N, d = 8, 5
    q, k, do = _rand((N, d), 9), _rand((N, d), 10), _rand((N, d), 11)
    v = np.tile(_rand((1, d), 12), (N, 1))
    for causal in (False, True):
        r = m.head_backward(q, k, v, do, 0.5, causal)
        assert np.allclose(r["o"], v, atol=1e-14)
        assert np.abs(r["dq"]).max() < 1e-13 and np.abs(r["dk"]).max() < 1e-13


def pin_key_shift(m):
    """Adding c to every K row adds scale q_i.c to row i's scores: O is unchanged and
    LSE_i moves by exactly scale q_i.c."""
    N, d = 10, 4
    q, k, v = _rand((N, d), 13), _rand((N, d), 14), _rand((N, d), 15)
    c = _rand((d,), 16)
    for causal in (False, True):
        O0, L0 = m.head_forward(q, k, v, 0.6, causal)
        O1, L1 = m.head_forward(q, k + c, v, 0.6, causal)
        assert np.allclose(O0, O1, atol=1e-13)
        assert np.allclose(L1 - L0, 0.6 * q @ c, atol=1e-13)


def pin_gradient_sums(m):
    """sum_j dS_ij = 0 for every row (the D term removes the softmax's common-mode
    gradient, 'flash-attention-backpropagation' Softmax梯度); hence sum_j dK_j = 0."""
    N, d = 12, 6
    q, k, v, do = (_rand((N, d), s) for s in (17, 18, 19, 20))
    for causal in (False, True):
        r = m.head_backward(q, k, v, do, 0.45, causal, return_ds=True)
        assert np.abs(r["ds"].sum(1)).max() < 1e-13
        assert np.abs(r["dk"].sum(0)).max() < 1e-13


def pin_dv_brute_force(m):
    """dV_j = sum_i P_ij dO_i, with P built by pure-Python loops from the definition."""
    N, d, scale = 5, 3, 0.8
    q, k, v, do = (_rand((N, d), s) for s in (21, 22, 23, 24))
    for causal in (False, True):
        P = [[0.0] * N for _ in range(N)]
        for i in range(N):
            vis = [j for j in range(N) if not (causal and j > i)]
            s = {j: scale * sum(q[i][c] * k[j][c] for c in range(d)) for j in vis}
            mx = max(s.values())
            z = sum(math.exp(s[j] - mx) for j in vis)
            for j in vis:
                P[i][j] = math.exp(s[j] - mx) / z
        dv = [[sum(P[i][j] * do[i][c] for i in range(N)) for c in range(d)] for j in range(N)]
        o = [[sum(P[i][j] * v[j][c] for j in range(N)) for c in range(d)] for i in range(N)]
        r = m.head_backward(q, k, v, do, scale, causal)
        assert np.allclose(r["dv"], dv, atol=1e-14)
        assert np.allclose(r["o"], o, atol=1e-14)


def _loss(m, q, k, v, do, scale, causal):
    O, _ = m.head_forward(q, k, v, scale, causal)
    return float((O * do).sum())


def pin_finite_differences(m):
    """Central differences of L = <O, dO> with respect to every element of Q, K and V
    match dQ, dK and dV (brute force, N <= 16)."""
    h = 1e-5
    for N, d, causal, seed in ((1, 3, False, 0), (5, 4, False, 1), (7, 4, True, 2), (16, 4, True, 3),
                               (16, 3, False, 4)):
        q, k, v, do = (_rand((N, d), 100 * seed + s) for s in range(4))
        scale = 1.0 / math.sqrt(d)
        r = m.head_backward(q, k, v, do, scale, causal)
        for name, x in (("dq", q), ("dk", k), ("dv", v)):
            g = np.empty_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args = {"dq": (0,), "dk": (1,), "dv": (2,)}[name][0]
                ap = [q, k, v]
                am = [q, k, v]
                ap[args], am[args] = xp, xm
                g[idx] = (_loss(m, *ap, do, scale, causal) - _loss(m, *am, do, scale, causal)) / (2 * h)
            err = np.abs(g - r[name]).max() / max(1e-300, np.abs(g).max())
            assert err < 1e-7, (name, N, causal, err)


def pin_mpmath_gradients(m):
    """A 40-digit mpmath evaluation of the forward definition, differentiated by central
    differences with step 1e-15, agrees with the oracle's O, LSE and gradients."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    N, d, scale = 4, 3, 0.55
    q, k, v, do = (_rand((N, d), 40 + s) for s in range(4))

    def fwd(Q, K, V, causal):
        O, L = [], []
        for i in range(N):
            vis = [j for j in range(N) if not (causal and j > i)]
            s = [scale * mp.fsum(Q[i][c] * K[j][c] for c in range(d)) for j in vis]
            z = mp.fsum(mp.exp(x) for x in s)
            O.append([mp.fsum(mp.exp(s[a]) / z * V[j][c] for a, j in enumerate(vis)) for c in range(d)])
            L.append(mp.log(z))
        return O, L

    def loss(Q, K, V, causal):
        O, _ = fwd(Q, K, V, causal)
        return mp.fsum(O[i][c] * mp.mpf(do[i][c]) for i in range(N) for c in range(d))

    h = mp.mpf("1e-15")
    for causal in (False, True):
        X = [[[mp.mpf(float(a[i][c])) for c in range(d)] for i in range(N)] for a in (q, k, v)]
        r = m.head_backward(q, k, v, do, scale, causal)
        O, L = fwd(*X, causal)
        assert np.allclose(r["o"], np.array(O, dtype=float), rtol=0, atol=1e-14)
        assert np.allclose(r["lse"], np.array(L, dtype=float), rtol=0, atol=1e-14)
        for which, name in enumerate(("dq", "dk", "dv")):
            g = np.empty((N, d))
            for i in range(N):
                for c in range(d):
                    Xp = [[row[:] for row in M] for M in X]
                    Xm = [[row[:] for row in M] for M in X]
                    Xp[which][i][c] += h
                    Xm[which][i][c] -= h
                    g[i, c] = float((loss(*Xp, causal) - loss(*Xm, causal)) / (2 * h))
            assert np.allclose(r[name], g, rtol=0, atol=1e-12), (name, causal)


def pin_torch_sdpa(m):
    """PyTorch's CPU float64 scaled_dot_product_attention and autograd agree."""
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 3, 37, 8
    arrs = [_rand((B, H, N, d), 60 + s) for s in range(4)]
    for causal in (False, True):
        t = [torch.tensor(a, dtype=torch.float64, requires_grad=(i < 3)) for i, a in enumerate(arrs)]
        o = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], is_causal=causal, scale=0.3)
        (o * t[3]).sum().backward()
        r = m.backward(*arrs, 0.3, causal)
        assert np.allclose(r["o"], o.detach().numpy(), rtol=0, atol=1e-12)
        for name, ten in zip(("dq", "dk", "dv"), t[:3]):
            assert np.allclose(r[name], ten.grad.numpy(), rtol=0, atol=1e-12), name
        s = 0.3 * torch.matmul(t[0], t[1].transpose(-1, -2)).detach()
        if causal:
            s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
        assert np.allclose(r["lse"], torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


# -- the pages' block-wise recurrences, restated independently -----------------------
def _blockwise_forward(q, k, v, scale, causal, block):
    """Tiled forward with the online softmax: per block, the local max and local exp-sum
    are merged into the running (m, l) as l_new = l e^{m - m_new} + l_loc e^{m_loc - m_new}
    ('知识点13', section 4), and the un-normalised output is rescaled by e^{m - m_new}
    and divided by l at the end ('flash-attention-backpropagation', Python 演示)."""
    N, d = q.shape
    O = np.zeros((N, v.shape[1]))
    mrun = np.full(N, -np.inf)
    lrun = np.zeros(N)
    for j0 in range(0, N, block):
        kb, vb = k[j0:j0 + block], v[j0:j0 + block]
        for i0 in range(0, N, block):
            if causal and j0 > i0 + block - 1:
                continue
            s = scale * q[i0:i0 + block] @ kb.T
            if causal:
                ii = np.arange(i0, min(N, i0 + block))[:, None]
                jj = np.arange(j0, min(N, j0 + block))[None, :]
                s = np.where(jj > ii, -np.inf, s)
            mloc = s.max(1)
            e = np.exp(s - mloc[:, None])
            e[~np.isfinite(s)] = 0.0
            lloc = e.sum(1)
            mo = mrun[i0:i0 + block]
            mn = np.maximum(mo, mloc)
            a = np.where(np.isfinite(mo), np.exp(mo - mn), 0.0)
            b = np.where(np.isfinite(mloc), np.exp(mloc - mn), 0.0)
            lrun[i0:i0 + block] = lrun[i0:i0 + block] * a + lloc * b
            O[i0:i0 + block] = O[i0:i0 + block] * a[:, None] + (e * b[:, None]) @ vb
            mrun[i0:i0 + block] = mn
    return O / lrun[:, None], mrun + np.log(lrun)


def _blockwise_backward(q, k, v, do, scale, causal, block):
    """Outer loop over key/value blocks, inner loop over query blocks; P is rebuilt from
    the forward's statistics and dV, dQ, dK are accumulated block by block
    ('flash-attention-backpropagation', QKV梯度)."""
    N = q.shape[0]
    O, lse = _blockwise_forward(q, k, v, scale, causal, block)
    D = (do * O).sum(1)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for j0 in range(0, N, block):
        for i0 in range(0, N, block):
            s = scale * q[i0:i0 + block] @ k[j0:j0 + block].T
            p = np.exp(s - lse[i0:i0 + block, None])
            if causal:
                ii = np.arange(i0, min(N, i0 + block))[:, None]
                jj = np.arange(j0, min(N, j0 + block))[None, :]
                p = np.where(jj > ii, 0.0, p)
            dv[j0:j0 + block] += p.T @ do[i0:i0 + block]
            dp = do[i0:i0 + block] @ v[j0:j0 + block].T
            ds = p * (dp - D[i0:i0 + block, None])
            dq[i0:i0 + block] += scale * ds @ k[j0:j0 + block]
            dk[j0:j0 + block] += scale * ds.T @ q[i0:i0 + block]
    return O, lse, dq, dk, dv


def pin_worked_examples(m):
    """The pages' worked examples: block-wise equals dense within the page's own bar."""
    ex = GOLDEN["fa2_pure_python_demo"]
    q, k, v = (np.array(ex[n], dtype=np.float64) for n in ("Q", "K", "V"))
    scale = 1 / math.sqrt(ex["d"])
    O, L = m.head_forward(q, k, v, scale, ex["causal"])
    Ob, Lb = _blockwise_forward(q, k, v, scale, ex["causal"], ex["block"])
    assert np.abs(O - Ob).max() < ex["max_abs_diff"]
    assert np.abs(L - Lb).max() < ex["max_abs_diff"]

    ex = GOLDEN["bwd_numpy_demo"]
    rng = np.random.default_rng(0)
    q, k, v, do = (rng.normal(size=(ex["N"], ex["d"])) for _ in range(4))
    scale = 1 / math.sqrt(ex["d"])
    r = m.head_backward(q, k, v, do, scale, ex["causal"])
    _, _, dq, dk, dv = _blockwise_backward(q, k, v, do, scale, ex["causal"], ex["block"])
    for a, b in ((r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
        assert np.abs(a - b).max() < ex["atol"]

    ex = GOLDEN["kp13_causal_equivalence"]
    rng = np.random.default_rng(0)
    shp = (ex["B"], ex["H"], ex["N"], ex["d"])
    q, k, v = (rng.standard_normal(shp, dtype=np.float32).astype(np.float64) for _ in range(3))
    do = rng.standard_normal(shp, dtype=np.float32).astype(np.float64)
    scale = 1 / math.sqrt(ex["d"])
    r = m.backward(q, k, v, do, scale, True)
    for b in range(ex["B"]):
        for h in range(ex["H"]):
            Ob, Lb, dq, dk, dv = _blockwise_backward(q[b, h], k[b, h], v[b, h], do[b, h], scale, True, ex["block"])
            assert np.abs(r["o"][b, h] - Ob).max() < ex["max_abs_diff"]
            # the same recurrences in float64 agree far below the page's float32 bar
            for a, bb in ((r["lse"][b, h], Lb), (r["dq"][b, h], dq), (r["dk"][b, h], dk), (r["dv"][b, h], dv)):
                assert np.abs(a - bb).max() < 1e-11


def pin_blockwise_random(m):
    """Block-wise recurrences equal the dense oracle to 1e-12 on ragged random cases."""
    for N, d, block, causal, seed in ((13, 5, 4, False, 0), (13, 5, 4, True, 1), (33, 8, 8, True, 2)):
        q, k, v, do = (_rand((N, d), 200 + 10 * seed + s) for s in range(4))
        scale = 0.9 / math.sqrt(d)
        r = m.head_backward(q, k, v, do, scale, causal)
        O, L, dq, dk, dv = _blockwise_backward(q, k, v, do, scale, causal, block)
        for a, b in ((r["o"], O), (r["lse"], L), (r["dq"], dq), (r["dk"], dk), (r["dv"], dv)):
            assert np.abs(a - b).max() < 1e-12


def pin_row_sampling(m):
    """Row subsets and row grouping give the same numbers as the whole head."""
    N, d = 40, 4
    q, k, v = (_rand((N, d), 300 + s) for s in range(3))
    for causal in (False, True):
        O, L = m.head_forward(q, k, v, 0.5, causal)
        rows = np.array([0, 7, 39, 20])
        Os, Ls = m.head_forward(q, k, v, 0.5, causal, rows=rows)
        assert np.array_equal(Os, O[rows]) or np.allclose(Os, O[rows], atol=1e-15)
        assert np.allclose(Ls, L[rows], atol=1e-15)


def pin_fewer_queries_than_keys(m):
    """N_q < N_k (bottom-right causal alignment): the N_q queries are the last N_q
    positions, so their outputs equal the last N_q rows of the square problem in which
    the same queries sit at those positions; one query sees every key."""
    Nk, Nq, d = 23, 5, 4
    qf, k, v = (_rand((Nk, d), 500 + s) for s in range(3))
    O_full, L_full = m.head_forward(qf, k, v, 0.5, True)
    O, L = m.head_forward(qf[-Nq:], k, v, 0.5, True)
    assert np.allclose(O, O_full[-Nq:], rtol=0, atol=1e-14)
    assert np.allclose(L, L_full[-Nq:], rtol=0, atol=1e-14)
    O1c, L1c = m.head_forward(qf[-1:], k, v, 0.5, True)
    O1n, L1n = m.head_forward(qf[-1:], k, v, 0.5, False)
    assert np.allclose(O1c, O1n, rtol=0, atol=1e-15) and np.allclose(L1c, L1n, rtol=0, atol=1e-15)
    # query i of the short block sees keys 0 .. i + Nk - Nq: brute force on row 0
    vis = Nk - Nq + 1
    s0 = 0.5 * k[:vis] @ qf[-Nq]
    p0 = np.exp(s0 - s0.max())
    assert np.allclose(O[0], (p0 / p0.sum()) @ v[:vis], rtol=0, atol=1e-14)


def pin_more_queries_than_keys(m):
    """N_q > N_k, causal, bottom-right: query i sits at position i - (N_q - N_k), so the first
    N_q - N_k queries see no key (no softmax: O = 0, LSE = -inf, dQ = 0, no share of dK or
    dV), and the last N_k queries are exactly the square causal problem on those queries."""
    Nq, Nk, d = 9, 4, 3
    q, do = (_rand((Nq, d), 520 + s) for s in range(2))
    k, v = (_rand((Nk, d), 530 + s) for s in range(2))
    r = m.head_backward(q, k, v, do, 0.7, True)
    hid = Nq - Nk
    assert np.array_equal(r["o"][:hid], np.zeros((hid, d))) and np.all(r["lse"][:hid] == -np.inf)
    assert np.array_equal(r["dq"][:hid], np.zeros((hid, d)))
    sq = m.head_backward(q[hid:], k, v, do[hid:], 0.7, True)
    for n in ("o", "lse", "dq"):
        assert np.allclose(r[n][hid:], sq[n], rtol=0, atol=1e-14), n
    for n in ("dk", "dv"):
        assert np.allclose(r[n], sq[n], rtol=0, atol=1e-14), n
    # non-causal: every query sees every key; brute force on each row
    On, Ln = m.head_forward(q, k, v, 0.7, False)
    for i in range(Nq):
        s = [0.7 * sum(q[i, c] * k[j, c] for c in range(d)) for j in range(Nk)]
        mx = max(s)
        w = [np.exp(x - mx) for x in s]
        tot = sum(w)
        assert abs(Ln[i] - (mx + np.log(tot))) < 1e-13
        for c in range(d):
            assert abs(On[i, c] - sum(w[j] * v[j, c] for j in range(Nk)) / tot) < 1e-13


def pin_rectangular_torch_autograd(m):
    """N_q != N_k: outputs and gradients equal PyTorch's CPU float64 attention with
    autograd; causal through an explicit bottom-right mask (N_q <= N_k, so no row is empty)."""
    torch = pytest.importorskip("torch")
    for Nq, Nk, causal in ((5, 11, False), (5, 11, True), (12, 7, False), (1, 6, True)):
        arrs = [_rand((Nq, 4), 540 + Nq), _rand((Nk, 4), 541 + Nk), _rand((Nk, 4), 542 + Nk), _rand((Nq, 4), 543)]
        t = [torch.tensor(a, dtype=torch.float64, requires_grad=(i < 3)) for i, a in enumerate(arrs)]
        mask = None
        if causal:
            mask = torch.arange(Nk)[None, :] <= torch.arange(Nq)[:, None] + (Nk - Nq)
        o = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], attn_mask=mask, scale=0.4)
        (o * t[3]).sum().backward()
        r = m.head_backward(*arrs, 0.4, causal)
        assert np.allclose(r["o"], o.detach().numpy(), rtol=0, atol=1e-12), (Nq, Nk, causal)
        for name, ten in zip(("dq", "dk", "dv"), t[:3]):
            assert np.allclose(r[name], ten.grad.numpy(), rtol=0, atol=1e-12), (Nq, Nk, causal, name)


# -- the additive mask ("知识点13" section 7: the mask fused into the softmax step) ---------
def _mask(N, seed, p_hide=0.2):
    """A random finite mask with about p_hide of its entries -inf; the diagonal stays
    finite, so no row is wholly hidden, causal or not."""
    rng = np.random.default_rng(seed)
    M = rng.standard_normal((N, N)) * 1.5
    hide = rng.random((N, N)) < p_hide
    hide[np.arange(N), np.arange(N)] = False
    return np.where(hide, -np.inf, M)


def pin_mask_zero_and_triangle(m):
    """A zero mask changes nothing; an upper-triangular -inf mask is the causal rule."""
    N, d = 10, 4
    q, k, v, do = (_rand((N, d), 700 + s) for s in range(4))
    ref = m.head_backward(q, k, v, do, 0.5, False)
    zero = m.head_backward(q, k, v, do, 0.5, False, mask=np.zeros((N, N)))
    tri = np.where(np.triu(np.ones((N, N), bool), 1), -np.inf, 0.0)
    caus = m.head_backward(q, k, v, do, 0.5, True)
    by_mask = m.head_backward(q, k, v, do, 0.5, False, mask=tri)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert np.allclose(ref[n], zero[n], rtol=0, atol=1e-14), n
        assert np.allclose(caus[n], by_mask[n], rtol=0, atol=1e-14), n


def pin_mask_brute_force(m):
    """O_i = sum_j w_ij e^{s_ij} v_j / sum_j w_ij e^{s_ij} with M_ij = ln w_ij, by loops."""
    N, d, scale = 5, 3, 0.6
    q, k, v = (_rand((N, d), 710 + s) for s in range(3))
    w = np.random.default_rng(713).random((N, N)) + 0.05
    w[1, 3] = w[4, 0] = 0.0  # -inf entries
    with np.errstate(divide="ignore"):
        M = np.log(w)
    O, L = m.head_forward(q, k, v, scale, False, mask=M)
    for i in range(N):
        num = [0.0] * d
        den = 0.0
        for j in range(N):
            e = w[i, j] * math.exp(scale * sum(q[i, c] * k[j, c] for c in range(d)))
            den += e
            for c in range(d):
                num[c] += e * v[j, c]
        for c in range(d):
            assert abs(O[i, c] - num[c] / den) < 1e-12, (i, c)
        assert abs(L[i] - math.log(den)) < 1e-12


def pin_mask_row_shift(m):
    """Adding c_i to every entry of row i leaves O and the gradients unchanged and moves
    LSE_i by c_i (softmax shift invariance)."""
    N, d = 9, 4
    q, k, v, do = (_rand((N, d), 720 + s) for s in range(4))
    M = _mask(N, 724)
    c = np.linspace(-3, 5, N)
    a = m.head_backward(q, k, v, do, 0.4, True, mask=M)
    b = m.head_backward(q, k, v, do, 0.4, True, mask=M + c[:, None])
    for n in ("o", "dq", "dk", "dv"):
        assert np.allclose(a[n], b[n], rtol=0, atol=1e-12), n
    assert np.allclose(b["lse"] - a["lse"], c, rtol=0, atol=1e-12)


def pin_mask_finite_differences(m):
    """Central differences of <O, dO> with a random finite mask with -inf entries."""
    h = 1e-5
    for N, d, causal, seed in ((6, 3, False, 730), (9, 4, True, 731)):
        q, k, v, do = (_rand((N, d), seed + s) for s in range(4))
        M = _mask(N, seed + 9)
        r = m.head_backward(q, k, v, do, 0.5, causal, mask=M)

        def loss(qq, kk, vv):
            return float((m.head_forward(qq, kk, vv, 0.5, causal, mask=M)[0] * do).sum())
        for pos, name in enumerate(("dq", "dk", "dv")):
            x = [q, k, v][pos]
            g = np.empty_like(x)
            for idx in np.ndindex(*x.shape):
                args_p, args_m = [q, k, v], [q, k, v]
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p[pos], args_m[pos] = xp, xm
                g[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            err = np.abs(g - r[name]).max() / max(1e-300, np.abs(g).max())
            assert err < 1e-7, (name, N, causal, err)


def pin_mask_torch_sdpa(m):
    """PyTorch's CPU float64 scaled_dot_product_attention with an additive float mask."""
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 2, 13, 5
    arrs = [_rand((B, H, N, d), 740 + s) for s in range(4)]
    M = np.stack([np.stack([_mask(N, 750 + 2 * b + h) for h in range(H)]) for b in range(B)])
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=(i < 3)) for i, a in enumerate(arrs)]
    o = torch.nn.functional.scaled_dot_product_attention(t[0], t[1], t[2], attn_mask=torch.tensor(M), scale=0.3)
    (o * t[3]).sum().backward()
    r = m.backward(*arrs, 0.3, False, mask=M)
    assert np.allclose(r["o"], o.detach().numpy(), rtol=0, atol=1e-12)
    for name, ten in zip(("dq", "dk", "dv"), t[:3]):
        assert np.allclose(r[name], ten.grad.numpy(), rtol=0, atol=1e-12), name
    # a mask broadcast over batch and heads
    M1 = M[:1, :1]
    o1 = torch.nn.functional.scaled_dot_product_attention(t[0].detach(), t[1].detach(), t[2].detach(),
                                                          attn_mask=torch.tensor(M1), scale=0.3)
    assert np.allclose(m.forward(*arrs[:3], 0.3, False, mask=M1)[0], o1.numpy(), rtol=0, atol=1e-12)


def pin_boolean_mask_is_key_removal(m):
    """A mask of 0 (visible) and -inf (hidden) entries, the boolean mask the packed-bit
    kernels take: each query's output and LSE equal attention over its visible keys alone,
    and a key's dK and dV collect only the queries that see it."""
    N, d, scale = 8, 3, 0.7
    q, k, v, do = (_rand((N, d), 780 + s) for s in range(4))
    vis = np.random.default_rng(784).random((N, N)) < 0.6
    vis[np.arange(N), (np.arange(N) * 3) % N] = True  # every query sees at least one key
    M = np.where(vis, 0.0, -np.inf)
    r = m.head_backward(q, k, v, do, scale, False, mask=M)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for i in range(N):
        keys = np.flatnonzero(vis[i])
        ri = m.head_backward(q[i:i + 1], k[keys], v[keys], do[i:i + 1], scale, False)
        assert np.allclose(r["o"][i], ri["o"][0], rtol=0, atol=1e-13), i
        assert abs(r["lse"][i] - ri["lse"][0]) < 1e-13, i
        assert np.allclose(r["dq"][i], ri["dq"][0], rtol=0, atol=1e-13), i
        dk[keys] += ri["dk"]
        dv[keys] += ri["dv"]
    assert np.allclose(r["dk"], dk, rtol=0, atol=1e-13)
    assert np.allclose(r["dv"], dv, rtol=0, atol=1e-13)


def pin_mask_hidden_row(m):
    """A row with every key hidden: O = 0, LSE = -inf, no gradient through it, and the
    other rows as without that row's queries."""
    N, d = 7, 3
    q, k, v, do = (_rand((N, d), 760 + s) for s in range(4))
    M = _mask(N, 765)
    M[3] = -np.inf
    r = m.head_backward(q, k, v, do, 0.5, False, mask=M)
    assert np.all(r["o"][3] == 0) and r["lse"][3] == -np.inf and np.all(r["dq"][3] == 0)
    for n in ("o", "dq", "dk", "dv", "lse"):
        assert not np.isnan(r[n]).any(), n
    keep = np.array([i for i in range(N) if i != 3])
    rk = m.head_backward(q[keep], k, v, do[keep], 0.5, False, mask=M[keep])
    assert np.allclose(r["o"][keep], rk["o"], rtol=0, atol=1e-13)
    assert np.allclose(r["dk"], rk["dk"], rtol=0, atol=1e-13)
    assert np.allclose(r["dv"], rk["dv"], rtol=0, atol=1e-13)


# -- dropout ("知识点13" section 7): O = (P o K c) V with a fixed 0/1 keep matrix K -------
def _keep(N, seed, p=0.3):
    return np.random.default_rng(seed).random((N, N)) >= p


def pin_dropout_keep_all(m):
    """Keeping every weight with scale 1 is no dropout."""
    N, d = 8, 3
    q, k, v, do = (_rand((N, d), 800 + s) for s in range(4))
    a = m.head_backward(q, k, v, do, 0.5, True)
    b = m.head_backward(q, k, v, do, 0.5, True, keep=np.ones((N, N), bool), keep_scale=1.0)
    for n in ("o", "lse", "dq", "dk", "dv"):
        assert np.allclose(a[n], b[n], rtol=0, atol=1e-14), n


def pin_dropout_finite_differences(m):
    """Central differences of <O, dO> with the keep matrix held fixed."""
    h = 1e-5
    for N, d, causal, seed in ((6, 3, False, 810), (9, 4, True, 811)):
        q, k, v, do = (_rand((N, d), seed + s) for s in range(4))
        K, c = _keep(N, seed + 9), 1.0 / 0.7
        r = m.head_backward(q, k, v, do, 0.5, causal, keep=K, keep_scale=c)

        def loss(qq, kk, vv):
            return float((m.head_forward(qq, kk, vv, 0.5, causal, keep=K, keep_scale=c)[0] * do).sum())
        for pos, name in enumerate(("dq", "dk", "dv")):
            x = [q, k, v][pos]
            g = np.empty_like(x)
            for idx in np.ndindex(*x.shape):
                ap, am = [q, k, v], [q, k, v]
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                ap[pos], am[pos] = xp, xm
                g[idx] = (loss(*ap) - loss(*am)) / (2 * h)
            err = np.abs(g - r[name]).max() / max(1e-300, np.abs(g).max())
            assert err < 1e-7, (name, N, causal, err)


def pin_dropout_torch_autograd(m):
    """PyTorch float64 autograd of O = (softmax(S) * K * c) V, and LSE of the undropped S."""
    torch = pytest.importorskip("torch")
    N, d, scale = 12, 5, 0.4
    arrs = [_rand((N, d), 820 + s) for s in range(4)]
    K, c = _keep(N, 825), 1.0 / 0.75
    t = [torch.tensor(a, dtype=torch.float64, requires_grad=(i < 3)) for i, a in enumerate(arrs)]
    s = scale * t[0] @ t[1].T
    s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    o = (torch.softmax(s, -1) * torch.tensor(K, dtype=torch.float64) * c) @ t[2]
    (o * t[3]).sum().backward()
    r = m.head_backward(*arrs, scale, True, keep=K, keep_scale=c)
    assert np.allclose(r["o"], o.detach().numpy(), rtol=0, atol=1e-12)
    assert np.allclose(r["lse"], torch.logsumexp(s, -1).detach().numpy(), rtol=0, atol=1e-12)
    for name, ten in zip(("dq", "dk", "dv"), t[:3]):
        assert np.allclose(r[name], ten.grad.numpy(), rtol=0, atol=1e-12), name


PINS = [v for n, v in sorted(globals().items()) if n.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pins_hold(pin):
    pin(oracle_attention)


def test_row_grouping_matches_single_group(monkeypatch):
    """The memory-bounding row groups change nothing beyond rounding."""
    N, d = 50, 4
    q, k, v, do = (_rand((N, d), 400 + s) for s in range(4))
    ref = oracle_attention.head_backward(q, k, v, do, 0.5, True)
    monkeypatch.setattr(oracle_attention, "_GROUP_ELEMS", 7 * N)
    got = oracle_attention.head_backward(q, k, v, do, 0.5, True)
    for n in ref:
        assert np.allclose(ref[n], got[n], rtol=0, atol=1e-13), n


# ----------------------------------------------------------- planted mistakes
MUTATIONS = [
    ("dropped D term in dS", "dS = P * (dP - D[r, None])", "dS = P * dP"),
    ("wrong sign in dS", "dS = P * (dP - D[r, None])", "dS = P * (D[r, None] - dP)"),
    ("scale missing on dK", "dK += scale * (dS.T @ q[r])", "dK += dS.T @ q[r]"),
    ("scale missing on dQ", "dQ[r] = scale * (dS @ k)", "dQ[r] = dS @ k"),
    ("dV uses V instead of dO", "dV += (P * Kc).T @ do[r]", "dV += (P * Kc).T @ v[r]"),
    ("dV without the transpose", "dV += (P * Kc).T @ do[r]", "dV += (P * Kc) @ do[r]"),
    ("dQ uses Q instead of K", "dQ[r] = scale * (dS @ k)", "dQ[r] = scale * (dS @ q)"),
    ("dP uses K instead of V", "dP = (do[r] @ v.T) * Kc", "dP = (do[r] @ k.T) * Kc"),
    ("dropout scale missing in O", "P = P * (np.asarray(keep, np.float64)[r] * keep_scale)",
     "P = P * np.asarray(keep, np.float64)[r]"),
    ("dropout not applied to dP", "dP = (do[r] @ v.T) * Kc", "dP = do[r] @ v.T"),
    ("dropout not applied to dV", "dV += (P * Kc).T @ do[r]", "dV += P.T @ do[r]"),
    ("mask hides diagonal", "j[None, :] > rows[:, None]", "j[None, :] >= rows[:, None]"),
    ("mask keeps the future", "j[None, :] > rows[:, None]", "j[None, :] < rows[:, None]"),
    ("top-left alignment for fewer queries", "offset = k.shape[0] - q.shape[0]", "offset = 0"),
    ("offset with the wrong sign", "offset = k.shape[0] - q.shape[0]", "offset = q.shape[0] - k.shape[0]"),
    ("max not subtracted from LSE", "LSE[a:a + g] = m + np.log(l)", "LSE[a:a + g] = np.log(l)"),
    ("log2 in LSE", "LSE[a:a + g] = m + np.log(l)", "LSE[a:a + g] = m + np.log2(l)"),
    ("D from dO.dO", 'np.einsum("ic,ic->i", np.asarray(do, np.float64), np.asarray(o, np.float64))',
     'np.einsum("ic,ic->i", np.asarray(do, np.float64), np.asarray(do, np.float64))'),
    ("scale missing on scores", "s = scale * (q[rows] @ k.T)", "s = q[rows] @ k.T"),
    ("no normalisation", "P = np.where(l[:, None] > 0, e / l[:, None], 0.0)", "P = np.where(l[:, None] > 0, e, 0.0)"),
    ("mask subtracted", "s = s + np.asarray(mask, np.float64)[rows]", "s = s - np.asarray(mask, np.float64)[rows]"),
    ("mask transposed", "s = s + np.asarray(mask, np.float64)[rows]", "s = s + np.asarray(mask, np.float64).T[rows]"),
    ("mask scaled", "s = s + np.asarray(mask, np.float64)[rows]", "s = s + scale * np.asarray(mask, np.float64)[rows]"),
    ("mask ignored", "s = s + np.asarray(mask, np.float64)[rows]", "s = s + 0.0"),
    ("no guard for a wholly hidden row", "P = np.where(l[:, None] > 0, e / l[:, None], 0.0)", "P = e / l[:, None]"),
]


def _mutant(old, new):
    src = open(oracle_attention.__file__).read()
    assert old in src, old
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("mut", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(mut):
    _, old, new = mut
    mod = _mutant(old, new)
    failed = []
    for pin in PINS:
        if pin is pin_mpmath_gradients:
            continue  # slow; the other pins already cover every mutation
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, FloatingPointError, ValueError, IndexError):  # a crash on a shape counts
            failed.append(pin.__name__)
    assert failed, f"no pin caught: {mut[0]}"
