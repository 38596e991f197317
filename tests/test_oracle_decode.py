"""Pins of oracle.decode_bwd (the decode-style backward from saved
probabilities; rullama training.rs, attention_backward_dq_chained /
attention_backward_dkv_chained) against things other than itself:

- the explicit-matrix backward oracle.bwd for the last row of a causal
  sequence whose other rows carry no gradient (dO = 0 there);
- central finite differences of f = sum_h d_out_h . O_h, O_h = sum_j
  softmax_j(sigma q_h . k_j) v_j, in q, k_hist, v_hist and in the scores;
- sum_j d_scores_hj = 0 when probs sum to one; history_len = 1 in closed form;
- GQA = the group sum of multi-head attention with K, V repeated per head.
"""
import math

import numpy as np
import pytest

import oracle


def _softmax_rows(s):
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def _probs(q, K, H, Hk, d, scale):
    G = H // Hk
    L = K.shape[0]
    s = np.zeros((H, L))
    for h in range(H):
        g = h // G
        s[h] = scale * K[:, g * d:(g + 1) * d] @ q[h * d:(h + 1) * d]
    return _softmax_rows(s), s


def _f(q, K, V, dout, H, Hk, d, scale):
    P, _ = _probs(q, K, H, Hk, d, scale)
    G = H // Hk
    tot = 0.0
    for h in range(H):
        g = h // G
        tot += dout[h * d:(h + 1) * d] @ (P[h] @ V[:, g * d:(g + 1) * d])
    return tot


def _case(rng, L, H, Hk, d):
    q = rng.standard_normal(H * d)
    K = rng.standard_normal((L, Hk * d))
    V = rng.standard_normal((L, Hk * d))
    dout = rng.standard_normal(H * d)
    return q, K, V, dout


@pytest.mark.parametrize("L,H,Hk,d", [(7, 4, 2, 8), (1, 2, 1, 4), (33, 6, 3, 16)])
def test_decode_equals_last_row_of_full_backward(L, H, Hk, d):
    rng = np.random.default_rng(L * 7 + H)
    scale = 1.0 / math.sqrt(d)
    q, K, V, dout = _case(rng, L, H, Hk, d)
    P, _ = _probs(q, K, H, Hk, d, scale)
    ds, dq, dk, dv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    # the same query as the last row of a causal sequence of length L
    Q = rng.standard_normal((L, H * d))
    Q[L - 1] = q
    dO = np.zeros((L, H * d))
    dO[L - 1] = dout
    seg = np.zeros(L, np.uint32)
    _, lse = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    rq, rk, rv = oracle.bwd(Q, K, V, dO, lse, seg, H, Hk, d, scale)
    np.testing.assert_allclose(dq, rq[L - 1], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, rk, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, rv, rtol=1e-10, atol=1e-12)


def test_decode_central_differences():
    rng = np.random.default_rng(3)
    L, H, Hk, d = 5, 4, 2, 4
    scale = 0.7
    q, K, V, dout = _case(rng, L, H, Hk, d)
    P, s = _probs(q, K, H, Hk, d, scale)
    ds, dq, dk, dv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    eps = 1e-6

    def grad(x, fn):
        g = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += eps
            xm[i] -= eps
            g[i] = (fn(xp) - fn(xm)) / (2 * eps)
        return g

    np.testing.assert_allclose(grad(q, lambda x: _f(x, K, V, dout, H, Hk, d, scale)), dq, atol=1e-7)
    np.testing.assert_allclose(grad(K, lambda x: _f(q, x, V, dout, H, Hk, d, scale)), dk, atol=1e-7)
    np.testing.assert_allclose(grad(V, lambda x: _f(q, K, x, dout, H, Hk, d, scale)), dv, atol=1e-7)

    # d_scores: the gradient with respect to the softmax input (scores)
    def f_scores(sc):
        Pp = _softmax_rows(sc)
        G = H // Hk
        return sum(dout[h * d:(h + 1) * d] @ (Pp[h] @ V[:, (h // G) * d:(h // G + 1) * d]) for h in range(H))

    np.testing.assert_allclose(grad(s, f_scores), ds, atol=1e-7)


def test_decode_invariants_and_single_key():
    rng = np.random.default_rng(9)
    L, H, Hk, d = 19, 8, 2, 8
    q, K, V, dout = _case(rng, L, H, Hk, d)
    P, _ = _probs(q, K, H, Hk, d, 0.3)
    ds, _, _, _ = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, 0.3)
    np.testing.assert_allclose(ds.sum(axis=1), 0.0, atol=1e-12)
    # history_len 1: probs = 1, no gradient through the softmax
    q, K, V, dout = _case(rng, 1, H, Hk, d)
    P = np.ones((H, 1))
    ds, dq, dk, dv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, 0.3)
    assert np.all(ds == 0) and np.all(dq == 0) and np.all(dk == 0)
    G = H // Hk
    for g in range(Hk):
        want = sum(dout[h * d:(h + 1) * d] for h in range(g * G, (g + 1) * G))
        np.testing.assert_allclose(dv[0, g * d:(g + 1) * d], want, rtol=1e-14)


def test_decode_gqa_is_group_sum_of_mha():
    rng = np.random.default_rng(21)
    L, H, Hk, d = 11, 6, 2, 8
    G = H // Hk
    scale = 0.5
    q, K, V, dout = _case(rng, L, H, Hk, d)
    P, _ = _probs(q, K, H, Hk, d, scale)
    ds, dq, dk, dv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    # multi-head: kv head per query head, K/V columns repeated
    Km = np.concatenate([K[:, (h // G) * d:(h // G + 1) * d] for h in range(H)], axis=1)
    Vm = np.concatenate([V[:, (h // G) * d:(h // G + 1) * d] for h in range(H)], axis=1)
    ds_m, dq_m, dk_m, dv_m = oracle.decode_bwd(q, Km, Vm, P, dout, H, H, d, scale)
    np.testing.assert_allclose(ds, ds_m, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dq, dq_m, rtol=1e-12, atol=1e-14)
    for g in range(Hk):
        np.testing.assert_allclose(dk[:, g * d:(g + 1) * d],
                                   sum(dk_m[:, h * d:(h + 1) * d] for h in range(g * G, (g + 1) * G)),
                                   rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(dv[:, g * d:(g + 1) * d],
                                   sum(dv_m[:, h * d:(h + 1) * d] for h in range(g * G, (g + 1) * G)),
                                   rtol=1e-12, atol=1e-14)


def _decode_mutant(kind, q, K, V, P, dout, H, Hk, d, scale):
    """A copy of the oracle's decode backward with one planted mistake."""
    G = H // Hk
    L = K.shape[0]
    ds_all, dq = np.zeros((H, L)), np.zeros(H * d)
    dk, dv = np.zeros((L, Hk * d)), np.zeros((L, Hk * d))
    for h in range(H):
        g = (h % Hk) if kind == "interleaved_gqa" else h // G
        Kg, Vg = K[:, g * d:(g + 1) * d], V[:, g * d:(g + 1) * d]
        qh, oh = q[h * d:(h + 1) * d], dout[h * d:(h + 1) * d]
        dP = Vg @ oh
        D = 0.0 if kind == "no_D" else P[h] @ dP
        ds = P[h] * (dP - D) if kind != "sign" else P[h] * (D - dP)
        ds_all[h] = ds
        dq[h * d:(h + 1) * d] = (1.0 if kind == "no_scale" else scale) * (Kg.T @ ds)
        dk[:, g * d:(g + 1) * d] += scale * np.outer(ds, qh)
        dv[:, g * d:(g + 1) * d] += np.outer(P[h], oh)
    return ds_all, dq, dk, dv


@pytest.mark.parametrize("kind", ["interleaved_gqa", "no_D", "sign", "no_scale"])
def test_planted_decode_mistakes_fail_the_pins(kind):
    rng = np.random.default_rng(44)
    L, H, Hk, d = 9, 4, 2, 4
    scale = 0.6
    q, K, V, dout = _case(rng, L, H, Hk, d)
    P, _ = _probs(q, K, H, Hk, d, scale)
    got = _decode_mutant(kind, q, K, V, P, dout, H, Hk, d, scale)
    ref = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    assert all(np.allclose(a, b) for a, b in zip(_decode_mutant("none", q, K, V, P, dout, H, Hk, d, scale), ref))
    # the full-backward pin and the finite-difference pin, applied to the mutant
    Q = rng.standard_normal((L, H * d))
    Q[L - 1] = q
    dO = np.zeros((L, H * d))
    dO[L - 1] = dout
    seg = np.zeros(L, np.uint32)
    _, lse = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    rq, rk, rv = oracle.bwd(Q, K, V, dO, lse, seg, H, Hk, d, scale)
    full_ok = (np.allclose(got[1], rq[L - 1]) and np.allclose(got[2], rk) and np.allclose(got[3], rv))
    eps = 1e-6
    fd_q = np.array([(_f(q + eps * e, K, V, dout, H, Hk, d, scale) - _f(q - eps * e, K, V, dout, H, Hk, d, scale))
                     / (2 * eps) for e in np.eye(H * d)])
    fd_ok = np.allclose(fd_q, got[1], atol=1e-7)
    assert not (full_ok and fd_ok), kind
