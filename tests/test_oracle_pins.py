"""Pins for the fp64 oracle: what mathematics and the pages fix, independently of
the oracle's own code (finite differences, closed forms, exact invariants, an
independent autograd of the forward definition, and the pages' worked examples).
"""
import math
import os

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, rng, sigma=1.0):
    return rng.standard_normal(shape) * sigma


def _case(S, H, Hk, d, seed, seg=None, sigma=1.0):
    rng = np.random.default_rng(seed)
    Q = _rand((S, H * d), rng, sigma)
    K = _rand((S, Hk * d), rng, sigma)
    V = _rand((S, Hk * d), rng, sigma)
    dO = _rand((S, H * d), rng, sigma)
    if seg is None:
        seg = np.zeros(S, dtype=np.uint32)
    return Q, K, V, dO, np.asarray(seg, dtype=np.uint32), 1.0 / math.sqrt(d)


def _grads(Q, K, V, dO, seg, H, Hk, d, scale):
    _, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    return oracle.bwd(Q, K, V, dO, LSE, seg, H, Hk, d, scale)


def _loss(Q, K, V, W, seg, H, Hk, d, scale):
    O, _ = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    return float(np.sum(O * W))


# ---------------------------------------------------------------------------
# whole backward: central finite differences of L = sum(O * dO)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seg", [None, [0, 0, 0, 3, 3, 5, 5]], ids=["causal", "docs"])
def test_backward_matches_central_differences(seg):
    S, H, Hk, d = 7, 4, 2, 4
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, 11, seg)
    dQ, dK, dV = _grads(Q, K, V, W, seg, H, Hk, d, scale)
    h = 1e-6
    for name, X, G in (("Q", Q, dQ), ("K", K, dK), ("V", V, dV)):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            old = X[idx]
            X[idx] = old + h
            lp = _loss(Q, K, V, W, seg, H, Hk, d, scale)
            X[idx] = old - h
            lm = _loss(Q, K, V, W, seg, H, Hk, d, scale)
            X[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        err = np.max(np.abs(num - G)) / max(1e-12, np.max(np.abs(num)))
        assert err < 1e-6, (name, err)


# ---------------------------------------------------------------------------
# independent implementation: float64 autograd of masked softmax attention
# ---------------------------------------------------------------------------
def _torch_reference(Q, K, V, W, seg, H, Hk, d, scale):
    torch = pytest.importorskip("torch")
    S = Q.shape[0]
    G = H // Hk
    q = torch.tensor(Q, dtype=torch.float64).view(S, H, d).requires_grad_(True)
    k = torch.tensor(K, dtype=torch.float64).view(S, Hk, d).requires_grad_(True)
    v = torch.tensor(V, dtype=torch.float64).view(S, Hk, d).requires_grad_(True)
    w = torch.tensor(W, dtype=torch.float64).view(S, H, d)
    kr = k.repeat_interleave(G, dim=1)          # blocked groups: head h reads kv h // G
    vr = v.repeat_interleave(G, dim=1)
    scores = torch.einsum("ihe,jhe->hij", q, kr) * scale
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    lo = torch.tensor(seg.astype(np.int64))[:, None]
    mask = (j <= i) & (j >= lo)
    scores = scores.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(scores, dim=-1)       # [H, S]
    out = torch.einsum("hij,jhe->ihe", torch.softmax(scores, dim=-1), vr)
    (out * w).sum().backward()
    return (out.detach().reshape(S, H * d).numpy(), lse.detach().T.numpy(),
            q.grad.reshape(S, H * d).numpy(), k.grad.reshape(S, Hk * d).numpy(),
            v.grad.reshape(S, Hk * d).numpy())


@pytest.mark.parametrize("S,H,Hk,d,seg_kind", [
    (9, 4, 2, 8, "causal"), (33, 6, 2, 16, "docs"), (20, 4, 4, 8, "nonmonotone"),
    (17, 8, 1, 4, "docs")])
def test_matches_float64_autograd(S, H, Hk, d, seg_kind):
    rng = np.random.default_rng(S * 7 + H)
    if seg_kind == "causal":
        seg = np.zeros(S, np.uint32)
    else:
        seg = workloads.random_seg(S, rng, monotone=(seg_kind == "docs"))
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, S + d, seg)
    O_ref, L_ref, dQ_ref, dK_ref, dV_ref = _torch_reference(Q, K, V, W, seg, H, Hk, d, scale)
    O, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    dQ, dK, dV = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    for got, ref in ((O, O_ref), (LSE, L_ref), (dQ, dQ_ref), (dK, dK_ref), (dV, dV_ref)):
        assert np.max(np.abs(got - ref)) <= 1e-11 * max(1.0, np.max(np.abs(ref)))


# ---------------------------------------------------------------------------
# exact invariants and closed forms
# ---------------------------------------------------------------------------
def test_dS_rows_sum_to_zero():
    """sum_j dS_ij = sigma * D_i * (1 - sum_j P_ij) = 0 when LSE is exact."""
    S, H, Hk, d = 40, 4, 2, 8
    seg = workloads.random_seg(S, np.random.default_rng(3))
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, 5, seg)
    _, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    for h in range(H):
        t = oracle.row_terms(Q, K, V, W, LSE, seg, h, H, Hk, d, scale, np.arange(S))
        np.testing.assert_allclose(t["P"].sum(axis=1), 1.0, rtol=0, atol=1e-13)
        assert np.max(np.abs(t["dS"].sum(axis=1))) < 1e-13 * np.max(np.abs(t["dS"]))


def test_seq_len_one():
    """One token: P = 1, D = dP, dS = 0, so dQ = dK = 0 and dV = sum of the group's dO."""
    H, Hk, d = 6, 2, 8
    Q, K, V, W, seg, scale = _case(1, H, Hk, d, 9)
    O, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    G = H // Hk
    for h in range(H):
        g = h // G
        np.testing.assert_array_equal(O[0, h * d:(h + 1) * d], V[0, g * d:(g + 1) * d])
    dQ, dK, dV = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    assert np.all(dQ == 0) and np.all(dK == 0)
    for g in range(Hk):
        want = sum(W[0, h * d:(h + 1) * d] for h in range(g * G, (g + 1) * G))
        np.testing.assert_allclose(dV[0, g * d:(g + 1) * d], want, rtol=1e-15, atol=1e-15)


def test_zero_keys_closed_form():
    """K = 0: uniform attention over each row's allowed keys.

    LSE_i = ln(n_i), O_i = mean of the allowed V rows, dQ = 0,
    dV_j = sum over rows i that see j of dO_i / n_i, with n_i = i - seg[i] + 1.
    """
    S, H, Hk, d = 23, 4, 2, 4
    seg = np.array([0] * 5 + [5] * 9 + [14] * 9, dtype=np.uint32)
    Q, _, V, W, seg, scale = _case(S, H, Hk, d, 21, seg)
    K = np.zeros((S, Hk * d))
    O, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    G = H // Hk
    n = np.array([i - int(seg[i]) + 1 for i in range(S)], dtype=np.float64)
    for h in range(H):
        g = h // G
        np.testing.assert_allclose(LSE[:, h], np.log(n), rtol=0, atol=1e-14)
        for i in range(S):
            mean_v = sum(V[j, g * d:(g + 1) * d] for j in range(int(seg[i]), i + 1)) / n[i]
            np.testing.assert_allclose(O[i, h * d:(h + 1) * d], mean_v, rtol=1e-13, atol=1e-14)
    dQ, dK, dV = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    assert np.all(dQ == 0)
    for g in range(Hk):
        for j in range(S):
            want = np.zeros(d)
            for h in range(g * G, (g + 1) * G):
                for i in range(j, S):
                    if seg[i] <= j:
                        want += W[i, h * d:(h + 1) * d] / n[i]
            np.testing.assert_allclose(dV[j, g * d:(g + 1) * d], want, rtol=1e-12, atol=1e-13)


def test_two_key_closed_form():
    """Second row of a 2-token sequence: a two-term softmax written out by hand."""
    H, Hk, d = 2, 1, 3
    Q, K, V, W, seg, scale = _case(2, H, Hk, d, 4)
    O, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    for h in range(H):
        q = Q[1, h * d:(h + 1) * d]
        a = scale * float(q @ K[0]); b = scale * float(q @ K[1])
        ea, eb = math.exp(a), math.exp(b)
        np.testing.assert_allclose(LSE[1, h], math.log(ea + eb), rtol=1e-15)
        np.testing.assert_allclose(O[1, h * d:(h + 1) * d], (ea * V[0] + eb * V[1]) / (ea + eb),
                                   rtol=1e-14)
        np.testing.assert_allclose(LSE[0, h], scale * float(Q[0, h * d:(h + 1) * d] @ K[0]), rtol=1e-15)


def test_key_translation_invariance():
    """Adding one vector c to every key shifts each row's logits by sigma q.c:
    O, dQ, dK and dV are unchanged (dQ only because sum_j dS_ij = 0)."""
    S, H, Hk, d = 19, 4, 2, 8
    seg = workloads.random_seg(S, np.random.default_rng(8))
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, 13, seg)
    c = np.random.default_rng(1).standard_normal(d)
    K2 = K + np.tile(c, Hk)[None, :]
    O1, _ = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    O2, _ = oracle.fwd(Q, K2, V, seg, H, Hk, d, scale)
    np.testing.assert_allclose(O1, O2, rtol=1e-10, atol=1e-11)
    g1 = _grads(Q, K, V, W, seg, H, Hk, d, scale)
    g2 = _grads(Q, K2, V, W, seg, H, Hk, d, scale)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-10)


def test_accumulates_into_given_arrays():
    S, H, Hk, d = 12, 4, 2, 4
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, 2)
    _, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    once = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    acc = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    acc = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale, *acc)
    for a, b in zip(once, acc):
        np.testing.assert_allclose(2 * a, b, rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------------------
# document mask: no gradient crosses a document boundary
# ---------------------------------------------------------------------------
def _docs_case():
    S, H, Hk, d = 21, 4, 2, 4
    seg = np.array([0] * 8 + [8] * 6 + [14] * 7, dtype=np.uint32)
    return (S, H, Hk, d) + _case(S, H, Hk, d, 31, seg)


def test_docs_block_diagonal_equivalence():
    """Packed documents give the same gradients as each document run alone."""
    S, H, Hk, d, Q, K, V, W, seg, scale = _docs_case()
    dQ, dK, dV = _grads(Q, K, V, W, seg, H, Hk, d, scale)
    for a, b in ((0, 8), (8, 14), (14, 21)):
        z = np.zeros(b - a, np.uint32)
        q, k, v, w = Q[a:b], K[a:b], V[a:b], W[a:b]
        sq, sk, sv = _grads(q, k, v, w, z, H, Hk, d, scale)
        np.testing.assert_allclose(dQ[a:b], sq, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dK[a:b], sk, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dV[a:b], sv, rtol=1e-12, atol=1e-13)


def test_docs_no_cross_flow():
    S, H, Hk, d, Q, K, V, W, seg, scale = _docs_case()
    _, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    # (1) no upstream gradient on document B -> no dK / dV on B's keys
    W0 = W.copy(); W0[8:14] = 0
    _, dK, dV = oracle.bwd(Q, K, V, W0, LSE, seg, H, Hk, d, scale)
    assert np.all(dK[8:14] == 0) and np.all(dV[8:14] == 0)
    # (2) changing K, V of document A leaves dQ of documents B, C bit-identical
    dQ1, _, _ = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    K2, V2 = K.copy(), V.copy()
    K2[:8] += 1.5; V2[:8] -= 0.75
    dQ2, _, _ = oracle.bwd(Q, K2, V2, W, LSE, seg, H, Hk, d, scale)
    np.testing.assert_array_equal(dQ1[8:], dQ2[8:])


# ---------------------------------------------------------------------------
# GQA: dK / dV of a kv head equal the sum over its query heads of an MHA run
# ---------------------------------------------------------------------------
def test_gqa_equals_group_sum_of_mha():
    S, H, Hk, d = 15, 6, 2, 4
    G = H // Hk
    seg = workloads.random_seg(S, np.random.default_rng(4))
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, 17, seg)
    dQ, dK, dV = _grads(Q, K, V, W, seg, H, Hk, d, scale)
    # repeat kv head g for its G query heads (blocked: head h reads g = h // G)
    Kr = np.concatenate([K[:, (h // G) * d:(h // G + 1) * d] for h in range(H)], axis=1)
    Vr = np.concatenate([V[:, (h // G) * d:(h // G + 1) * d] for h in range(H)], axis=1)
    mQ, mK, mV = _grads(Q, Kr, Vr, W, seg, H, H, d, scale)
    np.testing.assert_allclose(dQ, mQ, rtol=1e-12, atol=1e-13)
    for g in range(Hk):
        sk = sum(mK[:, h * d:(h + 1) * d] for h in range(g * G, (g + 1) * G))
        sv = sum(mV[:, h * d:(h + 1) * d] for h in range(g * G, (g + 1) * G))
        np.testing.assert_allclose(dK[:, g * d:(g + 1) * d], sk, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dV[:, g * d:(g + 1) * d], sv, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# the sampled forms used at large sizes agree with the whole backward
# ---------------------------------------------------------------------------
def test_sampled_outputs_match_whole_backward():
    S, H, Hk, d = 300, 4, 2, 8
    seg = workloads.random_seg(S, np.random.default_rng(6))
    Q, K, V, W, seg, scale = _case(S, H, Hk, d, 23, seg)
    _, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    dQ, dK, dV = oracle.bwd(Q, K, V, W, LSE, seg, H, Hk, d, scale)
    rows = np.array([0, 1, 127, 128, 255, 299])
    np.testing.assert_allclose(oracle.bwd_rows(Q, K, V, W, LSE, seg, H, Hk, d, scale, rows),
                               dQ[rows], rtol=1e-12, atol=1e-13)
    keys = np.array([0, 64, 200, 299])
    sk, sv = oracle.bwd_dkdv_keys(Q, K, V, W, LSE, seg, H, Hk, d, scale, keys)
    np.testing.assert_allclose(sk, dK[keys], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(sv, dV[keys], rtol=1e-12, atol=1e-13)
    _, Lr = oracle.fwd(Q, K, V, seg, H, Hk, d, scale, rows=rows)
    np.testing.assert_allclose(Lr[rows], LSE[rows], rtol=1e-14)
