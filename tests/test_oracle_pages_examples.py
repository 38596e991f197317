"""The pages' own worked examples (tests/golden/*.txt), run against the oracle,
plus RoPE-backward pins (orthogonality, position 0, inverse of the forward)."""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


def _rope_fwd(x, pos, base=10000.0):
    """The pages' forward rotation of one interleaved head vector
    (tang llm.rs, GpuInterleavedRoPE::forward: y0 = x0 c - x1 s, y1 = x0 s + x1 c;
    angle pos / base^(2i/d) in f64)."""
    d = len(x)
    y = np.array(x, dtype=np.float64)
    for i in range(d // 2):
        th = pos / base ** (2.0 * i / d)
        c, s = math.cos(th), math.sin(th)
        x0, x1 = x[2 * i], x[2 * i + 1]
        y[2 * i] = x0 * c - x1 * s
        y[2 * i + 1] = x0 * s + x1 * c
    return y


def test_rope_pages_examples():
    f = _fixture("tang_rope_backward.txt")
    # identity at position 0 (forward and backward)
    x = np.array([float(v) for v in f["identity_input"]])
    tol = float(f["identity_tol"][0])
    np.testing.assert_allclose(_rope_fwd(x, int(f["identity_pos"][0])), x, atol=tol)
    np.testing.assert_allclose(oracle.rope_bwd(x[None, :], 1, 4, int(f["identity_pos"][0])).ravel(),
                               x, atol=0)
    # rotation of e0 at position 5 -> (cos 5, sin 5) in pair 0
    x = np.array([float(v) for v in f["rotation_input"]])
    y = _rope_fwd(x, int(f["rotation_pos"][0]))
    assert abs(y[0] - math.cos(5.0)) < float(f["rotation_tol"][0])
    assert abs(y[1] - math.sin(5.0)) < float(f["rotation_tol"][0])
    # backward of grad e0 at position 3 == central difference of forward output[0]
    pos, h = int(f["fd_pos"][0]), float(f["fd_h"][0])
    x = np.array([float(v) for v in f["fd_input"]])
    g = np.array([float(v) for v in f["fd_grad_out"]])
    gi = oracle.rope_bwd(g[None, :], 1, 4, 0 + pos).ravel()
    for k in range(4):
        xp, xm = x.copy(), x.copy()
        xp[k] += h
        xm[k] -= h
        num = (_rope_fwd(xp, pos)[0] - _rope_fwd(xm, pos)[0]) / (2 * h)
        assert abs(gi[k] - num) < float(f["fd_tol"][0])


def test_rope_bwd_inverts_forward_and_is_orthogonal():
    rng = np.random.default_rng(0)
    S, H, d = 37, 3, 8
    X = rng.standard_normal((S, H * d))
    Y = np.stack([np.concatenate([_rope_fwd(X[s, h * d:(h + 1) * d], s + 11) for h in range(H)])
                  for s in range(S)])
    back = oracle.rope_bwd(Y, H, d, pos_offset=11)
    np.testing.assert_allclose(back, X, rtol=1e-12, atol=1e-12)
    # each pair keeps its norm
    Z = oracle.rope_bwd(X, H, d, pos_offset=3).reshape(S, H, d // 2, 2)
    Xp = X.reshape(S, H, d // 2, 2)
    np.testing.assert_allclose(np.hypot(Z[..., 0], Z[..., 1]), np.hypot(Xp[..., 0], Xp[..., 1]),
                               rtol=1e-13)


def test_rope_angle_convention_closed_form():
    """Pair p at position t rotates by t * 10000^(-2p/d): d = 4, p = 1, t = 5 gives 0.05 rad."""
    x = np.zeros((6, 4))
    x[5, 2] = 1.0
    y = oracle.rope_bwd(x, 1, 4)
    np.testing.assert_allclose(y[5], [0.0, 0.0, math.cos(0.05), -math.sin(0.05)], atol=1e-15)


def _weights(seed, rows, cols):
    return np.array([((i * seed + 3) % 17) * 0.1 - 0.8 for i in range(rows * cols)]).reshape(rows, cols)


def test_tang_attention_layer_gradient_check():
    """The pages' layer gradient check: input -> (Wq, Wk, Wv) -> causal GQA
    attention -> Wo -> sum; the attention part of the chain rule is the
    oracle's backward, checked against central differences of the forward."""
    f = _fixture("tang_attention_gradcheck.txt")
    S, dim = int(f["seq_len"][0]), int(f["dim"][0])
    H, Hk, d = int(f["n_heads"][0]), int(f["n_kv_heads"][0]), int(f["head_dim"][0])
    Wq = _weights(int(f["wq_seed"][0]), H * d, dim)
    Wk = _weights(int(f["wk_seed"][0]), Hk * d, dim)
    Wv = _weights(int(f["wv_seed"][0]), Hk * d, dim)
    Wo = _weights(int(f["wo_seed"][0]), dim, H * d)
    x = np.array([float(v) for v in f["input"]]).reshape(S, dim)
    scale = 1.0 / math.sqrt(d)
    seg = np.zeros(S, np.uint32)

    def total(inp):
        O, _ = oracle.fwd(inp @ Wq.T, inp @ Wk.T, inp @ Wv.T, seg, H, Hk, d, scale)
        return float(np.sum(O @ Wo.T))

    Q, K, V = x @ Wq.T, x @ Wk.T, x @ Wv.T
    _, LSE = oracle.fwd(Q, K, V, seg, H, Hk, d, scale)
    dO = np.full((S, dim), float(f["grad_out_all"][0])) @ Wo
    dQ, dK, dV = oracle.bwd(Q, K, V, dO, LSE, seg, H, Hk, d, scale)
    analytic = dQ @ Wq + dK @ Wk + dV @ Wv
    eps = float(f["fd_eps"][0])
    numeric = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += eps
        xm[idx] -= eps
        numeric[idx] = (total(xp) - total(xm)) / (2 * eps)
    # the page's bar (fp32, eps 1e-3) and a tight fp64 bar
    assert np.max(np.abs(analytic - numeric)) < float(f["abs_tol"][0])
    assert np.max(np.abs(analytic - numeric)) < 1e-6
