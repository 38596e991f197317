"""fp64 CPU oracle for causal grouped-query attention: forward (O, LSE) and the
backward pass from a saved log-sum-exp, plus the interleaved RoPE backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may use it. It shares no code with the CUDA path.

What it computes, and where the pages define it
-----------------------------------------------
Notation: S = seq_len, H = n_heads, Hk = n_kv_heads, G = H / Hk, d = head_dim,
sigma = scale. Query head h reads kv head g(h) = floor(h / G) ("blocked" GQA;
10_backward_attention.wgsl, kernel ``attention_backward``, ``kv_h = h /
q_per_group``; tang ``llm.rs``, ``causal_attention_fused``, ``kv_head = head /
heads_per_group``). Key j is visible to query i iff seg[i] <= j <= i
(10_backward_attention.wgsl, ``attention_backward``: the ``doc_start`` /
``causal_len`` test).

Forward (tang ``llm.rs``, ``causal_attention_fused``: row max, sum of exps,
weighted V; document mask added as in the wgsl kernels):
    s_ij = sigma * q_i . k_j             (allowed pairs)
    LSE_i = m_i + ln sum_j exp(s_ij - m_i),   m_i = max_j s_ij
    O_i = sum_j exp(s_ij - LSE_i) v_j

Backward from a given LSE (10_backward_attention.wgsl header and kernel
``attention_backward``; explicit-matrix form of tang ``llm.rs``,
``GpuTrainModule for GpuCausalAttention::backward``):
    P_ij  = exp(s_ij - LSE_i) if allowed else 0
    dP_ij = dO_i . v_j
    D_i   = sum_j P_ij dP_ij
    dS_ij = sigma * P_ij (dP_ij - D_i)
    dQ_i += sum_j dS_ij k_j
    dK_j += sum_{h in group} sum_i dS_ij q_i
    dV_j += sum_{h in group} sum_i P_ij dO_i
Gradients accumulate (``+=``) into the arrays passed in.

Interleaved RoPE backward (10_backward_attention.wgsl, ``rope_q_backward`` /
``rope_k_backward``; tang ``llm.rs``, ``interleaved_rope_backward`` and the
f64 angle tables of ``GpuInterleavedRoPE::new``): for pair p < d/2 at position
t = pos_offset + s, theta = t * base^(-2p/d) computed in fp64,
    (x0, x1) <- (x0 cos theta + x1 sin theta, -x0 sin theta + x1 cos theta).

The explicit matrices P, dP, dS are materialised for one head and one block of
query rows at a time (keys 0 .. last row of the block), which bounds memory;
every row is computed from its own definition, so the block size changes
nothing but rounding order inside the library matrix products.

Decode-style backward from saved probabilities (rullama ``training.rs``,
``attention_backward_dq_chained`` / ``attention_backward_dkv_chained``; the
page gives their buffer bindings and launch shapes, not the kernel bodies):
one query per head against history_len cached keys, with the softmax
probabilities of the forward stored instead of an LSE. Reading taken: the
probabilities are softmax_j(sigma q_h . k_j), ``d_scores`` is the gradient
with respect to those scores, and sigma is an argument (the page's parameter
block has none; 1/sqrt(d) is the usual value):
    dP_hj = d_out_h . v_j,   D_h = sum_j probs_hj dP_hj
    d_scores_hj = probs_hj (dP_hj - D_h)
    d_q_h  += sigma sum_j d_scores_hj k_j
    d_k_j  += sigma sum_{h in group} d_scores_hj q_h
    d_v_j  += sum_{h in group} probs_hj d_out_h

Pins: every function here is checked by ``tests/test_oracle_pins.py`` (and
``tests/test_oracle_decode.py`` for the decode backward) against
central finite differences, closed forms (K = 0, S = 1, position 0), exact
invariants (sum_j dS_ij = 0, no cross-document flow, GQA group sums) and an
independent float64 autograd of the forward definition.
"""
from __future__ import annotations

import concurrent.futures as _cf
import os
import sys

if "numpy" not in sys.modules:      # the pool below supplies the parallelism
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
import numpy as np  # noqa: E402

__all__ = ["fwd", "bwd", "bwd_rows", "bwd_dkdv_keys", "row_terms", "rope_bwd",
           "allowed", "decode_bwd"]

_ROW_BLOCK = 256


def _f64(x):
    return np.asarray(x, dtype=np.float64)


def allowed(seg: np.ndarray, rows: np.ndarray, n_keys: int) -> np.ndarray:
    """Boolean mask [len(rows), n_keys]: key j visible to query i iff seg[i] <= j <= i."""
    rows = np.asarray(rows, dtype=np.int64)
    j = np.arange(n_keys, dtype=np.int64)[None, :]
    lo = np.asarray(seg, dtype=np.int64)[rows][:, None]
    return (j >= lo) & (j <= rows[:, None])


def _check_shapes(S, H, Hk, d):
    if Hk <= 0 or H % Hk != 0:
        raise ValueError("n_heads must be a positive multiple of n_kv_heads")
    if d <= 0:
        raise ValueError("head_dim must be positive")


def _head_cols(h, d):
    return slice(h * d, (h + 1) * d)


def _workers() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def _for_each(fn, items):
    """Run fn(item) for independent items (distinct output columns) on a thread
    pool; numpy releases the GIL inside its kernels. Each item is computed by
    one thread in a fixed order, so results do not depend on scheduling."""
    items = list(items)
    if len(items) <= 1 or _workers() == 1:
        for it in items:
            fn(it)
        return
    with _cf.ThreadPoolExecutor(max_workers=min(len(items), _workers())) as ex:
        for f in [ex.submit(fn, it) for it in items]:
            f.result()


def _blocks(rows: np.ndarray):
    for b in range(0, len(rows), _ROW_BLOCK):
        yield rows[b:b + _ROW_BLOCK]


def fwd(Q, K, V, seg, n_heads, n_kv_heads, head_dim, scale, rows=None):
    """Forward attention: returns (O [S, H*d], LSE [S, H]) in fp64.

    With ``rows`` given, only those query rows are filled (others stay zero).
    LSE is the natural log, scale included, over allowed keys only, so that
    exp(sigma q.k - LSE) sums to one over a row.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    S = Q.shape[0]
    H, Hk, d = n_heads, n_kv_heads, head_dim
    _check_shapes(S, H, Hk, d)
    G = H // Hk
    O = np.zeros((S, H * d))
    LSE = np.zeros((S, H))
    all_rows = np.arange(S, dtype=np.int64) if rows is None else np.sort(np.asarray(rows, np.int64))

    def one_item(item):
        h, r = item
        g = h // G
        Kg, Vg = K[:, _head_cols(g, d)], V[:, _head_cols(g, d)]
        if True:
            n_keys = int(r[-1]) + 1
            s = scale * (Q[r, _head_cols(h, d)] @ Kg[:n_keys].T)
            s = np.where(allowed(seg, r, n_keys), s, -np.inf)
            m = s.max(axis=1)
            lse = m + np.log(np.exp(s - m[:, None]).sum(axis=1))
            p = np.exp(s - lse[:, None])
            O[r, _head_cols(h, d)] = p @ Vg[:n_keys]
            LSE[r, h] = lse

    _for_each(one_item, [(h, r) for h in range(H) for r in _blocks(all_rows)])
    return O, LSE


def row_terms(Q, K, V, dO, LSE, seg, h, n_heads, n_kv_heads, head_dim, scale, rows):
    """Explicit P, dP, D, dS for query head ``h`` and query ``rows``.

    Returns a dict of fp64 arrays; P, dP, dS are [len(rows), last_row + 1].
    """
    Q, K, V, dO, LSE = _f64(Q), _f64(K), _f64(V), _f64(dO), _f64(LSE)
    H, Hk, d = n_heads, n_kv_heads, head_dim
    _check_shapes(Q.shape[0], H, Hk, d)
    g = h // (H // Hk)
    r = np.asarray(rows, dtype=np.int64)
    n_keys = int(r.max()) + 1
    Kg, Vg = K[:n_keys, _head_cols(g, d)], V[:n_keys, _head_cols(g, d)]
    s = scale * (Q[r, _head_cols(h, d)] @ Kg.T)
    mask = allowed(seg, r, n_keys)
    P = np.exp(np.where(mask, s - LSE[r, h][:, None], -np.inf))
    dP = np.where(mask, dO[r, _head_cols(h, d)] @ Vg.T, 0.0)
    D = (P * dP).sum(axis=1)
    dS = scale * P * (dP - D[:, None])
    return {"P": P, "dP": dP, "D": D, "dS": dS, "keys": n_keys, "g": g}


def bwd(Q, K, V, dO, LSE, seg, n_heads, n_kv_heads, head_dim, scale,
        dQ=None, dK=None, dV=None, rows=None):
    """Backward from the given LSE; accumulates into dQ, dK, dV (fp64, created
    as zeros when not given) and returns them. ``rows`` (sorted query
    positions) restricts the sum to those query rows: the contributions of
    every other row are left out (used to time bounded samples).

    Follows the explicit-matrix backward of tang ``llm.rs``
    (``GpuCausalAttention::backward``: recompute P, dP = dO V^T, dV += P^T dO,
    D_i = sum_k dP P, dS = P (dP - D) scale, dQ += dS K, dK += dS^T Q, with the
    kv group shared by ``+=``), using the saved LSE and the document mask of
    10_backward_attention.wgsl (``attention_backward``: P = exp(scale q.k - lse)).
    """
    Q, K, V, dO, LSE = _f64(Q), _f64(K), _f64(V), _f64(dO), _f64(LSE)
    S = Q.shape[0]
    H, Hk, d = n_heads, n_kv_heads, head_dim
    _check_shapes(S, H, Hk, d)
    dQ = np.zeros((S, H * d)) if dQ is None else dQ
    dK = np.zeros((S, Hk * d)) if dK is None else dK
    dV = np.zeros((S, Hk * d)) if dV is None else dV
    all_rows = np.arange(S, dtype=np.int64) if rows is None else np.asarray(rows, np.int64)
    G = H // Hk
    # per query head: its dK / dV contribution, summed over its kv group below
    part_k = np.zeros((H, S, d))
    part_v = np.zeros((H, S, d))

    def one_head(h):
        g = h // G
        for r in _blocks(all_rows):
            t = row_terms(Q, K, V, dO, LSE, seg, h, H, Hk, d, scale, r)
            n = t["keys"]
            dQ[r, _head_cols(h, d)] += t["dS"] @ K[:n, _head_cols(g, d)]
            part_k[h, :n] += t["dS"].T @ Q[r, _head_cols(h, d)]
            part_v[h, :n] += t["P"].T @ dO[r, _head_cols(h, d)]

    _for_each(one_head, range(H))
    for h in range(H):
        g = h // G
        dK[:, _head_cols(g, d)] += part_k[h]
        dV[:, _head_cols(g, d)] += part_v[h]
    return dQ, dK, dV


def bwd_rows(Q, K, V, dO, LSE, seg, n_heads, n_kv_heads, head_dim, scale, rows, heads=None):
    """dQ of the backward for the given query ``rows`` (all heads, or ``heads``).

    Returns an fp64 array [len(rows), H*d]; columns of heads not asked for are
    zero. Each row follows the same definition as ``bwd``; this only restricts
    which outputs are formed, for spot checks at sizes where the whole backward
    would take too long.
    """
    H, Hk, d = n_heads, n_kv_heads, head_dim
    Q, K, V, dO, LSE = _f64(Q), _f64(K), _f64(V), _f64(dO), _f64(LSE)
    r_all = np.asarray(rows, dtype=np.int64)
    out = np.zeros((len(r_all), H * d))
    heads = range(H) if heads is None else heads

    def one_item(item):
        h, b = item
        g = h // (H // Hk)
        r = r_all[b:b + _ROW_BLOCK]
        t = row_terms(Q, K, V, dO, LSE, seg, h, H, Hk, d, scale, r)
        out[b:b + len(r), _head_cols(h, d)] = t["dS"] @ K[:t["keys"], _head_cols(g, d)]

    _for_each(one_item, [(h, b) for h in heads for b in range(0, len(r_all), _ROW_BLOCK)])
    return out


def bwd_dkdv_keys(Q, K, V, dO, LSE, seg, n_heads, n_kv_heads, head_dim, scale, keys, kv_heads=None):
    """dK and dV of the backward for the given key positions ``keys``.

    Returns two fp64 arrays [len(keys), Hk*d] (kv heads not asked for stay
    zero). Every query row that can see one of the keys (rows >= min(keys)) is
    formed in full, since its D needs the whole row; only the key columns asked
    for are summed.
    """
    Q, K, V, dO, LSE = _f64(Q), _f64(K), _f64(V), _f64(dO), _f64(LSE)
    S = Q.shape[0]
    H, Hk, d = n_heads, n_kv_heads, head_dim
    keys = np.asarray(keys, dtype=np.int64)
    dK = np.zeros((len(keys), Hk * d))
    dV = np.zeros((len(keys), Hk * d))
    if len(keys) == 0:
        return dK, dV
    rows = np.arange(int(keys.min()), S, dtype=np.int64)
    kv_heads = range(Hk) if kv_heads is None else kv_heads
    G = H // Hk

    items = [(h, b) for g in kv_heads for h in range(g * G, (g + 1) * G)
             for b in range(0, len(rows), _ROW_BLOCK)]
    part_k = {it: np.zeros((len(keys), d)) for it in items}
    part_v = {it: np.zeros((len(keys), d)) for it in items}

    def one_item(item):
        h, b = item
        r = rows[b:b + _ROW_BLOCK]
        t = row_terms(Q, K, V, dO, LSE, seg, h, H, Hk, d, scale, r)
        sel = keys < t["keys"]
        kk = keys[sel]
        part_k[item][sel] = t["dS"][:, kk].T @ Q[r, _head_cols(h, d)]
        part_v[item][sel] = t["P"][:, kk].T @ dO[r, _head_cols(h, d)]

    _for_each(one_item, items)
    for it in items:                      # fixed summation order
        g = it[0] // G
        dK[:, _head_cols(g, d)] += part_k[it]
        dV[:, _head_cols(g, d)] += part_v[it]
    return dK, dV


def rope_bwd(dX, n_heads, head_dim, pos_offset=0, base=10000.0):
    """Interleaved RoPE backward (transposed rotation), returned as a new fp64 array.

    dX is [S, n_heads*head_dim]; pair p of head h at row s is columns
    (h*d + 2p, h*d + 2p + 1); the angle is (pos_offset + s) * base^(-2p/d) in fp64.
    """
    X = _f64(dX).copy()
    S = X.shape[0]
    d = head_dim
    if d % 2:
        raise ValueError("head_dim must be even for RoPE")
    X = X.reshape(S, n_heads, d // 2, 2)
    pos = (np.arange(S, dtype=np.float64) + pos_offset)[:, None]
    inv_freq = np.array([base ** (-(2.0 * p) / d) for p in range(d // 2)], dtype=np.float64)
    theta = pos * inv_freq[None, :]                     # [S, d/2]
    c, s = np.cos(theta)[:, None, :], np.sin(theta)[:, None, :]
    x0, x1 = X[..., 0].copy(), X[..., 1].copy()
    X[..., 0] = x0 * c + x1 * s
    X[..., 1] = -x0 * s + x1 * c
    return X.reshape(S, n_heads * d)


def decode_bwd(q, k_hist, v_hist, probs, d_out, n_heads, n_kv_heads, head_dim, scale):
    """Decode-style attention backward from saved probabilities, in fp64.

    rullama ``training.rs``, ``attention_backward_dq_chained`` (pass 1: d_q and
    the staged d_scores [n_heads, history_len] from k_hist, v_hist, probs,
    d_out) and ``attention_backward_dkv_chained`` (pass 2: d_k_hist, d_v_hist
    from q, probs, d_out, d_scores). Layouts: q, d_out [H*d]; k_hist, v_hist
    [L, Hk*d] (row-major, kv head g in columns g*d .. g*d+d-1); probs [H, L].
    Per query head h with kv head g = h // (H/Hk), written out from the softmax
    backward (module docstring):
        dP = V_g d_out_h;  D = probs_h . dP;  d_scores_h = probs_h * (dP - D)
        d_q_h = sigma K_g^T d_scores_h
        d_k[:, g] += sigma outer(d_scores_h, q_h);  d_v[:, g] += outer(probs_h, d_out_h)
    Returns (d_scores [H, L], d_q [H*d], d_k [L, Hk*d], d_v [L, Hk*d]) as new
    fp64 arrays (the gradients' contributions, to be added by the caller).
    """
    H, Hk, d = n_heads, n_kv_heads, head_dim
    if H % Hk:
        raise ValueError("n_heads must be a multiple of n_kv_heads")
    G = H // Hk
    q, d_out = _f64(q).reshape(H * d), _f64(d_out).reshape(H * d)
    K, V, P = _f64(k_hist), _f64(v_hist), _f64(probs)
    L = K.shape[0]
    if K.shape != (L, Hk * d) or V.shape != (L, Hk * d) or P.shape != (H, L):
        raise ValueError("shape mismatch")
    d_scores = np.zeros((H, L))
    d_q = np.zeros(H * d)
    d_k = np.zeros((L, Hk * d))
    d_v = np.zeros((L, Hk * d))
    for h in range(H):
        g = h // G
        Kg, Vg = K[:, _head_cols(g, d)], V[:, _head_cols(g, d)]
        qh, oh = q[_head_cols(h, d)], d_out[_head_cols(h, d)]
        dP = Vg @ oh
        D = P[h] @ dP
        ds = P[h] * (dP - D)
        d_scores[h] = ds
        d_q[_head_cols(h, d)] = scale * (Kg.T @ ds)
        d_k[:, _head_cols(g, d)] += scale * np.outer(ds, qh)
        d_v[:, _head_cols(g, d)] += np.outer(P[h], oh)
    return d_scores, d_q, d_k, d_v
