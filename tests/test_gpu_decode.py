"""GPU parity of the decode-style backward from saved probabilities
(attn_decode_bwd; rullama training.rs, attention_backward_dq_chained /
attention_backward_dkv_chained) against the fp64 oracle (oracle.decode_bwd)
on the same seeded fp32 inputs, through the C ABI.

Acceptance per output tensor: max|gpu - oracle| <= 5e-3 * max|oracle| (the
bound of the main backward; the kernels run fp32 FMA chains, far inside it).
"""
import math

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 5e-3


@pytest.fixture(scope="module")
def ga():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_attn_gb300 import build
    build.build()
    import causal_gqa_attention_attn_gb300 as mod
    return mod


def _inputs(L, H, Hk, d, seed, softmax_probs=True):
    rng = np.random.default_rng(seed)
    G = H // Hk
    scale = 1.0 / math.sqrt(d)
    q = rng.standard_normal(H * d, dtype=np.float32)
    K = rng.standard_normal((L, Hk * d), dtype=np.float32)
    V = rng.standard_normal((L, Hk * d), dtype=np.float32)
    dout = rng.standard_normal(H * d, dtype=np.float32)
    if softmax_probs:   # the forward's probabilities of this query (fp64 softmax, stored fp32)
        s = np.stack([scale * K[:, (h // G) * d:(h // G + 1) * d].astype(np.float64) @ q[h * d:(h + 1) * d]
                      for h in range(H)])
        e = np.exp(s - s.max(axis=1, keepdims=True))
        P = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    else:               # any stored values: the method uses probs as given
        P = rng.uniform(0.0, 2.0 / max(L, 1), size=(H, L)).astype(np.float32)
    return q, K, V, P, dout, scale


def _check(name, got, ref):
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    mag = float(np.max(np.abs(ref))) if ref.size else 0.0
    assert err <= TOL * mag + 1e-30, f"{name}: max err {err:.3e} vs {TOL} * {mag:.3e}"


CASES = [(1, 4, 2, 32), (2, 4, 4, 64), (63, 8, 2, 32), (65, 8, 2, 128), (333, 6, 3, 96),
         (1000, 32, 8, 128), (4097, 32, 1, 128), (50, 16, 16, 64), (777, 64, 2, 64)]


@pytest.mark.parametrize("L,H,Hk,d", CASES)
def test_decode_backward_matches_oracle(ga, L, H, Hk, d):
    q, K, V, P, dout, scale = _inputs(L, H, Hk, d, seed=L * 13 + H + d)
    rs, rq, rk, rv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    t = [torch.from_numpy(a).cuda() for a in (q, K, V, P, dout)]
    ds, dq, dk, dv = ga.attn_decode_bwd(*t, H, Hk, d, scale)
    torch.cuda.synchronize()
    _check("d_scores", ds.cpu().numpy(), rs)
    _check("d_q", dq.cpu().numpy(), rq)
    _check("d_k_hist", dk.cpu().numpy(), rk)
    _check("d_v_hist", dv.cpu().numpy(), rv)


def test_decode_backward_arbitrary_probs_and_accumulation(ga):
    L, H, Hk, d = 517, 8, 2, 128
    q, K, V, P, dout, scale = _inputs(L, H, Hk, d, seed=5, softmax_probs=False)
    rs, rq, rk, rv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    rng = np.random.default_rng(6)
    q0 = rng.standard_normal(H * d, dtype=np.float32)
    k0 = rng.standard_normal((L, Hk * d), dtype=np.float32)
    v0 = rng.standard_normal((L, Hk * d), dtype=np.float32)
    t = [torch.from_numpy(a).cuda() for a in (q, K, V, P, dout)]
    dq, dk, dv = (torch.from_numpy(a.copy()).cuda() for a in (q0, k0, v0))
    ds = torch.full((H, L), float("nan"), device="cuda")          # overwritten
    ga.attn_decode_bwd(*t, H, Hk, d, scale, d_q=dq, d_k_hist=dk, d_v_hist=dv, d_scores=ds)
    torch.cuda.synchronize()
    _check("d_scores", ds.cpu().numpy(), rs)
    _check("d_q (+=)", dq.cpu().numpy() - q0, rq)
    _check("d_k_hist (+=)", dk.cpu().numpy() - k0, rk)
    _check("d_v_hist (+=)", dv.cpu().numpy() - v0, rv)


def test_decode_backward_full_size(ga):
    """The decode shape of the 16k workload: one query of each of 32 heads
    against 16384 cached keys of 8 kv heads, d = 128 (all outputs compared)."""
    L, H, Hk, d = 16384, 32, 8, 128
    q, K, V, P, dout, scale = _inputs(L, H, Hk, d, seed=16384)
    rs, rq, rk, rv = oracle.decode_bwd(q, K, V, P, dout, H, Hk, d, scale)
    t = [torch.from_numpy(a).cuda() for a in (q, K, V, P, dout)]
    ds, dq, dk, dv = ga.attn_decode_bwd(*t, H, Hk, d, scale)
    torch.cuda.synchronize()
    _check("d_scores", ds.cpu().numpy(), rs)
    _check("d_q", dq.cpu().numpy(), rq)
    _check("d_k_hist", dk.cpu().numpy(), rk)
    _check("d_v_hist", dv.cpu().numpy(), rv)
    # and the sum over keys of d_scores vanishes (probs sum to one)
    assert float(np.max(np.abs(ds.cpu().numpy().astype(np.float64).sum(axis=1)))) < 1e-3 * float(np.max(np.abs(rs)))
