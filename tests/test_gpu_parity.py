"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.

Acceptance (per output tensor): max|gpu - oracle| <= 5e-3 * max|oracle|, the
bound of each tensor taken from that tensor alone. The one exception is a
tensor whose exact value is zero everywhere (seq_len 1: dQ = dK = 0): its
bound uses the magnitude of dV instead, since the GPU only reaches zero up to
fp32 rounding of P = exp(s - LSE) ~ 1 (zero_ref below).
"""
import math

import numpy as np
import pytest

import oracle
import workloads

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _seg_dev(seg):
    return _dev(np.asarray(seg, dtype=np.int32))


def assert_parity(name, got, ref, zero_ref=None):
    """Per-tensor bound. Pass zero_ref only for a tensor whose exact value is
    zero everywhere (seq_len 1: dQ, dK): it has no magnitude of its own (the
    oracle, fed the fp32 LSE, gives ~1e-8 there, not 0), so the bound takes
    the magnitude of zero_ref (dV) instead."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    mag = float(np.max(np.abs(ref))) if ref.size else 0.0
    if zero_ref is not None:
        mag = max(mag, float(np.max(np.abs(zero_ref))))
    err = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    assert err <= TOL * mag, f"{name}: max|gpu-oracle| = {err:.3e} > {TOL} * {mag:.3e}"
    return err / mag if mag else 0.0


class short_path_off:
    """attn_bwd and its variants with the single-launch short path switched
    off: shapes it would take run the tensor-core (or CUDA-core) kernels."""

    def __init__(self, ga, off=True):
        self.ga, self.off = ga, off

    def __enter__(self):
        self.prev = self.ga.set_short_path(not self.off)

    def __exit__(self, *exc):
        self.ga.set_short_path(self.prev)


def short_ok(S, H, d):
    """The shapes attn_bwd_short accepts (its documented limits)."""
    nt = (S + 31) // 32
    hp = 32 if d <= 32 else (64 if d <= 64 else 128)
    return 1 <= S <= 2048 and nt * (nt + 1) // 2 * 1024 * H * hp <= 1 << 27


def gpu_bwd(ga, fn, x, lse32, init=None, calls=1):
    """fn: an entry point of the binding, or "attn_bwd_tc" = attn_bwd with the
    short path switched off."""
    if fn == "attn_bwd_tc":
        with short_path_off(ga):
            return gpu_bwd(ga, "attn_bwd", x, lse32, init, calls)
    S, H, Hk, d = x["seq_len"], x["n_heads"], x["n_kv_heads"], x["head_dim"]
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    if init is None:
        dQ = torch.zeros(S, H * d, device="cuda")
        dK = torch.zeros(S, Hk * d, device="cuda")
        dV = torch.zeros(S, Hk * d, device="cuda")
    else:
        dQ, dK, dV = (_dev(a.astype(np.float32)) for a in init)
    seg, LSE = _seg_dev(x["seg"]), _dev(lse32)
    ws = None
    for _ in range(calls):
        ws = getattr(ga, fn)(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, dQ, dK, dV, H, Hk, d,
                             x["scale"], workspace=ws)
    ga.read_device_status(ws)
    torch.cuda.synchronize()
    return dQ.cpu().numpy(), dK.cpu().numpy(), dV.cpu().numpy()


_REF = {}


def reference(name):
    """Inputs, fp32 LSE from the oracle forward, and the oracle backward."""
    if name not in _REF:
        w = workloads.WORKLOADS[name]
        x = workloads.make_inputs(w)
        O, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], w.n_heads, w.n_kv_heads,
                            w.head_dim, w.scale)
        lse32 = lse.astype(np.float32)
        g = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], w.n_heads,
                       w.n_kv_heads, w.head_dim, w.scale)
        _REF[name] = (x, O, lse, lse32, g)
    return _REF[name]


BWD_FNS = ["attn_bwd", "attn_bwd_tc", "attn_bwd_simt", "attn_bwd_short"]


@pytest.mark.parametrize("fn", BWD_FNS)
@pytest.mark.parametrize("name", ["tiny", "causal512", "docs2k", "docs4k"])
def test_backward_matches_oracle(ga, name, fn):
    w = workloads.WORKLOADS[name]
    if fn == "attn_bwd_short" and not short_ok(w.seq_len, w.n_heads, w.head_dim):
        pytest.skip("beyond the short path's limits")
    x, _, _, lse32, (rq, rk, rv) = reference(name)
    dQ, dK, dV = gpu_bwd(ga, fn, x, lse32)
    assert_parity("dQ", dQ, rq)
    assert_parity("dK", dK, rk)
    assert_parity("dV", dV, rv)


def gpu_fwd(ga, fn, x):
    """The forward through attn_fwd (tensor cores where built; device status
    checked) or attn_fwd_lse (CUDA cores, no workspace)."""
    S, H, Hk, d = x["seq_len"], x["n_heads"], x["n_kv_heads"], x["head_dim"]
    args = (_dev(x["Q"]), _dev(x["K"]), _dev(x["V"]), _seg_dev(x["seg"]), H, Hk, d, x["scale"])
    if fn == "attn_fwd":
        ws = torch.empty(int(ga.lib().attn_fwd_workspace_bytes(S, H, Hk, d)), dtype=torch.uint8,
                         device="cuda")
        O, LSE = ga.attn_fwd(*args, workspace=ws)
        ga.read_device_status(ws)
    else:
        O, LSE = ga.attn_fwd_lse(*args)
    torch.cuda.synchronize()
    return O.cpu().numpy(), LSE.cpu().numpy()


@pytest.mark.parametrize("fn", ["attn_fwd", "attn_fwd_lse"])
@pytest.mark.parametrize("name", ["tiny", "causal512", "docs2k", "docs4k"])
def test_forward_matches_oracle(ga, name, fn):
    x, O_ref, lse_ref, _, _ = reference(name)
    O, LSE = gpu_fwd(ga, fn, x)
    assert_parity("O", O, O_ref)
    assert_parity("LSE", LSE, lse_ref)


@pytest.mark.parametrize("S,H,Hk,d,seg_kind", [
    (1, 4, 2, 32, "causal"), (65, 8, 2, 128, "docs"), (127, 4, 1, 32, "nonmonotone"),
    (129, 6, 3, 64, "docs"), (333, 16, 2, 64, "nonmonotone"), (97, 4, 2, 100, "docs"),
    (300, 8, 1, 128, "docs"), (513, 4, 2, 32, "docs"), (200, 32, 1, 128, "causal")])
def test_forward_edge_shapes(ga, S, H, Hk, d, seg_kind):
    """attn_fwd on ragged tails, documents, non-monotone seg, G up to 32, the
    CUDA-core fallback (d = 100) and seq_len 1."""
    x = _edge_inputs(S, H, Hk, d, seg_kind, seed=S * 17 + d)
    O_ref, lse_ref = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, x["scale"])
    O, LSE = gpu_fwd(ga, "attn_fwd", x)
    assert_parity("O", O, O_ref)
    assert_parity("LSE", LSE, lse_ref)


@pytest.mark.parametrize("S,H,Hk,d,seg_kind", [(1000, 8, 2, 128, "causal"), (700, 4, 1, 64, "docs"),
                                               (513, 4, 4, 32, "causal")])
def test_forward_growing_scores(ga, S, H, Hk, d, seg_kind):
    """attn_fwd where a row's running max keeps growing past the first chunks:
    key j is scaled by 0.1 + 4 j / S, so the scores of later keys exceed the
    early maxima by far more than 2^8 (in log2 units) and the online softmax
    raises its max and rescales its O accumulators mid-row, repeatedly."""
    x = _edge_inputs(S, H, Hk, d, seg_kind, seed=S + d)
    grow = (0.1 + 4.0 * np.arange(S) / S).astype(np.float32)[:, None]
    x["K"] = (x["K"] * grow).astype(np.float32)
    O_ref, lse_ref = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, x["scale"])
    O, LSE = gpu_fwd(ga, "attn_fwd", x)
    assert_parity("O", O, O_ref)
    assert_parity("LSE", LSE, lse_ref)


def _edge_inputs(S, H, Hk, d, seg_kind, seed):
    rng = np.random.default_rng(seed)
    if seg_kind == "causal":
        seg = np.zeros(S, np.uint32)
    else:
        seg = workloads.random_seg(S, rng, monotone=(seg_kind == "docs"))
    f = lambda c: rng.standard_normal((S, c), dtype=np.float32)  # noqa: E731
    return {"Q": f(H * d), "K": f(Hk * d), "V": f(Hk * d), "dO": f(H * d), "seg": seg,
            "scale": 1.0 / math.sqrt(d), "seq_len": S, "n_heads": H, "n_kv_heads": Hk,
            "head_dim": d}


EDGE = [
    (1, 4, 2, 32, "causal"), (2, 4, 4, 64, "causal"), (65, 8, 2, 128, "docs"),
    (127, 4, 1, 32, "nonmonotone"), (129, 6, 3, 64, "docs"), (200, 8, 8, 128, "causal"),
    (333, 16, 2, 64, "nonmonotone"), (97, 4, 2, 100, "docs"), (64, 2, 1, 16, "causal"),
    (300, 8, 1, 128, "docs"), (513, 4, 2, 32, "docs"), (256, 16, 2, 128, "causal"),
    # wide groups: at d = 128 a key-major Q sub-tile of 16 rows is one query's
    # 16 heads (G = 16) or half of one query's heads (G = 32); G = 64 at d = 64
    # is too wide for the SM-pair key-major kernel and runs on one SM
    (90, 16, 1, 128, "docs"), (160, 32, 1, 128, "causal"), (70, 64, 1, 64, "nonmonotone"),
]


@pytest.mark.parametrize("fn", BWD_FNS)
@pytest.mark.parametrize("S,H,Hk,d,seg_kind", EDGE)
def test_edge_shapes(ga, S, H, Hk, d, seg_kind, fn):
    if fn == "attn_bwd_short" and not short_ok(S, H, d):
        pytest.skip("beyond the short path's limits")
    x = _edge_inputs(S, H, Hk, d, seg_kind, seed=S * 31 + d)
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, x["scale"])
    lse32 = lse.astype(np.float32)
    rq, rk, rv = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], H, Hk, d, x["scale"])
    dQ, dK, dV = gpu_bwd(ga, fn, x, lse32)
    exact_zero = rv if S == 1 else None     # seq_len 1: the exact dQ and dK are zero
    assert_parity("dQ", dQ, rq, zero_ref=exact_zero)
    assert_parity("dK", dK, rk, zero_ref=exact_zero)
    assert_parity("dV", dV, rv)


@pytest.mark.parametrize("S,H,Hk,d,seg_kind", [
    (2000, 2, 1, 32, "docs"),            # 63 tiles, 2^26.98 multiply-adds per contraction
    (2048, 1, 1, 32, "causal"),          # seq_len 2048: all 64 query tiles
    (900, 2, 1, 64, "nonmonotone"), (33, 8, 4, 128, "causal"), (31, 3, 1, 8, "docs")])
def test_short_path_limits(ga, S, H, Hk, d, seg_kind):
    """attn_bwd_short near its work limit (2^27 multiply-adds per contraction)
    and at odd sizes, against the oracle; just past the limit it refuses."""
    assert short_ok(S, H, d)
    x = _edge_inputs(S, H, Hk, d, seg_kind, seed=S * 3 + d)
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, x["scale"])
    lse32 = lse.astype(np.float32)
    rq, rk, rv = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], H, Hk, d, x["scale"])
    dQ, dK, dV = gpu_bwd(ga, "attn_bwd_short", x, lse32)
    assert_parity("dQ", dQ, rq)
    assert_parity("dK", dK, rk)
    assert_parity("dV", dV, rv)
    S2 = S + 32 * 8 if S < 2000 else 2049
    if not short_ok(S2, H, d):
        y = _edge_inputs(S2, H, Hk, d, seg_kind, seed=1)
        with pytest.raises(ga.GqaError) as e:
            gpu_bwd(ga, "attn_bwd_short", y, np.zeros((S2, H), np.float32))
        assert e.value.status == 2


@pytest.mark.parametrize("fn", BWD_FNS)
def test_gradients_accumulate(ga, fn):
    """+= semantics: two calls on non-zero initial gradients give init + 2 * grad."""
    x, _, _, lse32, (rq, rk, rv) = reference("causal512")
    rng = np.random.default_rng(5)
    init = [rng.standard_normal(a.shape) for a in (rq, rk, rv)]
    dQ, dK, dV = gpu_bwd(ga, fn, x, lse32, init=init, calls=2)
    assert_parity("dQ", dQ, init[0].astype(np.float32) + 2 * rq)
    assert_parity("dK", dK, init[1].astype(np.float32) + 2 * rk)
    assert_parity("dV", dV, init[2].astype(np.float32) + 2 * rv)


@pytest.mark.parametrize("fn", BWD_FNS)
def test_seq_len_one(ga, fn):
    x = _edge_inputs(1, 8, 2, 64, "causal", seed=1)
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], 8, 2, 64, x["scale"])
    dQ, dK, dV = gpu_bwd(ga, fn, x, lse.astype(np.float32))
    want_v = np.stack([x["dO"][0].reshape(8, 64)[4 * g:4 * g + 4].sum(0) for g in range(2)]).reshape(1, -1)
    assert_parity("dV", dV, want_v)
    assert_parity("dQ", dQ, np.zeros_like(dQ), zero_ref=want_v)
    assert_parity("dK", dK, np.zeros_like(dK), zero_ref=want_v)


@pytest.mark.parametrize("pos_offset", [0, 100000])
def test_rope_backward_matches_oracle(ga, pos_offset):
    rng = np.random.default_rng(pos_offset + 3)
    S, H, d = 300, 5, 64
    X = rng.standard_normal((S, H * d), dtype=np.float32)
    t = _dev(X)
    ga.rope_bwd_inplace(t, H, d, pos_offset=pos_offset, base=10000.0)
    torch.cuda.synchronize()
    ref = oracle.rope_bwd(X, H, d, pos_offset=pos_offset, base=10000.0)
    got = t.cpu().numpy()
    assert np.max(np.abs(got - ref)) <= 2e-6 * np.max(np.abs(ref))


FUSED_ROPE = [
    (300, 8, 2, 128, "docs", 0), (200, 16, 4, 64, "causal", 7), (129, 4, 2, 32, "nonmonotone", 0),
    (97, 4, 2, 100, "docs", 0), (256, 8, 2, 128, "causal", 40000), (65, 4, 1, 64, "docs", 40000),
]


@pytest.mark.parametrize("short", [True, False])
@pytest.mark.parametrize("S,H,Hk,d,seg_kind,pos", FUSED_ROPE)
def test_fused_rope_backward_matches_oracle(ga, S, H, Hk, d, seg_kind, pos, short):
    """attn_bwd_rope: dQ += R^T(attention dQ), dK += R^T(attention dK), dV += dV
    on non-zero initial gradients (only the new contribution is rotated);
    tensor-core shapes and a CUDA-core one (d = 100), both angle paths, with
    the short path allowed (it takes these shapes) and switched off."""
    with short_path_off(ga, off=not short):
        _fused_rope_case(ga, S, H, Hk, d, seg_kind, pos)


def _fused_rope_case(ga, S, H, Hk, d, seg_kind, pos):
    x = _edge_inputs(S, H, Hk, d, seg_kind, seed=S * 7 + d + pos)
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, x["scale"])
    lse32 = lse.astype(np.float32)
    rq, rk, rv = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], H, Hk, d, x["scale"])
    rng = np.random.default_rng(S + pos)
    init = [rng.standard_normal(a.shape).astype(np.float32) for a in (rq, rk, rv)]
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    dQ, dK, dV = (_dev(a) for a in init)
    ws = ga.attn_bwd_rope(t["Q"], t["K"], t["V"], t["dO"], _dev(lse32), _seg_dev(x["seg"]),
                          dQ, dK, dV, H, Hk, d, x["scale"], pos_offset=pos, base=10000.0)
    ga.read_device_status(ws)
    torch.cuda.synchronize()
    want_q = init[0] + oracle.rope_bwd(rq, H, d, pos_offset=pos, base=10000.0)
    want_k = init[1] + oracle.rope_bwd(rk, Hk, d, pos_offset=pos, base=10000.0)
    assert_parity("dQ", dQ.cpu().numpy() - init[0], want_q - init[0])
    assert_parity("dK", dK.cpu().numpy() - init[1], want_k - init[1])
    assert_parity("dV", dV.cpu().numpy() - init[2], rv)


@pytest.mark.parametrize("name", ["causal512", "docs2k", "docs4k"])
def test_backward_given_o_matches_oracle(ga, name):
    """attn_bwd_o: D from the row dot dO . O (O from the oracle forward,
    rounded to fp32) instead of the D pass; same result as attn_bwd."""
    x, O_ref, _, lse32, (rq, rk, rv) = reference(name)
    S, H, Hk, d = x["seq_len"], x["n_heads"], x["n_kv_heads"], x["head_dim"]
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    out = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
    with short_path_off(ga):   # the tensor-core kernels' given-O path at every size
        ws = ga.attn_bwd_o(t["Q"], t["K"], t["V"], t["dO"], _dev(O_ref.astype(np.float32)),
                           _dev(lse32), _seg_dev(x["seg"]), *out, H, Hk, d, x["scale"])
    ga.read_device_status(ws)
    torch.cuda.synchronize()
    for nm, g, r in (("dQ", out[0], rq), ("dK", out[1], rk), ("dV", out[2], rv)):
        assert_parity(nm, g.cpu().numpy(), r)


@pytest.mark.parametrize("short", [True, False])
@pytest.mark.parametrize("S,H,Hk,d,seg_kind", [(300, 8, 2, 128, "docs"), (129, 4, 2, 32, "nonmonotone"),
                                               (97, 4, 2, 100, "docs"), (200, 16, 4, 64, "causal")])
def test_backward_given_o_from_gpu_forward(ga, S, H, Hk, d, seg_kind, short):
    """attn_bwd_o fed this library's own forward (O, LSE), on non-zero initial
    gradients, against the oracle backward with the same fp32 LSE (with the
    short path allowed, which forms D itself, and switched off)."""
    with short_path_off(ga, off=not short):
        _given_o_case(ga, S, H, Hk, d, seg_kind)


def _given_o_case(ga, S, H, Hk, d, seg_kind):
    x = _edge_inputs(S, H, Hk, d, seg_kind, seed=S * 13 + d)
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    seg = _seg_dev(x["seg"])
    O, LSE = ga.attn_fwd_lse(t["Q"], t["K"], t["V"], seg, H, Hk, d, x["scale"])
    torch.cuda.synchronize()
    lse32 = LSE.cpu().numpy()
    rq, rk, rv = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], H, Hk, d, x["scale"])
    rng = np.random.default_rng(S)
    init = [rng.standard_normal(a.shape).astype(np.float32) for a in (rq, rk, rv)]
    out = [_dev(a) for a in init]
    ws = ga.attn_bwd_o(t["Q"], t["K"], t["V"], t["dO"], O, LSE, seg, *out, H, Hk, d, x["scale"])
    ga.read_device_status(ws)
    torch.cuda.synchronize()
    for nm, g, r, i0 in (("dQ", out[0], rq, init[0]), ("dK", out[1], rk, init[1]), ("dV", out[2], rv, init[2])):
        assert_parity(nm, g.cpu().numpy() - i0, r)


@pytest.mark.parametrize("short", [True, False])
def test_backward_captured_in_cuda_graph(ga, short):
    """attn_bwd captured in a CUDA graph (with the gradients' zeroing) and
    replayed twice: the short path's cooperative launch and the tensor-core
    kernels' cluster launches replay to the oracle's result each time."""
    x, _, _, lse32, (rq, rk, rv) = reference("causal512")
    S, H, Hk, d, sc = x["seq_len"], x["n_heads"], x["n_kv_heads"], x["head_dim"], x["scale"]
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    seg, LSE = _seg_dev(x["seg"]), _dev(lse32)
    out = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
    with short_path_off(ga, off=not short):
        ws = torch.empty(ga.workspace_bytes(S, H, Hk, d), dtype=torch.uint8, device="cuda")

        def step():
            for o in out:
                o.zero_()
            ga.attn_bwd(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *out, H, Hk, d, sc, workspace=ws)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()                       # first call outside capture (one-time set-up)
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        for _ in range(2):
            for o in out:
                o.fill_(7.0)             # replays must overwrite this through their own zeroing
            g.replay()
            torch.cuda.synchronize()
            ga.read_device_status(ws)
            for nm, got, r in (("dQ", out[0], rq), ("dK", out[1], rk), ("dV", out[2], rv)):
                assert_parity(nm, got.cpu().numpy(), r)


DETERMINISM = [("attn_bwd_tc", "docs2k"), ("attn_bwd_tc", "docs4k"), ("attn_bwd_short", "causal512"),
               ("attn_bwd_short", "tiny"), ("attn_bwd_simt", "docs2k"), ("attn_bwd", "causal512")]


@pytest.mark.parametrize("fn,name", DETERMINISM)
def test_backward_is_deterministic(ga, fn, name):
    """No atomics on any gradient and every partial sum reduced in a fixed
    order: two calls on the same inputs into freshly zeroed gradients give
    bit-identical dQ, dK, dV (the packed 2k documents split the key-major
    walk into parts that km_split_reduce adds in order)."""
    x, _, _, lse32, _ = reference(name)
    a = gpu_bwd(ga, fn, x, lse32)
    b = gpu_bwd(ga, fn, x, lse32)
    for nm, u, v in zip(("dQ", "dK", "dV"), a, b):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32)), f"{nm} differs between runs"


@pytest.mark.parametrize("short", [True, False])
def test_fused_rope_backward_is_deterministic(ga, short):
    """attn_bwd_rope twice on the same inputs: bit-identical gradients."""
    x, _, _, lse32, _ = reference("docs2k")
    S, H, Hk, d = x["seq_len"], x["n_heads"], x["n_kv_heads"], x["head_dim"]
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    seg, LSE = _seg_dev(x["seg"]), _dev(lse32)
    runs = []
    with short_path_off(ga, off=not short):
        for _ in range(2):
            out = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
            ws = ga.attn_bwd_rope(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *out, H, Hk, d,
                                  x["scale"], pos_offset=3, base=10000.0)
            ga.read_device_status(ws)
            runs.append([o.cpu().numpy() for o in out])
    for nm, u, v in zip(("dQ", "dK", "dV"), *runs):
        assert np.array_equal(u.view(np.uint32), v.view(np.uint32)), f"{nm} differs between runs"
