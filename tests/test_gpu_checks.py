"""Stand-ins for a memory checker (compute-sanitizer is not used here).

1. The debug build, libgqa_attn_checks.so (the same sources compiled with
   -DGQA_CHECKS): device-side checks of the seg precondition (seg[s] <= s)
   and of the kernels' load / store indices and TMA box coordinates, which set
   a bit in the workspace status word and skip the access instead of
   trapping. On valid inputs it must match the oracle with a clean status
   word; on a seg that breaks the precondition it must report
   GQA_ERR_DEVICE_CHECK with the seg bit. (The pages' counterparts are the
   defensive clamps and uniform-control-flow guards of
   backward_attention.wgsl, attention_backward_short and attention_backward.)
2. Canaries (release build): every output buffer and the workspace sit
   between guard regions filled with a known pattern; after each entry point
   the guards must be untouched (no write outside the buffers it was given).
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


def _inputs(S, H, Hk, d, seg_kind, seed):
    rng = np.random.default_rng(seed)
    if seg_kind == "causal":
        seg = np.zeros(S, np.uint32)
    else:
        seg = workloads.random_seg(S, rng, monotone=(seg_kind == "docs"))
    f = lambda c: rng.standard_normal((S, c), dtype=np.float32)  # noqa: E731
    return {"Q": f(H * d), "K": f(Hk * d), "V": f(Hk * d), "dO": f(H * d), "seg": seg,
            "scale": 1.0 / math.sqrt(d)}


def _parity(name, got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), name
    err, mag = float(np.max(np.abs(got - ref))), float(np.max(np.abs(ref)))
    assert err <= TOL * mag, f"{name}: {err:.3e} > {TOL} * {mag:.3e}"


CHECK_SHAPES = [(65, 8, 2, 128, "docs"), (127, 4, 1, 32, "nonmonotone"), (300, 8, 1, 128, "docs"),
                (97, 4, 2, 100, "docs"), (160, 32, 1, 128, "causal"), (2048, 16, 4, 64, "docs"),
                (513, 4, 2, 32, "docs")]


@pytest.mark.parametrize("path", ["tc", "short", "simt"])
@pytest.mark.parametrize("S,H,Hk,d,seg_kind", CHECK_SHAPES)
def test_checks_build_matches_oracle(ga, S, H, Hk, d, seg_kind, path):
    """The debug build on valid inputs: oracle parity and a clean status word
    (every device-side check passed) on the tensor-core, short and CUDA-core
    paths, including a split key-tile walk (2048 tokens, packed documents)."""
    x = _inputs(S, H, Hk, d, seg_kind, seed=S * 5 + d)
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, x["scale"])
    lse32 = lse.astype(np.float32)
    rq, rk, rv = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], H, Hk, d, x["scale"])
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    seg, LSE = _dev(x["seg"].astype(np.int32)), _dev(lse32)
    out = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
    with ga.checks_build():
        if path == "short":
            nt = (S + 31) // 32
            hp = 32 if d <= 32 else (64 if d <= 64 else 128)
            if not (S <= 2048 and nt * (nt + 1) // 2 * 1024 * H * hp <= 1 << 27):
                pytest.skip("beyond the short path's limits")
            fn = ga.attn_bwd_short
        else:
            fn = ga.attn_bwd_simt if path == "simt" else ga.attn_bwd
        prev = ga.set_short_path(False)
        try:
            ws = fn(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *out, H, Hk, d, x["scale"])
            ga.read_device_status(ws)          # raises on any failed device-side check
        finally:
            ga.set_short_path(prev)
        if path == "tc":                       # the forward of the debug build as well
            O, LSE2 = ga.attn_fwd(t["Q"], t["K"], t["V"], seg, H, Hk, d, x["scale"])
            torch.cuda.synchronize()
    for nm, g, r in (("dQ", out[0], rq), ("dK", out[1], rk), ("dV", out[2], rv)):
        _parity(nm, g.cpu().numpy(), r)
    if path == "tc":
        _parity("LSE", LSE2.cpu().numpy(), lse)


@pytest.mark.parametrize("path", ["tc", "short", "simt"])
def test_checks_build_flags_seg_precondition(ga, path):
    """seg[s] = s + 1 at two positions (every value still inside the
    sequence, so nothing reads out of bounds: those rows just see no key):
    the debug build reports GQA_ERR_DEVICE_CHECK with the seg bit (0x1) and
    no other; the release build does not check (clean status word)."""
    S, H, Hk, d = 200, 8, 2, 64
    x = _inputs(S, H, Hk, d, "causal", seed=11)
    seg_np = x["seg"].copy()
    seg_np[[5, 77]] = [6, 78]
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    seg, LSE = _dev(seg_np.astype(np.int32)), torch.zeros(S, H, device="cuda")
    fn = {"tc": "attn_bwd", "short": "attn_bwd_short", "simt": "attn_bwd_simt"}[path]

    def run():
        out = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
        prev = ga.set_short_path(False)    # attn_bwd: the tensor-core kernels at this size
        try:
            return getattr(ga, fn)(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *out, H, Hk, d,
                                   x["scale"])
        finally:
            ga.set_short_path(prev)

    with ga.checks_build():
        ws = run()
        with pytest.raises(ga.GqaError) as e:
            ga.read_device_status(ws)
    assert e.value.status == 5
    assert "0x40000001" in str(e.value), str(e.value)
    ga.read_device_status(run())


# ---------------------------------------------------------------------------
# canaries
# ---------------------------------------------------------------------------
GUARD = 4096                       # 16 KB of guard on each side
PATTERN = 0x7FC0DEAD               # a NaN bit pattern no kernel writes


class Guarded:
    """A float32 (or uint8) device buffer of n elements between two guard
    regions that hold PATTERN (0xA5 bytes for uint8)."""

    def __init__(self, n, dtype=torch.float32, init=None):
        if dtype == torch.uint8:
            self.buf = torch.full((n + 8 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
            self.g = 4 * GUARD
            self.t = self.buf[self.g:self.g + n]
        else:
            self.buf = torch.full((n + 2 * GUARD,), PATTERN, dtype=torch.int32, device="cuda")
            self.g = GUARD
            self.t = self.buf.view(torch.float32)[GUARD:GUARD + n]
            self.t.zero_() if init is None else self.t.copy_(init.reshape(-1))

    def check(self, name):
        torch.cuda.synchronize()
        want = 0xA5 if self.buf.dtype == torch.uint8 else PATTERN
        lo, hi = self.buf[:self.g], self.buf[self.g + self.t.numel():]
        assert bool((lo == want).all()), f"{name}: guard before the buffer overwritten"
        assert bool((hi == want).all()), f"{name}: guard after the buffer overwritten"


def _bwd_case(ga, fn, S, H, Hk, d, seg_kind, **kw):
    x = _inputs(S, H, Hk, d, seg_kind, seed=S + d)
    t = {k: _dev(x[k]) for k in ("Q", "K", "V", "dO")}
    seg = _dev(x["seg"].astype(np.int32))
    _, LSE = ga.attn_fwd_lse(t["Q"], t["K"], t["V"], seg, H, Hk, d, x["scale"])
    outs = [Guarded(S * n * d) for n in (H, Hk, Hk)]
    views = [o.t.view(S, -1) for o in outs]
    ws = Guarded(ga.workspace_bytes(S, H, Hk, d), torch.uint8)
    if fn == "attn_bwd_o":
        O, _ = ga.attn_fwd_lse(t["Q"], t["K"], t["V"], seg, H, Hk, d, x["scale"])
        ga.attn_bwd_o(t["Q"], t["K"], t["V"], t["dO"], O, LSE, seg, *views, H, Hk, d, x["scale"],
                      workspace=ws.t)
    elif fn == "attn_bwd_rope":
        ga.attn_bwd_rope(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *views, H, Hk, d, x["scale"],
                         pos_offset=kw.get("pos", 0), base=10000.0, workspace=ws.t)
    else:
        getattr(ga, fn)(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *views, H, Hk, d, x["scale"],
                        workspace=ws.t)
    ga.read_device_status(ws.t)
    for nm, o in zip(("dQ", "dK", "dV"), outs):
        o.check(f"{fn} {nm}")
        assert bool(torch.isfinite(o.t).all()), f"{fn} {nm}: non-finite"
    ws.check(f"{fn} workspace")


CANARY = [
    ("attn_bwd", 2048, 16, 4, 64, "docs", False),   # tensor cores, split key-tile walk + part sums
    ("attn_bwd", 300, 8, 2, 128, "docs", False),    # tensor cores, ragged tail
    ("attn_bwd", 333, 16, 2, 64, "nonmonotone", True),   # the short path
    ("attn_bwd_short", 129, 6, 3, 64, "docs", True),
    ("attn_bwd_simt", 97, 4, 2, 100, "docs", True),
    ("attn_bwd_rope", 300, 8, 2, 128, "docs", False),
    ("attn_bwd_rope", 200, 16, 4, 64, "causal", True),
    ("attn_bwd_o", 300, 8, 2, 128, "docs", False),
    ("attn_bwd", 160, 32, 1, 128, "causal", False),   # one kv head, single-SM key-major kernel
]


@pytest.mark.parametrize("fn,S,H,Hk,d,seg_kind,short", CANARY)
def test_backward_writes_stay_inside_their_buffers(ga, fn, S, H, Hk, d, seg_kind, short):
    prev = ga.set_short_path(short)
    try:
        _bwd_case(ga, fn, S, H, Hk, d, seg_kind)
    finally:
        ga.set_short_path(prev)


@pytest.mark.parametrize("S,H,Hk,d", [(300, 8, 2, 128), (65, 4, 1, 64), (97, 4, 2, 100)])
def test_forward_writes_stay_inside_their_buffers(ga, S, H, Hk, d):
    x = _inputs(S, H, Hk, d, "docs", seed=S)
    t = {k: _dev(x[k]) for k in ("Q", "K", "V")}
    seg = _dev(x["seg"].astype(np.int32))
    O, LSE = Guarded(S * H * d), Guarded(S * H)
    ws = Guarded(int(ga.lib().attn_fwd_workspace_bytes(S, H, Hk, d)), torch.uint8)
    ga.attn_fwd(t["Q"], t["K"], t["V"], seg, H, Hk, d, x["scale"], O=O.t.view(S, -1),
                LSE=LSE.t.view(S, H), workspace=ws.t)
    ga.read_device_status(ws.t)
    O.check("attn_fwd O")
    LSE.check("attn_fwd LSE")
    ws.check("attn_fwd workspace")


def test_decode_and_rope_writes_stay_inside_their_buffers(ga):
    L, H, Hk, d = 1000, 8, 2, 128
    rng = np.random.default_rng(3)
    q = _dev(rng.standard_normal(H * d, dtype=np.float32))
    k = _dev(rng.standard_normal((L, Hk * d), dtype=np.float32))
    v = _dev(rng.standard_normal((L, Hk * d), dtype=np.float32))
    d_out = _dev(rng.standard_normal(H * d, dtype=np.float32))
    probs = torch.softmax(_dev(rng.standard_normal((H, L), dtype=np.float32)), dim=1).contiguous()
    dq, ds = Guarded(H * d), Guarded(H * L)
    dk, dv = Guarded(L * Hk * d), Guarded(L * Hk * d)
    ws = Guarded(int(ga.lib().attn_decode_bwd_workspace_bytes(L, H, Hk, d)), torch.uint8)
    ga.attn_decode_bwd(q, k, v, probs, d_out, H, Hk, d, 1.0 / math.sqrt(d), d_q=dq.t,
                       d_k_hist=dk.t.view(L, -1), d_v_hist=dv.t.view(L, -1),
                       d_scores=ds.t.view(H, L), workspace=ws.t)
    for nm, g in (("d_q", dq), ("d_scores", ds), ("d_k", dk), ("d_v", dv), ("workspace", ws)):
        g.check(f"attn_decode_bwd {nm}")
    X = Guarded(333 * 5 * 64, init=_dev(rng.standard_normal((333, 5 * 64), dtype=np.float32)))
    ga.rope_bwd_inplace(X.t.view(333, -1), 5, 64, pos_offset=40000, base=10000.0)
    X.check("rope_bwd_inplace")
