"""attn_bwd_noalloc: the backward for callers that cannot allocate device
memory (a plugin given only its I/O buffers, a process whose memory manager
forbids raw cudaMalloc, a binding without a device allocator). It uses a fixed
scratch array inside the library instead of a caller workspace.

Collected last on purpose: the GPU test runs after every other test when the
whole suite runs, and also passes alone in a fresh process.
"""
import math

import numpy as np
import pytest

import workloads

TOL = 5e-3
FAKE = 0x10000   # aligned, non-null; never dereferenced (the size check fails first)


def _lib():
    from causal_gqa_attention_attn_gb300 import build
    build.build()
    import causal_gqa_attention_attn_gb300 as ga
    return ga, ga.lib()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    _, L = _lib()
    # 65536 x 64 needs 16 MiB of scratch: refused on the host, nothing launched
    r = L.attn_bwd_noalloc(*([FAKE] * 9), 65536, 64, 8, 64, 0.125, None)
    assert r == 2
    assert "scratch" in L.gqa_last_error().decode()
    assert L.attn_bwd_noalloc(*([FAKE] * 9), 64, 6, 4, 32, 0.2, None) == 1
    assert L.attn_bwd_noalloc(*([FAKE] * 9), 0, 4, 2, 32, 0.2, None) == 0


def _case(S, H, Hk, d, seed, docs):
    rng = np.random.default_rng(seed)
    seg = workloads.random_seg(S, rng) if docs else np.zeros(S, np.uint32)
    f = lambda c: rng.standard_normal((S, c), dtype=np.float32)  # noqa: E731
    return dict(Q=f(H * d), K=f(Hk * d), V=f(Hk * d), dO=f(H * d), seg=seg, S=S, H=H, Hk=Hk,
                d=d, scale=1.0 / math.sqrt(d))


@pytest.mark.gpu
def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls():
    """Two calls in a row on each shape: both match the fp64 oracle (per-tensor
    bound) and the workspace entry point attn_bwd_simt, and the second call,
    which finds the first call's contents in the shared scratch array, gives
    the same bits as the first."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    ga, L = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    for case in (_case(512, 8, 2, 64, 1, docs=False), _case(777, 16, 4, 128, 2, docs=True)):
        t = {k: torch.from_numpy(case[k]).cuda() for k in ("Q", "K", "V", "dO")}
        seg = torch.from_numpy(case["seg"].astype(np.int32)).cuda()
        S, H, Hk, d, sc = case["S"], case["H"], case["Hk"], case["d"], case["scale"]
        _, lse = oracle.fwd(case["Q"], case["K"], case["V"], case["seg"], H, Hk, d, sc)
        lse32 = lse.astype(np.float32)
        want = oracle.bwd(case["Q"], case["K"], case["V"], case["dO"], lse32, case["seg"], H, Hk,
                          d, sc)
        LSE = torch.from_numpy(lse32).cuda()
        ref = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
        ga.attn_bwd_simt(t["Q"], t["K"], t["V"], t["dO"], LSE, seg, *ref, H, Hk, d, sc)
        ref = [r.cpu().numpy().astype(np.float64) for r in ref]
        calls = []
        for _ in range(2):
            got = [torch.zeros(S, n * d, device="cuda") for n in (H, Hk, Hk)]
            status = L.attn_bwd_noalloc(t["Q"].data_ptr(), t["K"].data_ptr(), t["V"].data_ptr(),
                                        t["dO"].data_ptr(), LSE.data_ptr(), seg.data_ptr(),
                                        got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                                        S, H, Hk, d, sc, stream)
            assert status == 0, L.gqa_last_error().decode()
            torch.cuda.synchronize()
            got = [g.cpu().numpy() for g in got]
            for name, g, r, o in zip(("dQ", "dK", "dV"), got, ref, want):
                g64 = g.astype(np.float64)
                assert np.all(np.isfinite(g64))
                for what, target in (("oracle", o), ("attn_bwd_simt", r)):
                    err, mag = np.max(np.abs(g64 - target)), np.max(np.abs(target))
                    assert err <= TOL * mag, f"{name} vs {what}: {err:.3e} > {TOL} * {mag:.3e}"
            calls.append(got)
        for name, a, b in zip(("dQ", "dK", "dV"), *calls):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), f"{name}: calls differ"
