"""Device-side failure detection without a GPU fault: a bounded wait that runs
out reports GQA_ERR_DEVICE_TIMEOUT through the workspace status word, the
kernel returns, and the context keeps working (a backward after it is exact)."""
import math
import numpy as np
import pytest

import oracle
import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ga():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from causal_gqa_attention_attn_gb300 import build
    build.build()
    import causal_gqa_attention_attn_gb300 as mod
    return mod


def test_bounded_wait_reports_timeout_and_context_survives(ga):
    L = ga.lib()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert L.gqa_wait_selftest(ws.data_ptr(), ws.numel(), 2_000_000, stream) == 0
    with pytest.raises(ga.GqaError) as e:
        ga.read_device_status(ws)
    assert e.value.status == 4            # GQA_ERR_DEVICE_TIMEOUT
    word = int(ws[:4].view(torch.int32).item()) & 0xffffffff
    assert word & 0x80000000 and word & (1 << 12)
    # the context is still usable: a small backward afterwards matches the oracle
    x = workloads.make_inputs(workloads.WORKLOADS["tiny"])
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], 4, 2, 32, x["scale"])
    lse32 = lse.astype(np.float32)
    ref = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], 4, 2, 32, x["scale"])
    t = {k: torch.from_numpy(x[k]).cuda() for k in ("Q", "K", "V", "dO")}
    out = [torch.zeros(64, n, device="cuda") for n in (128, 64, 64)]
    w2 = ga.attn_bwd(t["Q"], t["K"], t["V"], t["dO"], torch.from_numpy(lse32).cuda(),
                     torch.from_numpy(x["seg"].astype(np.int32)).cuda(), *out, 4, 2, 32, x["scale"])
    ga.read_device_status(w2)                 # a fresh call clears the word
    for got, r in zip(out, ref):
        assert np.max(np.abs(got.cpu().numpy() - r)) <= 5e-3 * np.max(np.abs(r))


def test_selftest_rejects_bad_limits(ga):
    L = ga.lib()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    assert L.gqa_wait_selftest(ws.data_ptr(), ws.numel(), 0, None) == 1
    assert L.gqa_wait_selftest(ws.data_ptr(), 16, 1000, None) == 1


def test_grid_barrier_timeout_reports_and_context_survives(ga):
    """The short path's grid barrier: a wait for an arrival that never comes
    gives up after the limit, reports GQA_ERR_DEVICE_TIMEOUT (site bit 0x400),
    and a short-path backward afterwards is exact."""
    L = ga.lib()
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert L.gqa_grid_barrier_selftest(ws.data_ptr(), ws.numel(), 2_000_000, stream) == 0
    with pytest.raises(ga.GqaError) as e:
        ga.read_device_status(ws)
    assert e.value.status == 4
    word = int(ws[:4].view(torch.int32).item()) & 0xffffffff
    assert word & 0x80000000 and word & 0x400
    assert L.gqa_grid_barrier_selftest(ws.data_ptr(), ws.numel(), 0, stream) == 1
    x = workloads.make_inputs(workloads.WORKLOADS["causal512"])
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], 4, 2, 32, x["scale"])
    lse32 = lse.astype(np.float32)
    ref = oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, x["seg"], 4, 2, 32, x["scale"])
    t = {k: torch.from_numpy(x[k]).cuda() for k in ("Q", "K", "V", "dO")}
    out = [torch.zeros(512, n, device="cuda") for n in (128, 64, 64)]
    w2 = ga.attn_bwd_short(t["Q"], t["K"], t["V"], t["dO"], torch.from_numpy(lse32).cuda(),
                           torch.from_numpy(x["seg"].astype(np.int32)).cuda(), *out, 4, 2, 32,
                           x["scale"])
    ga.read_device_status(w2)
    for got, r in zip(out, ref):
        assert np.max(np.abs(got.cpu().numpy() - r)) <= 5e-3 * np.max(np.abs(r))
