"""Host-side logic of bench.py (no GPU): counted flops, peaks, clock parsing,
and the multi-rank timing reduction over a 2-rank gloo group on CPU."""
import os
import socket

import pytest

import bench
import workloads


def test_counted_flops_and_pairs():
    w = workloads.WORKLOADS["causal16k"]
    x = workloads.make_seg(w.seq_len, None, None, None)
    pairs = workloads.n_pairs(x)
    assert pairs == w.seq_len * (w.seq_len + 1) // 2 == 134225920
    assert bench.counted_flops(128, 32, pairs) == pytest.approx(5.4978936832e12)
    # nine executed contractions against five counted
    assert bench.executed_flops(128, 32, pairs) == pytest.approx(bench.counted_flops(128, 32, pairs) * 9 / 5)


def test_executed_contractions():
    assert bench.executed_contractions(128, False, {}) == 8
    assert bench.executed_contractions(64, False, {}) == 9
    assert bench.executed_contractions(128, True, {}) == 7
    assert bench.executed_contractions(128, False, {"GQA_QM_TWO_PASS": "1"}) == 9
    assert bench.executed_contractions(128, False, {"GQA_TC_CTA_GROUP": "1"}) == 9
    assert bench.executed_contractions(128, False, {"GQA_TC_CTA_GROUP": "2"}) == 8


def test_tf32_peak_from_measured_bf16():
    p = {"bf16_tflops": 1925.9, "bf16_tflops_sustained": 1732.4}
    assert bench.tf32_peak(p, sustained=False) == pytest.approx(1925.9 * 1100 / 2250)
    assert bench.tf32_peak(p, sustained=True) < bench.tf32_peak(p, sustained=False)
    assert bench.fp32_simt_peak_tflops(152, 2070.0) == pytest.approx(80.54784)


def test_clock_summary():
    lines = ["2002, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Active",
             "1950, 2070, 1001.0, 0x4, Not Active, Not Active, Not Active, Active",
             "300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = bench.summarize_clocks(lines)
    assert s["sm_max_mhz"] == 2070 and s["sm_mhz"] == pytest.approx(1976.0)
    assert s["reasons"] == ["sw_power_cap"]
    assert bench.summarize_clocks([])["samples"] == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    bench.barrier()
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 15.0, 1: 15.0}
    assert bench.max_over_ranks(3.0) == 3.0      # no process group: identity


def test_decode_bytes_and_inputs():
    import numpy as np
    import bench
    # K, V read; d_k, d_v read and written; probs read, d_scores written
    assert bench.decode_bytes(16384, 32, 8, 128) == 6 * 16384 * 8 * 128 * 4 + 2 * 32 * 16384 * 4
    cfg = dict(bench.DECODE, history_len=5, n_heads=4, n_kv_heads=2, head_dim=8)
    a, b = bench.decode_inputs(cfg), bench.decode_inputs(cfg)
    assert a["K"].shape == (5, 16) and a["q"].shape == (32,) and a["K"].dtype == np.float32
    assert all(np.array_equal(a[k], b[k]) for k in a)          # seeded


def test_traffic_records_name_known_stages():
    """Every DRAM-traffic record in profiles/ names a stage whose source files
    exist, so bench.py can tell whether the record still matches the kernels
    (the hash itself changes with every kernel edit and is not pinned here)."""
    import json
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    csrc = os.path.join(root, "causal_gqa_attention_attn_gb300", "csrc")
    assert rec
    for key, r in rec.items():
        workload, stage = key.split(":", 1)
        assert stage in bench.STAGE_SOURCES, key
        for src in bench.STAGE_SOURCES[stage]:
            assert os.path.exists(os.path.join(csrc, src)), (key, src)
        assert r["bytes_per_launch"] > 0 and len(r["source_hash"]) == 16
        assert bench._source_hash(stage) and "ncu" in r["command"]
