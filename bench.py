"""Benchmark: causal GQA attention backward from a saved LSE on GB300.

One step = the whole hot path over one batch of synthetic input: zero the
gradient buffers, attention backward (query-tile work: D and dQ, in one pass
over the keys at head_dim 128 on SM pairs; key-tile work: dK and dV), then
the interleaved RoPE backward on dQ and dK, fused into the final writes (the
16k-token workload's recipe). Metric: attention-backward TFLOP/s counted over unmasked
(query, key) pairs, 10 * head_dim * n_heads * N_pairs per step (five d-deep
contractions per pair and head), and the fraction of the dense TF32 tensor
peak.

Prints ONE JSON line (rank 0). ``--impl reference`` times the fp64 CPU
oracle instead, on a bounded sample of the same workload. Other lines for the
rest of the path: ``--forward`` (the tensor-core forward, TFLOP/s),
``--given-o`` (the backward given the forward's O), ``--decode`` (the
decode-style backward, HBM GB/s); ``--workload`` picks one of the five
synthetic workloads, ``--path tc|simt`` a kernel family and ``--graph``
replays the step as a captured CUDA graph (launch-bound short workloads).

Multi-GPU (torchrun): every rank runs its own copy of the workload (the kv-head
groups, batches or documents of a training step are independent problems), so
per-GPU work is fixed and scaling is weak; the only collectives are the
barrier and the max-over-ranks of the timed region.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")   # the oracle's thread pool is the parallelism

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attn-backward TFLOP/s (unmasked pairs) and % of GB300 dense TF32 peak"
UNIT = "TFLOP/s"


# ---------------------------------------------------------------------------
# host-side helpers (covered by CPU tests)
# ---------------------------------------------------------------------------
def counted_flops(head_dim: int, n_heads: int, pairs: int) -> float:
    """Five d-deep contractions (QK^T, dO V^T, P^T dO, dS^T Q, dS K) per pair and head."""
    return 10.0 * head_dim * n_heads * pairs


def executed_flops(head_dim: int, n_heads: int, pairs: int, contractions: int = 9) -> float:
    """What the tensor-core path multiplies: ``contractions`` d-deep
    contractions per pair and head (``executed_contractions``)."""
    return 2.0 * contractions * head_dim * n_heads * pairs


def _env_flag(env, name: str) -> bool:
    try:
        return int(env.get(name, "0") or 0) == 1
    except ValueError:
        return False


def executed_contractions(head_dim: int, given_o: bool, env=None) -> int:
    """Contractions per pair and head that the tensor-core backward runs. The
    key-major kernel always runs four (S^T, dP^T, P^T dO, dS^T Q). The
    query-major kernel runs three with O given (S, dP, dS K), four in its
    single pass at d = 128 on SM pairs (S, dP, (P dP) K, P K), else five (S
    and dP in the D pass and again in the dS pass, dS K). GQA_TC_CTA_GROUP=1
    and GQA_QM_TWO_PASS=1 select the forms without the single pass, as in the
    library."""
    env = os.environ if env is None else env
    if given_o:
        return 7
    single = head_dim == 128 and not _env_flag(env, "GQA_TC_CTA_GROUP") and not _env_flag(env, "GQA_QM_TWO_PASS")
    return 8 if single else 9


def dist_env() -> tuple[int, int, int]:
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """Max of a host float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        p["source"] = "measured"
        return p
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# Nominal dense rates (TFLOP/s): bf16 2250, tf32 1100. The secondary TF32
# figure: the measured bf16 peak times this ratio.
TF32_PER_BF16 = 1100.0 / 2250.0


def tf32_peak(peaks: dict, sustained: bool) -> float:
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    return peaks[key] * TF32_PER_BF16


_TF32_MEASURED: dict = {}


def measure_tf32(torch, dev, n: int = 8192, best_of: int = 10, sustain_s: float = 4.0) -> dict:
    """Dense TF32 rate of this GPU, measured in this run the way the bf16 peak
    was: torch.matmul of fp32 n x n x n with TF32 allowed (cuBLAS, tcgen05
    kind::tf32), 2 n^3 flop per call. burst = best of `best_of` single calls
    timed by CUDA events; sustained = calls back to back for `sustain_s`
    seconds under the power cap. Measured once per process, outside every
    timed region (after it, so that the GEMM's heat does not touch it)."""
    if _TF32_MEASURED:
        return _TF32_MEASURED
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device=dev).manual_seed(1)
        a = torch.randn(n, n, device=dev, generator=g)
        b = torch.randn(n, n, device=dev, generator=g)
        c = torch.empty(n, n, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        flop = 2.0 * n ** 3
        best = float("inf")
        for _ in range(best_of):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        per = max(1, int(sustain_s * 1e3 / best))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(per):
            torch.matmul(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        sus_ms = e0.elapsed_time(e1) / per
        del a, b, c
        _TF32_MEASURED.update({
            "burst": flop / (best / 1e3) / 1e12, "sustained": flop / (sus_ms / 1e3) / 1e12,
            "how": f"torch.matmul fp32 {n}^3 with allow_tf32 (cuBLAS): best of {best_of} "
                   f"(burst) and {per} back to back (sustained), this run"})
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    return _TF32_MEASURED


def tensor_roofline_peak(torch, dev, peaks: dict) -> tuple[float, dict]:
    """The TF32 roofline denominator: the burst rate measured in this run
    (measure_tf32), with the measured-bf16 x nominal-ratio figure kept as a
    secondary field."""
    m = measure_tf32(torch, dev)
    return m["burst"], {"peak_source": f"measured tf32 ({m['how']})",
                        "tf32_sustained": m["sustained"],
                        "peak_bf16_ratio": tf32_peak(peaks, sustained=False),
                        "peak_bf16_ratio_source":
                            f"{peaks['source']} bf16 burst x nominal tf32/bf16 ratio "
                            f"{TF32_PER_BF16:.4f}"}


def fp32_simt_peak_tflops(n_sm: int, max_mhz: float) -> float:
    """CUDA-core fp32 peak: 128 FMA lanes per SM, 2 flops per FMA, at the max SM clock."""
    return n_sm * 128 * 2 * max_mhz * 1e6 / 1e12


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id, self.proc, self.lines = gpu_id, None, []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self) -> dict:
        return summarize_clocks(self.lines)


def summarize_clocks(lines: list[str]) -> dict:
    sm, mx, reasons = [], [], set()
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    for ln in lines:
        parts = [p.strip() for p in ln.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx.append(float(parts[1]))
        except ValueError:
            continue
        for name, val in zip(names, parts[4:8]):
            if val.lower() in ("active", "1", "yes"):
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    # median over samples under load (clock above half of max)
    top = max(mx) if mx else max(sm)
    loaded = [s for s in sm if s >= 0.5 * top] or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": top, "reasons": sorted(reasons),
            "samples": len(sm)}


# The sources each measured stage's kernels are compiled from (device code and
# the headers it includes); a traffic record holds only while they are unchanged.
STAGE_SOURCES = {
    "tc_query_major+tc_key_major": ["tc_bwd.cu", "tc_common.cuh", "common.cuh", "rope_common.cuh"],
    "tc_forward": ["tc_fwd.cu", "tc_common.cuh", "common.cuh"],
    "short_bwd": ["short_bwd.cu", "common.cuh", "rope_common.cuh"],
    "decode": ["decode_bwd.cu", "common.cuh"],
}


def _source_hash(stage: str) -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "causal_gqa_attention_attn_gb300", "csrc")
    for f in sorted(STAGE_SOURCES.get(stage, [])):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def _traffic(stage: str, workload: str):
    """DRAM bytes per launch of the dominant stage from the committed ncu
    summary, when it was taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or stage not in STAGE_SOURCES:
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{workload}:{stage}")
    if not rec or rec.get("source_hash") != _source_hash(stage):
        return None
    return rec.get("bytes_per_launch")


def _gpu_uuid(torch, dev) -> str | None:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


def run_gpu(args) -> dict | None:
    import torch
    import causal_gqa_attention_attn_gb300 as ga

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w, seed=w.seed + rank)      # each rank: its own problem
    S, H, Hk, d, sc = w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim, w.scale
    pairs = workloads.n_pairs(x["seg"])
    flops = counted_flops(d, H, pairs)
    impl_fn = ga.attn_bwd_simt if args.path == "simt" else ga.attn_bwd
    # "tc": the short path (one cooperative launch for short sequences) off,
    # so that short workloads run the tensor-core kernels too
    ga.set_short_path(args.path == "auto")

    host = {k: torch.from_numpy(np.ascontiguousarray(x[k])).pin_memory()
            for k in ("Q", "K", "V", "dO")}
    host["seg"] = torch.from_numpy(x["seg"].astype(np.int32)).pin_memory()
    t = {k: v.to(dev) for k, v in host.items()}
    _, LSE = ga.attn_fwd(t["Q"], t["K"], t["V"], t["seg"], H, Hk, d, sc)   # setup, untimed
    host["LSE"] = LSE.cpu().pin_memory()
    t["LSE"] = LSE
    dQ = torch.zeros(S, H * d, device=dev)
    dK = torch.zeros(S, Hk * d, device=dev)
    dV = torch.zeros(S, Hk * d, device=dev)
    ws = torch.empty(ga.workspace_bytes(S, H, Hk, d), dtype=torch.uint8, device=dev)

    fused_rope = w.rope and args.path != "simt" and not args.given_o
    O_dev = None
    if args.given_o:       # the forward output O, as a training step keeps it (setup, untimed)
        O_dev, _ = ga.attn_fwd(t["Q"], t["K"], t["V"], t["seg"], H, Hk, d, sc)

    def step():
        dQ.zero_()
        dK.zero_()
        dV.zero_()
        if fused_rope:       # RoPE backward on dQ, dK fused into the kernels' final writes
            ga.attn_bwd_rope(t["Q"], t["K"], t["V"], t["dO"], t["LSE"], t["seg"], dQ, dK, dV, H,
                             Hk, d, sc, pos_offset=0, base=10000.0, workspace=ws)
            return
        if args.given_o:
            ga.attn_bwd_o(t["Q"], t["K"], t["V"], t["dO"], O_dev, t["LSE"], t["seg"], dQ, dK, dV,
                          H, Hk, d, sc, workspace=ws)
        else:
            impl_fn(t["Q"], t["K"], t["V"], t["dO"], t["LSE"], t["seg"], dQ, dK, dV, H, Hk, d, sc,
                    workspace=ws)
        if w.rope:
            ga.rope_bwd_inplace(dQ, H, d, 0, 10000.0)
            ga.rope_bwd_inplace(dK, Hk, d, 0, 10000.0)

    for _ in range(args.warmup):
        step()
    ga.read_device_status(ws)
    torch.cuda.synchronize()

    K = args.steps
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in ev_a + ev_b:            # create the underlying cudaEvent_t now
        e.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    graph = None
    if args.graph:
        # the whole step (gradient fills + the backward) captured once as a
        # CUDA graph and replayed: one host call per step instead of the
        # binding's and the library's per-launch host work. (Events recorded
        # during capture become graph dependencies, not timestamps: the stage
        # time is read from eager steps after the timed region.)
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        cap0 = ga.launch_count()
        with torch.cuda.graph(graph):
            step()
        launches_per_step = ga.launch_count() - cap0
        graph.replay()
        torch.cuda.synchronize()
    launches0 = ga.launch_count()
    with ClockSampler(_gpu_uuid(torch, dev)) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record()
        for k in range(K):
            if graph is not None:
                graph.replay()
            else:
                ga.profile_events(ev_a[k], ev_b[k])
                step()
        end.record()
        torch.cuda.synchronize()
        barrier()
    launches = ga.launch_count() - launches0
    if graph is not None:
        launches = launches_per_step * K      # replays do not pass through the library's host code
    stage = ga.profile_stage_name()
    ga.read_device_status(ws)
    ms = start.elapsed_time(end)
    ms_max = max_over_ranks(ms, dev)
    if graph is not None:     # the same kernels, run eagerly: their stage time
        n_eager = min(K, 10)
        for k in range(n_eager):
            ga.profile_events(ev_a[k], ev_b[k])
            step()
        torch.cuda.synchronize()
        stage = ga.profile_stage_name()
        stage_ms = sum(ev_a[k].elapsed_time(ev_b[k]) for k in range(n_eager)) / n_eager
    else:
        stage_ms = sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / K
    value = world * flops / (ms_max / K / 1e3) / 1e12

    # End to end through the public API with host buffers (pinned) every step:
    # each step uploads its inputs and downloads its gradients. Two device
    # buffer sets let the upload of step k+1 and the download of step k-1 run
    # on copy streams while step k computes.
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("Q", "K", "V", "dO", "LSE", "seg"))
    names = ("Q", "K", "V", "dO", "LSE", "seg")
    if args.given_o:
        host["O"] = O_dev.cpu().pin_memory()
        t["O"] = O_dev
        names = names + ("O",)
        h2d += host["O"].numel() * host["O"].element_size()
    ins = [t, {k: torch.empty_like(t[k]) for k in names}]
    grads = [(dQ, dK, dV), tuple(torch.empty_like(g) for g in (dQ, dK, dV))]
    outs = [tuple(torch.empty(g.shape, pin_memory=True) for g in (dQ, dK, dV)) for _ in range(2)]
    d2h = sum(g.numel() * g.element_size() for g in outs[0])
    comp = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + ev_down:
        e.record(comp)

    def upload(k):
        j = k % 2
        up.wait_event(ev_comp[j])            # step k-2 has finished reading set j
        with torch.cuda.stream(up):
            for n in names:
                ins[j][n].copy_(host[n], non_blocking=True)
        ev_up[j].record(up)

    def compute(k):
        j = k % 2
        comp.wait_event(ev_up[j])
        comp.wait_event(ev_down[j])          # step k-2's gradients have left set j
        x, (gq, gk, gv) = ins[j], grads[j]
        for g_ in (gq, gk, gv):
            g_.zero_()
        if fused_rope:
            ga.attn_bwd_rope(x["Q"], x["K"], x["V"], x["dO"], x["LSE"], x["seg"], gq, gk, gv, H,
                             Hk, d, sc, pos_offset=0, base=10000.0, workspace=ws)
        else:
            if args.given_o:
                ga.attn_bwd_o(x["Q"], x["K"], x["V"], x["dO"], x["O"], x["LSE"], x["seg"], gq, gk,
                              gv, H, Hk, d, sc, workspace=ws)
            else:
                impl_fn(x["Q"], x["K"], x["V"], x["dO"], x["LSE"], x["seg"], gq, gk, gv, H, Hk, d,
                        sc, workspace=ws)
            if w.rope:
                ga.rope_bwd_inplace(gq, H, d, 0, 10000.0)
                ga.rope_bwd_inplace(gk, Hk, d, 0, 10000.0)
        ev_comp[j].record(comp)

    def download(k):
        j = k % 2
        down.wait_event(ev_comp[j])
        with torch.cuda.stream(down):
            for dst, src in zip(outs[j], grads[j]):
                dst.copy_(src, non_blocking=True)
        ev_down[j].record(down)

    def e2e_run(n):
        upload(0)
        for k in range(n):
            if k + 1 < n:
                upload(k + 1)
            compute(k)
            download(k)
        comp.wait_event(ev_down[(n - 1) % 2])

    e2e_run(2)
    torch.cuda.synchronize()
    barrier()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(comp)
    up.wait_event(s2)
    e2e_run(K)
    e2.record(comp)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2), dev)
    e2e_value = world * flops / (e2e_ms / K / 1e3) / 1e12

    peaks = load_peaks()
    props = torch.cuda.get_device_properties(dev)
    tensor_path = "tc" in stage
    clocks = clk.summary()
    tf32, tf32_info = tensor_roofline_peak(torch, dev, peaks)
    if tensor_path:
        peak = tf32
        roof = {"bound": "tensor", "unit": UNIT, **tf32_info}
    else:
        peak = fp32_simt_peak_tflops(props.multi_processor_count, peaks.get("sm_max_mhz", 2070.0))
        roof = {"bound": "alu", "unit": UNIT, "peak_source":
                f"{props.multi_processor_count} SMs x 128 fp32 FMA/clk x 2 x max SM clock"}
    achieved = flops / (stage_ms / 1e3) / 1e12
    roof.update({"kernel": stage, "achieved": achieved, "peak": peak, "frac": achieved / peak,
                 "traffic": _traffic(stage, w.name), "stage_ms": stage_ms,
                 "flops_per_launch": flops})
    if tensor_path:
        ex = executed_flops(d, H, pairs, executed_contractions(d, args.given_o))
        roof.update({"executed_flops_per_launch": ex,
                     "executed_tflops": ex / (stage_ms / 1e3) / 1e12,
                     "executed_frac": ex / (stage_ms / 1e3) / 1e12 / peak,
                     "frac_of_bf16_ratio_peak": achieved / tf32_info["peak_bf16_ratio"],
                     # the steps run back to back under the power cap, the
                     # condition the sustained TF32 figure is measured in
                     "frac_of_tf32_sustained": achieved / tf32_info["tf32_sustained"]})
    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "tf32" if tensor_path else "f32",
        "data": "synthetic (seeded N(0,sigma^2) Q,K,V,dO; LSE from this library's forward)",
        "pct_of_tf32_peak": 100.0 * value / tf32,
        "config": {"workload": w.name, "shape": w.describe, "seq_len": S, "n_heads": H,
                   "n_kv_heads": Hk, "head_dim": d, "n_pairs": pairs,
                   "counted_flop_per_step": flops,
                   "step": ("zero grads + attn_bwd_rope (RoPE backward of dQ, dK fused)" if fused_rope else
                            "zero grads + " + ("attn_bwd_o (D from the forward's O)" if args.given_o else "attn_bwd") +
                            (" + rope_bwd(dQ) + rope_bwd(dK)" if w.rope else "")),
                   "l2": "inputs larger than L2 (129 MB)" if 4 * S * H * d > 129e6 else
                         "inputs smaller than L2: steps run back to back (warm L2)",
                   "path": stage,
                   "launch": "CUDA graph replay of the step" if args.graph else "eager (Python-driven)"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "overlap": "two device buffer sets: step k+1's upload and step k-1's download "
                           "run on copy streams while step k computes"},
        "gpu_launches": launches,
        "roofline": roof,
        "clocks": clocks,
    }
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# --decode: the decode-style backward from saved probabilities (one query per
# head against a key history), an HBM-bound path measured in GB/s
# ---------------------------------------------------------------------------
DECODE = {"name": "decode16k", "history_len": 16384, "n_heads": 32, "n_kv_heads": 8,
          "head_dim": 128, "seed": 606}


def decode_bytes(L: int, H: int, Hk: int, d: int) -> int:
    """Algorithmic bytes of one attn_decode_bwd call: K and V read, d_k and d_v
    read and written, probs read and d_scores written."""
    return 6 * L * Hk * d * 4 + 2 * H * L * 4


def decode_inputs(cfg: dict, seed_offset: int = 0) -> dict:
    """Seeded q, K, V, d_out (N(0,1), fp32) of the decode workload."""
    L, H, Hk, d = cfg["history_len"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    rng = np.random.default_rng(cfg["seed"] + seed_offset)
    return {"q": rng.standard_normal(H * d, dtype=np.float32),
            "K": rng.standard_normal((L, Hk * d), dtype=np.float32),
            "V": rng.standard_normal((L, Hk * d), dtype=np.float32),
            "d_out": rng.standard_normal(H * d, dtype=np.float32)}


def run_decode(args) -> dict | None:
    import torch
    import causal_gqa_attention_attn_gb300 as ga

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    cfg = DECODE
    L, H, Hk, d = cfg["history_len"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    G, sc = H // Hk, 1.0 / math.sqrt(d)
    x = decode_inputs(cfg, rank)
    host = {k: torch.from_numpy(v).pin_memory() for k, v in x.items()}
    t = {k: v.to(dev) for k, v in host.items()}
    # the forward's probabilities of this query (setup, untimed)
    Kg = t["K"].view(L, Hk, d).repeat_interleave(G, dim=1)          # [L, H, d]
    t["probs"] = torch.softmax(sc * torch.einsum("lhd,hd->hl", Kg, t["q"].view(H, d)), dim=1).contiguous()
    host["probs"] = t["probs"].cpu().pin_memory()
    dq = torch.zeros(H * d, device=dev)
    dk = torch.zeros(L, Hk * d, device=dev)
    dv = torch.zeros(L, Hk * d, device=dev)
    ds = torch.empty(H, L, device=dev)
    ws = torch.empty(int(ga.lib().attn_decode_bwd_workspace_bytes(L, H, Hk, d)), dtype=torch.uint8,
                     device=dev)

    def step(src):
        ga.attn_decode_bwd(src["q"], src["K"], src["V"], src["probs"], src["d_out"], H, Hk, d, sc,
                           d_q=dq, d_k_hist=dk, d_v_hist=dv, d_scores=ds, workspace=ws)

    for _ in range(args.warmup):
        step(t)
    torch.cuda.synchronize()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = ga.launch_count()
    with ClockSampler(_gpu_uuid(torch, dev)) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record()
        for _ in range(K):
            step(t)
        end.record()
        torch.cuda.synchronize()
        barrier()
    launches = ga.launch_count() - launches0
    ms_max = max_over_ranks(start.elapsed_time(end), dev)
    nbytes = decode_bytes(L, H, Hk, d)
    value = world * nbytes / (ms_max / K / 1e3) / 1e9

    # end to end with host buffers: each step uploads q, K, V, probs, d_out and
    # reads back d_scores, d_q, d_k_hist, d_v_hist (no overlap)
    outs = {n: torch.empty(g.shape, pin_memory=True) for n, g in
            (("d_scores", ds), ("d_q", dq), ("d_k_hist", dk), ("d_v_hist", dv))}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    dbuf = {k: torch.empty_like(v) for k, v in t.items()}

    def e2e_step():
        for k_, v_ in host.items():
            dbuf[k_].copy_(v_, non_blocking=True)
        step(dbuf)
        for (n, o), g in zip(outs.items(), (ds, dq, dk, dv)):
            o.copy_(g, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record()
    for _ in range(K):
        e2e_step()
    e2.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2), dev)

    peaks = load_peaks()
    hbm = float(peaks.get("hbm_gbs") or 6800.0)
    per_call_gbs = nbytes / (ms_max / K / 1e3) / 1e9
    result = {
        "metric": "decode attn-backward HBM GB/s (algorithmic bytes)", "value": value,
        "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded N(0,1) q, K, V, d_out; probs = softmax(scale q.K) of this query)",
        "config": {"workload": cfg["name"], "history_len": L, "n_heads": H, "n_kv_heads": Hk,
                   "head_dim": d, "bytes_per_step": nbytes,
                   "step": "attn_decode_bwd (+= into d_q, d_k_hist, d_v_hist)",
                   "l2": "working set (0.4 GB) larger than L2 (129 MB)"},
        "e2e": {"value": world * nbytes / (e2e_ms / K / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "none: copies and kernels in order on one stream"},
        "gpu_launches": launches,
        "roofline": {"bound": "hbm", "unit": "GB/s", "achieved": per_call_gbs, "peak": hbm,
                     "frac": per_call_gbs / hbm, "traffic": _traffic("decode", "decode16k"),
                     "peak_source": "measured HBM copy rate (MEASURED_PEAKS.json hbm_gbs)"},
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        t0 = time.perf_counter()
        oracle.decode_bwd(x["q"], x["K"], x["V"], host["probs"].numpy(), x["d_out"], H, Hk, d, sc)
        secs = time.perf_counter() - t0
        result["cpu_baseline"] = {"value": nbytes / secs / 1e9, "unit": "GB/s", "cores": 1,
                                  "kind": "oracle", "seconds": secs,
                                  "sample": f"oracle.decode_bwd (fp64, numpy) on the whole {cfg['name']} call"}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# the tensor-core forward (attn_fwd: O and LSE), the setup step of the
# backward, measured on its own
# ---------------------------------------------------------------------------
def forward_counted_flops(head_dim: int, n_heads: int, pairs: int) -> float:
    """Two d-deep contractions (Q K^T, P V) per unmasked pair and head."""
    return 4.0 * head_dim * n_heads * pairs


def run_forward(args) -> dict | None:
    import torch
    import causal_gqa_attention_attn_gb300 as ga

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w, seed=w.seed + rank)
    S, H, Hk, d, sc = w.seq_len, w.n_heads, w.n_kv_heads, w.head_dim, w.scale
    pairs = workloads.n_pairs(x["seg"])
    flops = forward_counted_flops(d, H, pairs)
    host = {k: torch.from_numpy(np.ascontiguousarray(x[k])).pin_memory() for k in ("Q", "K", "V")}
    host["seg"] = torch.from_numpy(x["seg"].astype(np.int32)).pin_memory()
    t = {k: v.to(dev) for k, v in host.items()}
    O = torch.empty(S, H * d, device=dev)
    LSE = torch.empty(S, H, device=dev)
    ws = torch.empty(int(ga.lib().attn_fwd_workspace_bytes(S, H, Hk, d)), dtype=torch.uint8,
                     device=dev)

    def step(src):
        ga.attn_fwd(src["Q"], src["K"], src["V"], src["seg"], H, Hk, d, sc, O=O, LSE=LSE,
                    workspace=ws)

    for _ in range(args.warmup):
        step(t)
    ga.read_device_status(ws)
    torch.cuda.synchronize()
    K = args.steps
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for e in ev_a + ev_b:
        e.record()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    launches0 = ga.launch_count()
    with ClockSampler(_gpu_uuid(torch, dev)) as clk:
        barrier()
        torch.cuda.synchronize()
        start.record()
        for k in range(K):
            ga.profile_events(ev_a[k], ev_b[k])
            step(t)
        end.record()
        torch.cuda.synchronize()
        barrier()
    launches = ga.launch_count() - launches0
    stage = ga.profile_stage_name()
    ga.read_device_status(ws)
    ms_max = max_over_ranks(start.elapsed_time(end), dev)
    stage_ms = sum(a.elapsed_time(b) for a, b in zip(ev_a, ev_b)) / K
    value = world * flops / (ms_max / K / 1e3) / 1e12

    # end to end with host buffers: each step uploads Q, K, V, seg and reads
    # back O and LSE (in order on one stream)
    outs = {"O": torch.empty(O.shape, pin_memory=True), "LSE": torch.empty(LSE.shape, pin_memory=True)}
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    dbuf = {k: torch.empty_like(v) for k, v in t.items()}

    def e2e_step():
        for k_, v_ in host.items():
            dbuf[k_].copy_(v_, non_blocking=True)
        step(dbuf)
        outs["O"].copy_(O, non_blocking=True)
        outs["LSE"].copy_(LSE, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record()
    for _ in range(K):
        e2e_step()
    e2.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(s2.elapsed_time(e2), dev)

    peaks = load_peaks()
    tensor_path = stage == "tc_forward"
    if tensor_path:
        peak, tf32_info = tensor_roofline_peak(torch, dev, peaks)
        roof = {"bound": "tensor", "unit": UNIT, **tf32_info}
    else:   # CUDA-core forward (head dims without a tensor-core kernel): no stage events
        props = torch.cuda.get_device_properties(dev)
        peak = fp32_simt_peak_tflops(props.multi_processor_count, peaks.get("sm_max_mhz", 2070.0))
        roof = {"bound": "alu", "unit": UNIT, "peak_source":
                f"{props.multi_processor_count} SMs x 128 fp32 FMA/clk x 2 x max SM clock"}
        stage, stage_ms = "fwd_kernel (whole call)", ms_max / K
    achieved = flops / (stage_ms / 1e3) / 1e12
    roof.update({"kernel": stage, "achieved": achieved, "peak": peak, "frac": achieved / peak,
                 "traffic": _traffic(stage, w.name), "stage_ms": stage_ms,
                 "flops_per_launch": flops})
    if tensor_path:   # one pass, online softmax: Q K^T and P V, the counted two
        ex = 4.0 * d * H * pairs
        roof.update({"executed_flops_per_launch": ex,
                     "executed_tflops": ex / (stage_ms / 1e3) / 1e12,
                     "executed_frac": ex / (stage_ms / 1e3) / 1e12 / peak,
                     "frac_of_tf32_sustained": achieved / tf32_info["tf32_sustained"]})
    result = {
        "metric": "attn-forward TFLOP/s (unmasked pairs)", "value": value, "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms_max / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "tf32" if tensor_path else "f32",
        "data": "synthetic (seeded N(0,sigma^2) Q, K, V)",
        "config": {"workload": w.name, "shape": w.describe.split(" +")[0], "seq_len": S,
                   "n_heads": H, "n_kv_heads": Hk, "head_dim": d, "n_pairs": pairs,
                   "counted_flop_per_step": flops, "step": "attn_fwd (O, LSE overwritten)",
                   "l2": "inputs larger than L2 (129 MB)" if 4 * S * (H + 2 * Hk) * d > 129e6
                   else "inputs smaller than L2: steps run back to back (warm L2)"},
        "e2e": {"value": world * flops / (e2e_ms / K / 1e3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "overlap": "none: copies and kernels in order on one stream"},
        "gpu_launches": launches,
        "roofline": roof,
        "clocks": clk.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = CPU_SAMPLE_ROWS.get(w.name, 256)
        rows = np.arange(max(0, S - n), S)
        sp = int(np.sum(rows - x["seg"][rows].astype(np.int64) + 1))
        t0 = time.perf_counter()
        oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], H, Hk, d, sc, rows=rows)
        secs = time.perf_counter() - t0
        result["cpu_baseline"] = {
            "value": forward_counted_flops(d, H, sp) / secs / 1e12, "unit": UNIT,
            "cores": oracle._workers(), "kind": "oracle", "seconds": secs,
            "sample": f"oracle.fwd (fp64, numpy) on query rows [{rows[0]}, {S}) of all {H} heads "
                      f"({sp} unmasked pairs per head) of workload {w.name}"}
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# the fp64 oracle on the host cores: CPU baseline and the reference arm
# ---------------------------------------------------------------------------
def oracle_sample(w, x, lse32, n_rows: int) -> tuple[float, float, str, int]:
    """Time the oracle's backward over the last ``n_rows`` query rows of every
    head (each row against all of its visible keys). Returns (seconds,
    counted flops of the sample, description, threads)."""
    import oracle
    S = w.seq_len
    rows = np.arange(max(0, S - n_rows), S)
    seg = x["seg"]
    pairs = int(np.sum(rows - seg[rows].astype(np.int64) + 1))
    t0 = time.perf_counter()
    oracle.bwd(x["Q"], x["K"], x["V"], x["dO"], lse32, seg, w.n_heads, w.n_kv_heads,
               w.head_dim, w.scale, rows=rows)
    dt = time.perf_counter() - t0
    desc = (f"oracle.bwd (fp64, numpy) on query rows [{rows[0]}, {S}) of all {w.n_heads} heads "
            f"({pairs} unmasked pairs per head) of workload {w.name}")
    return dt, counted_flops(w.head_dim, w.n_heads, pairs), desc, oracle._workers()


def sample_lse(w, x, n_rows: int) -> np.ndarray:
    """LSE for the sampled rows from the oracle forward (other rows unused)."""
    import oracle
    rows = np.arange(max(0, w.seq_len - n_rows), w.seq_len)
    _, lse = oracle.fwd(x["Q"], x["K"], x["V"], x["seg"], w.n_heads, w.n_kv_heads, w.head_dim,
                        w.scale, rows=rows)
    return lse.astype(np.float32)


CPU_SAMPLE_ROWS = {"tiny": 64, "causal512": 512, "docs2k": 2048, "docs4k": 4096, "causal16k": 4096}
REF_SAMPLE_ROWS = {"tiny": 64, "causal512": 512, "docs2k": 2048, "docs4k": 2048, "causal16k": 2048}


def cpu_baseline(w) -> dict:
    x = workloads.make_inputs(w)
    n = CPU_SAMPLE_ROWS.get(w.name, 256)
    lse32 = sample_lse(w, x, n)
    dt, fl, desc, cores = oracle_sample(w, x, lse32, n)
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": desc, "seconds": dt}


def run_reference(args) -> dict | None:
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w)
    n = REF_SAMPLE_ROWS.get(w.name, 256)
    lse32 = sample_lse(w, x, n)
    for _ in range(args.warmup):
        oracle_sample(w, x, lse32, n)
    times, fl, desc, cores = [], 0.0, "", 1
    for _ in range(args.steps):
        dt, fl, desc, cores = oracle_sample(w, x, lse32, n)
        times.append(dt)
    mean = sum(times) / len(times)
    value = fl / mean / 1e12
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * mean,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "shape": w.describe, "sample_rows": n},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(workloads.WORKLOADS), default="causal16k")
    ap.add_argument("--path", choices=["auto", "tc", "simt"], default="auto",
                    help="auto: attn_bwd (the single-launch short path for short sequences, "
                         "else tensor cores where built); tc: attn_bwd with the short path off; "
                         "simt: attn_bwd_simt")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--given-o", action="store_true",
                    help="time attn_bwd_o (D = rowsum(dO*O) from the forward's O) instead of the LSE-only call")
    ap.add_argument("--graph", action="store_true",
                    help="replay the step as a captured CUDA graph (for launch-bound short workloads)")
    ap.add_argument("--forward", action="store_true",
                    help="time attn_fwd (the tensor-core forward producing O and LSE) on the workload")
    ap.add_argument("--decode", action="store_true",
                    help="time attn_decode_bwd (one query per head against a 16384-key history) in GB/s")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.forward:
        if args.impl == "reference" or args.decode or args.given_o:
            ap.error("--forward times this library's attn_fwd alone")
        res = run_forward(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.decode:
        if args.impl == "reference":
            ap.error("--decode times this library's kernels only")
        res = run_decode(args)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.impl == "reference":
        res = run_reference(args)
    else:
        res = run_gpu(args)
        rank, world, _ = dist_env()
        if res is not None and world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(workloads.WORKLOADS[args.workload])
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
