"""Benchmark of the context-parallel causal ring-attention step on GB300.

One bench step = one pass of the whole hot path over the workload: the
emulated ring forward (R step launches with the running LSE merge, the last
one writing bf16 O) and the ring backward (delta preprocess and R backward
step launches), on inputs already resident in HBM. The metric is attention
TFLOPS counting unmasked FLOPs only: forward 4*d*Hq per visible (query, key)
pair, backward 2.5x that.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica (the ring is
emulated inside one GPU; nothing is exchanged between ranks), timing is
max-over-ranks and the value is the whole-job FLOP rate ("scaling": "weak").
``--impl reference`` times the CPU fp64 oracle on a bounded sample of the
same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import WORKLOADS, bf16_bits_to_f64, make_inputs  # noqa: E402

METRIC = "causal attn TFLOPS fwd/bwd (unmasked FLOPs) and % of GB300 dense BF16 peak"

# DRAM traffic per launch from the ncu captures summarised in profiles/, valid
# only while the kernel source is the one that was profiled.
PROFILED_TRAFFIC = {
    "step_bwd": ("context_causal_attention_ring_gb300/csrc/step_bwd.cu",
                 "a662b08e9cd0ec616e01d1bf47a75b9b02a3a44f8c008dc149a884986215c990", 3.102382e9),
    "step_fwd": ("context_causal_attention_ring_gb300/csrc/step_fwd.cu",
                 "03b628acb6c1b91979d4fd63e73eb892fc399c09de174a82b5d742f1cb4af938", 1.293140e9),
}


def _profiled_traffic(kernel):
    import hashlib
    if kernel not in PROFILED_TRAFFIC:
        return None
    rel, digest, nbytes = PROFILED_TRAFFIC[kernel]
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() == digest:
                return nbytes
    except OSError:
        pass
    return None
UNIT = "TFLOPS"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return pk, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0,
                "bf16_tflops_sustained": 1700.0}, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, device) -> float:
    """The maximum of a per-rank float over all ranks of the default process
    group (the value itself when there is no group or a single rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(n_ranks: int, flops_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job rate: every rank runs its own replica of the step, so the
    job processes n_ranks times one rank's FLOPs in the slowest rank's time."""
    return n_ranks * flops_per_rank_step / (ms_per_step * 1e-3) / 1e12


def roofline_record(kernel, achieved, flops_per_launch, peaks, peak_kind, clocks):
    """Roofline of a tensor-bound kernel timed in a sub-second loop.

    frac is against the measured burst bf16 peak (a GEMM timed alone, the
    regime of this loop). Two secondary figures: the peak scaled to the SM
    clock seen during the timed region (peak x median MHz / max MHz), and
    the sustained peak (a seconds-long GEMM loop under the power cap)."""
    peak = peaks["bf16_tflops"]
    rec = {"bound": "tensor", "kernel": kernel, "achieved": achieved, "peak": peak,
           "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
           "peak_kind": f"bf16_tflops burst ({peak_kind}): the kernel is timed in a "
                        "sub-second loop, the regime of the burst measurement",
           "flops_per_launch": flops_per_launch}
    sust = peaks.get("bf16_tflops_sustained")
    if sust:
        rec["peak_sustained"] = sust
        rec["frac_sustained"] = achieved / sust
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz"):
        scale = clocks["sm_mhz"] / clocks["sm_max_mhz"]
        rec["clock_normalised"] = {
            "sm_mhz_median": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
            "peak_at_clock": peak * scale, "frac": achieved / (peak * scale),
            "basis": "burst peak x (median SM MHz in the timed region / max SM MHz)"}
    return rec


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx = max(mx, float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_sample(w, n_heads_sample: int, inp=None):
    """Time the fp64 oracle's forward and backward of one off-diagonal ring
    pair (step 1, rank 1) over `n_heads_sample` query heads. Returns
    (TFLOPS, seconds, description)."""
    import oracle
    if inp is None:
        inp = make_inputs(w)
    q_pos, kv_pos = oracle.plan_positions(w.seq_len, w.cp, w.layout, w.kv_prefix_len)
    qo, ko = 1 % w.cp, 0
    H = min(n_heads_sample, w.n_q_heads)
    G = w.group
    Hk = max(1, H // G)
    qrows = q_pos[qo] - w.kv_prefix_len
    q = bf16_bits_to_f64(inp.q[qrows][:, :H])
    k = bf16_bits_to_f64(inp.k[kv_pos[ko]][:, :Hk])
    v = bf16_bits_to_f64(inp.v[kv_pos[ko]][:, :Hk])
    do = bf16_bits_to_f64(inp.dout[qrows][:, :H])
    pairs = oracle.count_visible(q_pos[qo], kv_pos[ko])
    flops = 4.0 * w.head_dim * H * pairs * (1 + 2.5)
    t0 = time.perf_counter()
    O, L = oracle.partial_attention(q, k, v, q_pos[qo], kv_pos[ko])
    # backward share of the pair with the pair's own softmax (same work)
    oracle.attention_backward(q, k, v, do, O, L, q_pos[qo], kv_pos[ko])
    dt = time.perf_counter() - t0
    desc = (f"oracle fp64 forward+backward of ring pair (q_owner={qo}, kv_owner={ko}) "
            f"of {w.name}: {len(qrows)} queries x {len(kv_pos[ko])} keys, "
            f"{H} of {w.n_q_heads} query heads, {pairs} visible pairs per head")
    return flops / dt / 1e12, dt, desc


def run_reference(args, w):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    heads = int(os.environ.get("CP_BENCH_CPU_HEADS", "4"))
    inp = make_inputs(w, with_dout=True)  # the step times forward and backward
    cpu_oracle_sample(w, 1, inp)  # warm-up (page-in, BLAS threads)
    vals, times = [], []
    desc = ""
    for _ in range(args.steps):
        v, dt, desc = cpu_oracle_sample(w, heads, inp)
        vals.append(v)
        times.append(dt)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": statistics.median(times) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "seq_len": w.seq_len, "cp": w.cp,
                   "n_q_heads": w.n_q_heads, "n_kv_heads": w.n_kv_heads,
                   "head_dim": w.head_dim, "layout": w.layout, "variant": "pass_kv",
                   "sample": "one ring pair, subset of heads"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_config(w, steps: int, warmup: int, dev):
    """Forward and backward ring passes of another workload (per-step calls,
    chained, fp32 accumulators), timed with CUDA events on the launching
    stream: median fwd, bwd and whole-pass times and TFLOPS (unmasked FLOPs)."""
    import torch
    import context_causal_attention_ring_gb300 as cpa

    stream = torch.cuda.current_stream()
    inp = make_inputs(w, with_dout=True)
    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
                    layout=w.layout, variant="pass_kv", cu_seqlens=inp.cu_seqlens,
                    kv_prefix_len=w.kv_prefix_len)

    def dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    nat = [dev_bf16(x) for x in (inp.q, inp.k, inp.v, inp.dout)]
    del inp
    q, k, v, do = (torch.empty_like(x) for x in nat)
    for kind, x, y in zip((cpa.TENSOR_Q, cpa.TENSOR_KV, cpa.TENSOR_KV, cpa.TENSOR_Q), nat,
                          (q, k, v, do)):
        plan.layout_apply(kind, cpa.TO_RANK_MAJOR, x, y)
    del nat
    R, Hq, Hkv, d = plan.R, plan.Hq, plan.Hkv, plan.d
    o = torch.empty_like(q)
    lse = torch.empty((Hq, plan.T_q), dtype=torch.float32, device=dev)
    o_acc = torch.empty((plan.T_q, Hq, d), dtype=torch.float32, device=dev)
    delta = torch.empty((Hq, plan.T_q), dtype=torch.float32, device=dev)
    half_ops = torch.empty(plan.half_ops_size(), dtype=torch.uint8, device=dev)
    dq = torch.empty((plan.T_q, Hq, d), dtype=torch.float32, device=dev)
    dk = torch.empty((plan.T_kv, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)
    plan.set_chaining(True)
    fwd_flops = 4.0 * d * Hq * plan.visible_pairs()

    def one(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for t in range(R):
            plan.step_fwd(t, q, k, v, o_acc, lse, cpa.ACCUMULATE, o if t == R - 1 else None,
                          stream)
        if ev is not None:
            ev[1].record(stream)
        plan.bwd_preprocess(q, k, v, o, do, delta, half_ops, dq, dk, dv, o_f32=o_acc,
                            stream=stream)
        if ev is not None:
            ev[2].record(stream)
        for t in range(R):
            plan.step_bwd_half(t, half_ops, lse, delta, dq, dk, dv, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for e in evs:
        one(e)
    torch.cuda.synchronize()
    plan.sync_status(stream)
    fwd = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    bwd = statistics.median(e[2].elapsed_time(e[3]) for e in evs)
    whole = statistics.median(e[0].elapsed_time(e[3]) for e in evs)
    out = {"workload": w.name, "seq_len": w.seq_len, "cp": w.cp, "n_q_heads": Hq,
           "n_kv_heads": Hkv, "head_dim": d, "steps": steps, "warmup": warmup,
           "fwd_ms": fwd, "bwd_ms": bwd, "step_ms": whole,
           "fwd_tflops": fwd_flops / (fwd * 1e-3) / 1e12,
           "bwd_tflops": 2.5 * fwd_flops / (bwd * 1e-3) / 1e12,
           "step_tflops": 3.5 * fwd_flops / (whole * 1e-3) / 1e12}
    del q, k, v, do, o, lse, o_acc, delta, half_ops, dq, dk, dv, plan
    torch.cuda.empty_cache()
    return out


def cpu_oracle_plan_runs():
    """The oracle as planned for the CPU baseline: the whole tiny ring
    (forward ring with its merge, and the ring backward) and a sampled
    million-token forward (a few seeded rows, exact full-prefix softmax each;
    labelled sampled, not extrapolated)."""
    import oracle
    from workloads import sample_rows
    runs = []
    w = WORKLOADS["tiny_ring"]
    inp = make_inputs(w, with_dout=True)
    q_pos, kv_pos = oracle.plan_positions(w.seq_len, w.cp, w.layout)
    qperm, kperm = np.concatenate(q_pos), np.concatenate(kv_pos)
    q, k, v, do = (bf16_bits_to_f64(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    pairs = oracle.count_visible(np.arange(w.seq_len), np.arange(w.seq_len))
    t0 = time.perf_counter()
    O, L = oracle.ring_forward(q[qperm], k[kperm], v[kperm], q_pos, kv_pos)
    oracle.ring_backward(q[qperm], k[kperm], v[kperm], do[qperm], O, L, q_pos, kv_pos)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.head_dim * w.n_q_heads * pairs * 3.5
    runs.append({"workload": w.name, "kind": "full", "what": "ring forward + ring backward",
                 "seconds": dt, "us": dt * 1e6, "gflops": flops / dt / 1e9})
    w = WORKLOADS["million_token_group"]
    N = w.seq_len
    rows = sample_rows(N, 30)
    # the sample's operands are drawn directly with the workload's recipe
    # (N(0,1), Q and K x 0.5, bf16) from their own seeded stream: the
    # oracle's time does not depend on the values, and drawing the whole
    # workload first would dominate the bench
    from workloads import draw_bf16
    rng = np.random.default_rng(w.seed)
    qr = bf16_bits_to_f64(draw_bf16(rng, (len(rows), w.n_q_heads, w.head_dim), w.qk_scale))
    k = bf16_bits_to_f64(draw_bf16(rng, (N, w.n_kv_heads, w.head_dim), w.qk_scale))
    v = bf16_bits_to_f64(draw_bf16(rng, (N, w.n_kv_heads, w.head_dim)))
    t0 = time.perf_counter()
    oracle.sampled_forward(qr, k, v, np.arange(len(rows)), rows, np.arange(N))
    dt = time.perf_counter() - t0
    flops = 4.0 * w.head_dim * w.n_q_heads * float(np.sum(rows + 1))
    runs.append({"workload": w.name, "kind": "sampled",
                 "what": f"forward O and LSE at {len(rows)} seeded rows of the 1M-token "
                         "sequence, all heads, operands drawn for the sample",
                 "rows": int(len(rows)), "seconds": dt, "gflops": flops / dt / 1e9})
    return runs


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    import context_causal_attention_ring_gb300 as cpa

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()

    plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
                    layout=w.layout, variant="pass_kv", kv_prefix_len=w.kv_prefix_len)
    inp = make_inputs(w, with_dout=True)  # the step times forward and backward

    def dev_bf16(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)

    qn, kn, vn, don = (dev_bf16(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    q, k, v, do = (torch.empty_like(x) for x in (qn, kn, vn, don))
    plan.layout_apply(cpa.TENSOR_Q, cpa.TO_RANK_MAJOR, qn, q)
    plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, kn, k)
    plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, vn, v)
    plan.layout_apply(cpa.TENSOR_Q, cpa.TO_RANK_MAJOR, don, do)
    R, Hq, Hkv, d = plan.R, plan.Hq, plan.Hkv, plan.d
    o = torch.empty_like(q)
    lse = torch.empty((Hq, plan.T_q), dtype=torch.float32, device=dev)
    o_acc = torch.empty((plan.T_q, Hq, d), dtype=torch.float32, device=dev)
    delta = torch.empty((Hq, plan.T_q), dtype=torch.float32, device=dev)
    half_ops = torch.empty(plan.half_ops_size(), dtype=torch.uint8, device=dev)
    dq = torch.empty((plan.T_q, Hq, d), dtype=torch.float32, device=dev)
    dk = torch.empty((plan.T_kv, Hkv, d), dtype=torch.float32, device=dev)
    dv = torch.empty_like(dk)

    # consecutive ring steps on this stream are each other's only producers
    plan.set_chaining(True)
    pairs = [plan.visible_pairs(t) for t in range(R)]
    fwd_flops = 4.0 * d * Hq * sum(pairs)
    bwd_flops = 2.5 * fwd_flops

    def step(ev=None):
        # forward: R ring steps, running merge, last step writes bf16 O
        if ev is not None:
            ev[0].record(stream)
        for t in range(R):
            plan.step_fwd(t, q, k, v, o_acc, lse, cpa.ACCUMULATE,
                          o if t == R - 1 else None, stream)
        if ev is not None:
            ev[1].record(stream)
        # delta, zeroed accumulators and the fp16 operand copies, so that the
        # backward phase times the K2 launches alone
        plan.bwd_preprocess(q, k, v, o, do, delta, half_ops, dq, dk, dv, o_f32=o_acc,
                            stream=stream)
        if ev is not None:
            ev[2].record(stream)
        for t in range(R):
            plan.step_bwd_half(t, half_ops, lse, delta, dq, dk, dv, stream)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    plan.sync_status(stream)

    graphs = None
    launches_per_step = 0
    if args.graph:
        # the three phases captured once each; the timed region replays them
        graphs = []
        n0 = cpa.launch_count()
        cap = torch.cuda.Stream()  # capture needs a stream other than the default one

        def fwd_part():
            for t in range(R):
                plan.step_fwd(t, q, k, v, o_acc, lse, cpa.ACCUMULATE,
                              o if t == R - 1 else None, cap)

        def pre_part():
            plan.bwd_preprocess(q, k, v, o, do, delta, half_ops, dq, dk, dv, o_f32=o_acc,
                                stream=cap)

        def bwd_part():
            for t in range(R):
                plan.step_bwd_half(t, half_ops, lse, delta, dq, dk, dv, cap)

        cap.wait_stream(stream)
        for part in (fwd_part, pre_part, bwd_part):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                part()
            graphs.append(g)
        stream.wait_stream(cap)
        launches_per_step = cpa.launch_count() - n0
        for _ in range(args.warmup):
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()
        plan.sync_status(stream)

        def step(ev=None):  # noqa: F811 -- the replaying version
            with torch.cuda.stream(stream):
                for i, g in enumerate(graphs):
                    if ev is not None:
                        ev[i].record(stream)
                    g.replay()
                if ev is not None:
                    ev[3].record(stream)

    events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)]
              for _ in range(args.steps)]
    clocks_csv = (args.clocks_csv.replace("{rank}", str(rank)) if args.clocks_csv
                  else os.path.join(tempfile.gettempdir(), f"cp_attn_clocks_rank{rank}.csv"))
    sampler = ClockSampler(local, clocks_csv)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n_launch0 = cpa.launch_count()
    for i in range(args.steps):
        step(events[i])
    torch.cuda.synchronize()
    n_launches = cpa.launch_count() - n_launch0 + launches_per_step * args.steps
    if ws > 1:
        dist.barrier()
    clocks = sampler.stop()
    plan.sync_status(stream)

    fwd_ms = [e[0].elapsed_time(e[1]) for e in events]
    pre_ms = [e[1].elapsed_time(e[2]) for e in events]
    bwd_ms = [e[2].elapsed_time(e[3]) for e in events]
    step_ms = [e[0].elapsed_time(e[3]) for e in events]
    total_ms = max_over_ranks(events[0][0].elapsed_time(events[-1][3]), dev)
    ms_per_step = total_ms / args.steps
    q_mib = plan.T_q * Hq * d * 2 / 2**20
    l2_note = (f"inputs larger than L2 (Q {q_mib:.0f} MiB, dO {q_mib:.0f} MiB)"
               if 2 * q_mib > 129 else
               f"inputs fit in L2 (Q {q_mib:.1f} MiB): a launch-bound small case, warm L2")
    value = whole_job_tflops(ws, fwd_flops + bwd_flops, ms_per_step)
    fwd_tflops = fwd_flops / (statistics.median(fwd_ms) * 1e-3) / 1e12
    bwd_tflops = bwd_flops / (statistics.median(bwd_ms) * 1e-3) / 1e12

    peaks, peak_kind = _peaks()
    # dominant kernel: the one with more device time per step
    if sum(bwd_ms) >= sum(fwd_ms):
        dom, dom_flops, dom_ms = "step_bwd", bwd_flops, sum(bwd_ms) / args.steps
    else:
        dom, dom_flops, dom_ms = "step_fwd", fwd_flops, sum(fwd_ms) / args.steps
    achieved = (dom_flops / R) / (dom_ms / R * 1e-3) / 1e12
    roofline = roofline_record(dom, achieved, dom_flops / R, peaks, peak_kind, clocks)
    roofline["traffic"] = _profiled_traffic(dom)

    # end to end through the public whole-op calls with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, plan, inp, dev, stream, fwd_flops + bwd_flops, ws)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        heads = int(os.environ.get("CP_BENCH_CPU_HEADS", str(w.n_q_heads)))
        val, dt, desc = cpu_oracle_sample(w, heads, inp)
        cpu = {"value": val, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
               "sample": desc, "seconds": dt}
        if not args.no_configs:
            cpu["plan_runs"] = cpu_oracle_plan_runs()

    # the other workloads' figures (not the headline): the tiny ring in
    # microseconds and the packed documents in TFLOPS
    configs = None
    if rank == 0 and ws == 1 and not args.no_configs:
        del inp
        configs = [time_config(WORKLOADS[name], n, 3, dev)
                   for name, n in (("tiny_ring", 20), ("packed_docs", 5))]
        configs[0]["fwd_us"] = configs[0]["fwd_ms"] * 1e3
        configs[0]["bwd_us"] = configs[0]["bwd_ms"] * 1e3
        configs[0]["step_us"] = configs[0]["step_ms"] * 1e3

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "seq_len": w.seq_len, "cp": w.cp,
                       "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": d,
                       "layout": w.layout, "variant": "pass_kv", "parallelism": f"replicas{ws}",
                       "l2": l2_note,
                       "launch": "cuda_graph replay" if args.graph else "stream",
                       "flops_per_step": fwd_flops + bwd_flops},
            "fwd_tflops": fwd_tflops, "bwd_tflops": bwd_tflops,
            "fwd_ms": statistics.median(fwd_ms), "bwd_ms": statistics.median(bwd_ms),
            "preprocess_ms": statistics.median(pre_ms),
            "pct_of_peak_burst": 100.0 * value / ws / peaks["bf16_tflops"],
            "gpu_launches": n_launches,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_variant_sweep(args):
    """Pass KV against Pass Q for partial prefill at several KV-cache hit
    rates (405B-shaped heads: 128 query / 8 KV heads, d = 128, R = 8, 65536
    tokens in all): the forward time of each ordering on this GPU, the
    library's choice (cp_attn_select_variant) and the per-hop ring message
    each ordering would send. On one GPU the ring is emulated, so the times
    show the compute side only; the messages show the communication side the
    choice is made on."""
    import torch
    import context_causal_attention_ring_gb300 as cpa
    from workloads import Workload

    torch.cuda.set_device(0)
    R, Hq, Hkv, d, total = 8, 128, 8, 128, 65536
    rows = []
    for n_new in (65536, 32768, 16384, 8192, 4096, 2048):
        w = Workload(f"sweep_{n_new}", n_new, Hq, Hkv, d, R, kv_prefix_len=total - n_new)
        inp = make_inputs(w, with_dout=False)
        dev_bf16 = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
        qn, kn, vn = (dev_bf16(x) for x in (inp.q, inp.k, inp.v))
        del inp
        row = {"n_new": n_new, "n_cached": total - n_new, "hit_rate": 1 - n_new / total,
               "chosen": cpa.select_variant(n_new, total - n_new, Hq, Hkv),
               "q_msg_bytes_per_hop": n_new // R * Hq * d * 2,
               "kv_msg_bytes_per_hop": 2 * (total // R) * Hkv * d * 2}
        for variant in ("pass_kv", "pass_q"):
            plan = cpa.Plan(n_new, R, Hq, Hkv, d, variant=variant, kv_prefix_len=total - n_new)
            q, k, v = torch.empty_like(qn), torch.empty_like(kn), torch.empty_like(vn)
            plan.layout_apply(cpa.TENSOR_Q, cpa.TO_RANK_MAJOR, qn, q)
            plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, kn, k)
            plan.layout_apply(cpa.TENSOR_KV, cpa.TO_RANK_MAJOR, vn, v)
            o = torch.empty_like(q)
            lse = torch.empty((Hq, plan.T_q), dtype=torch.float32, device="cuda")
            ws = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
            for _ in range(max(1, args.warmup)):
                plan.forward(q, k, v, o, lse, ws)
            times = []
            for _ in range(max(3, args.steps)):
                e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
                e0.record()
                plan.forward(q, k, v, o, lse, ws)
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1))
            plan.sync_status()
            flops = 4.0 * d * Hq * plan.visible_pairs()
            ms = statistics.median(times)
            row[variant] = {"fwd_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
            del q, k, v, o, lse, ws, plan
            torch.cuda.empty_cache()
        rows.append(row)
        del qn, kn, vn
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "pass_kv_vs_pass_q_forward", "unit": "ms", "config": {
        "workload": "405B-shaped partial prefill sweep", "total_tokens": total, "cp": R,
        "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": d}, "rows": rows}), flush=True)


def run_usp_sweep(args):
    """The 32768-token 32/8-head layer on D = 8 emulated devices, as a plain
    zigzag ring (a2a = 1, 8 steps), USP with a2a = 2 and 4 (4 and 2 steps of
    longer chunks) and pure Ulysses (a2a = 8, one step). Per arrangement: the
    forward and backward time of all a2a head-group rings, and the head
    all-to-all kernel's bandwidth on Q."""
    import torch
    import context_causal_attention_ring_gb300 as cpa

    torch.cuda.set_device(0)
    w = WORKLOADS["llama3_8b_layer"]
    N, Hq, Hkv, d, D = w.seq_len, w.n_q_heads, w.n_kv_heads, w.head_dim, w.cp
    inp = make_inputs(w, with_dout=True)  # the step times forward and backward
    dev_bf16 = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).cuda()
    qn, kn, vn, don = (dev_bf16(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    del inp
    peaks, _ = _peaks()
    rows = []
    for U in (1, 2, 4, 8):
        R = D // U
        hq, hkv = Hq // U, Hkv // U
        plan = cpa.Plan(N, R, hq, hkv, d, layout="usp", a2a=U)
        T = plan.T_q

        def pooled(x, heads, kind):
            y = torch.empty_like(x)
            plan.layout_apply(kind, cpa.TO_RANK_MAJOR, x, y, row_bytes=heads * d * 2)
            s_ = torch.empty((U, T, heads // U, d), dtype=x.dtype, device="cuda")
            cpa.head_a2a(y, s_, U, cpa.SPLIT_HEADS)
            return y, s_

        qy, qs = pooled(qn, Hq, cpa.TENSOR_Q)
        _, ks = pooled(kn, Hkv, cpa.TENSOR_KV)
        _, vs = pooled(vn, Hkv, cpa.TENSOR_KV)
        _, dos = pooled(don, Hq, cpa.TENSOR_Q)
        os_ = torch.empty_like(qs)
        lse = torch.empty((Hq, T), dtype=torch.float32, device="cuda")
        dqs = torch.empty((U, T, hq, d), device="cuda")
        dks = torch.empty((U, T, hkv, d), device="cuda")
        dvs = torch.empty_like(dks)
        wsf = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device="cuda")
        wsb = torch.empty(plan.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device="cuda")

        def fwd():
            for u in range(U):
                plan.forward(qs[u], ks[u], vs[u], os_[u], lse[u * hq:(u + 1) * hq], wsf)

        def bwd():
            for u in range(U):
                plan.backward(qs[u], ks[u], vs[u], os_[u], lse[u * hq:(u + 1) * hq], dos[u],
                              dqs[u], dks[u], dvs[u], wsb, o_f32=wsf)

        def a2a():
            cpa.head_a2a(qy, qs, U, cpa.SPLIT_HEADS)

        def timed(fn, n):
            for _ in range(max(1, args.warmup)):
                fn()
            ts = []
            for _ in range(n):
                e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
                e0.record()
                fn()
                e1.record()
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            return statistics.median(ts)

        # the backward of each head group needs its own forward's fp32 O:
        # time them as a pair, and the forward alone
        f_ms = timed(fwd, max(3, args.steps))

        def fb():
            for u in range(U):
                plan.forward(qs[u], ks[u], vs[u], os_[u], lse[u * hq:(u + 1) * hq], wsf)
                plan.backward(qs[u], ks[u], vs[u], os_[u], lse[u * hq:(u + 1) * hq], dos[u],
                              dqs[u], dks[u], dvs[u], wsb, o_f32=wsf)

        fb_ms = timed(fb, max(3, args.steps))
        a_ms = timed(a2a, max(3, args.steps))
        plan.sync_status()
        flops = 4.0 * d * Hq * plan.visible_pairs()
        a2a_bytes = 2 * T * Hq * d * 2
        rows.append({"a2a": U, "ring_steps": R, "chunk_tokens": N // (2 * D) * U,
                     "fwd_ms": f_ms, "fwd_tflops": flops / (f_ms * 1e-3) / 1e12,
                     "fwd_bwd_ms": fb_ms, "fwd_bwd_tflops": 3.5 * flops / (fb_ms * 1e-3) / 1e12,
                     "head_a2a_q_ms": a_ms, "head_a2a_q_gbs": a2a_bytes / (a_ms * 1e-3) / 1e9,
                     "head_a2a_frac_of_hbm": a2a_bytes / (a_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]})
        del plan, qy, qs, ks, vs, dos, os_, lse, dqs, dks, dvs, wsf, wsb
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "usp_arrangements", "unit": "ms", "config": {
        "workload": w.name, "seq_len": N, "devices": D, "n_q_heads": Hq, "n_kv_heads": Hkv,
        "head_dim": d}, "rows": rows}), flush=True)


def run_decode_bench(args):
    """One-row decode over the emulated ring (cp_attn_decode: the partials over
    runs of keys and the K4 merge) on two shapes: a 405B-shaped row (128 / 8
    heads) over 131072 keys on 8 ranks, and a batch of 16 sequences with
    8B-shaped heads (32 / 8) over 32768 keys each; each with a bf16 KV cache
    and with an E4M3 one (cp_attn_decode_fp8, K and V quantized per tensor
    before the timed calls). Both read more K/V than the L2 holds. The
    roofline is HBM: algorithmic bytes = K + V (at their element size) + q + o
    (+ the LSE), once."""
    import torch
    import context_causal_attention_ring_gb300 as cpa
    from workloads import make_decode_inputs

    torch.cuda.set_device(0)
    peaks, peak_kind = _peaks()
    rows = []

    def time_calls(call):
        """(GPU ms per call, host-inclusive median ms per call, launches per
        call). The GPU time is that of n back-to-back calls enqueued behind a
        ~20 ms device sleep, so that the host's enqueue time never leaves the
        stream idle; the second figure brackets each call with its own events
        as it is enqueued, and so also holds the host's per-call overhead
        whenever that is longer than the call."""
        for _ in range(max(3, args.warmup)):
            call()
        n = max(20, args.steps)
        ev = [(torch.cuda.Event(True), torch.cuda.Event(True)) for _ in range(n)]
        n0 = cpa.launch_count()
        for e0, e1 in ev:
            e0.record()
            call()
            e1.record()
        torch.cuda.synchronize()
        host_ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        launches = (cpa.launch_count() - n0) // n
        a, b = torch.cuda.Event(True), torch.cuda.Event(True)
        torch.cuda._sleep(40_000_000)
        a.record()
        for _ in range(n):
            call()
        b.record()
        torch.cuda.synchronize()
        cpa.decode_sync_status()
        return a.elapsed_time(b) / n, host_ms, launches

    def quantize(x, n_rows, heads, d, transpose):
        amax = torch.zeros(4, dtype=torch.float32, device="cuda")
        scale = torch.zeros(4, dtype=torch.float32, device="cuda")
        cpa.fp8_absmax(x, n_rows * heads * d, amax)
        out = torch.empty((heads, d, n_rows) if transpose else (n_rows, heads, d),
                          dtype=torch.uint8, device="cuda")
        cpa.fp8_quantize(x, n_rows, heads, d, amax, out, scale, transpose=transpose)
        return out, scale

    for name, B, T, Hq, Hkv, d, R in (("405b_row_131072", 1, 131072, 128, 8, 128, 8),
                                      ("8b_batch16_32768", 16, 32768, 32, 8, 128, 8)):
        q, k, v = make_decode_inputs(B, T, Hq, Hkv, d, seed=3)
        dev_bf16 = lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(
            torch.bfloat16).cuda()
        qd, kd, vd = dev_bf16(q), dev_bf16(k), dev_bf16(v)
        del q, k, v
        o = torch.empty_like(qd)
        lse = torch.empty((Hq, B), dtype=torch.float32, device="cuda")
        ws = torch.empty(cpa.decode_workspace_size(B, R, T, Hq, Hkv, d), dtype=torch.uint8,
                         device="cuda")
        k8, sk = quantize(kd.view(B * T, Hkv, d), B * T, Hkv, d, False)
        vt8, sv = quantize(vd.view(B * T, Hkv, d), B * T, Hkv, d, True)
        scales = torch.stack([sk[0], sv[0]])
        for kv_dtype, elt, call in (
                ("bf16", 2, lambda: cpa.decode(qd, kd, vd, o, lse, ws, R)),
                ("e4m3", 1, lambda: cpa.decode_fp8(qd, k8, vt8, scales, o, lse, ws, R))):
            ms, host_ms, launches = time_calls(call)
            algo = 2 * B * T * Hkv * d * elt + 2 * B * Hq * d * 2 + Hq * B * 4
            gbs = algo / (ms * 1e-3) / 1e9
            rows.append({"workload": name, "kv_dtype": kv_dtype, "batch": B, "kv_len": T,
                         "n_q_heads": Hq, "n_kv_heads": Hkv, "head_dim": d, "cp": R, "ms": ms,
                         "ms_per_call_host": host_ms,
                         "algorithmic_bytes": algo, "achieved_gbs": gbs,
                         "frac_of_hbm": gbs / peaks["hbm_gbs"], "launches_per_call": launches})
        del qd, kd, vd, o, lse, ws, k8, vt8
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "decode_hbm_bandwidth", "unit": "GB/s",
                      "peak": peaks["hbm_gbs"], "peak_kind": f"hbm_gbs ({peak_kind})",
                      "timing": "ms: GPU time per call, back-to-back calls on a stream kept busy; "
                                "ms_per_call_host: median of calls bracketed one by one",
                      "rows": rows}), flush=True)


def run_fp8_bench(args):
    """FP8 (E4M3) against bf16 on the 405B-shaped prefill (131072 new tokens,
    128 query / 8 KV heads, d = 128, CP = 8 zigzag), both orderings, forward
    only: the ring of K1 steps (cp_attn_forward_fp8 / cp_attn_forward), each
    timed with CUDA events after warm-up; the quantization kernels (absmax,
    quantize, V^T) are timed apart. TFLOPS count unmasked FLOPs (4 d per
    visible pair per query head). The FP8 roofline peak is the measured bf16
    burst peak times the nominal fp8 / bf16 ratio (2)."""
    import torch
    import context_causal_attention_ring_gb300 as cpa

    torch.cuda.set_device(0)
    peaks, peak_kind = _peaks()
    w = WORKLOADS[args.fp8_workload]
    inp = make_inputs(w, with_dout=False)
    dev = torch.device("cuda:0")
    rows = []
    for variant in ("pass_kv", "pass_q"):
        plan = cpa.Plan(w.seq_len, w.cp, w.n_q_heads, w.n_kv_heads, w.head_dim,
                        layout=w.layout, variant=variant, kv_prefix_len=w.kv_prefix_len)
        R, Hq, Hkv, d = plan.R, plan.Hq, plan.Hkv, plan.d
        flops = 4.0 * d * Hq * plan.visible_pairs()
        bf = {}
        for name, bits in (("q", inp.q), ("k", inp.k), ("v", inp.v)):
            x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(dev)
            y = torch.empty_like(x)
            plan.layout_apply(cpa.TENSOR_Q if name == "q" else cpa.TENSOR_KV, cpa.TO_RANK_MAJOR,
                              x, y)
            bf[name] = y
            del x
        T_q, T_kv = plan.T_q, plan.T_kv
        amax = torch.zeros(4, dtype=torch.float32, device=dev)
        scales = torch.zeros(4, dtype=torch.float32, device=dev)
        q8 = torch.empty((T_q, Hq, d), dtype=torch.uint8, device=dev)
        k8 = torch.empty((T_kv, Hkv, d), dtype=torch.uint8, device=dev)
        vt8 = torch.empty((Hkv, d, T_kv), dtype=torch.uint8, device=dev)

        def quantize():
            for i, (x, out, rws, hh, tr) in enumerate(((bf["q"], q8, T_q, Hq, False),
                                                        (bf["k"], k8, T_kv, Hkv, False),
                                                        (bf["v"], vt8, T_kv, Hkv, True))):
                cpa.fp8_absmax(x, rws * hh * d, amax[i:i + 1])
                cpa.fp8_quantize(x, rws, hh, d, amax[i:i + 1], out, scales[i:i + 1], transpose=tr)

        o = torch.empty((T_q, Hq, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((Hq, T_q), dtype=torch.float32, device=dev)
        ws = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device=dev)
        calls = {"fp8": lambda: plan.forward_fp8(q8, k8, vt8, scales, o, lse, ws),
                 "bf16": lambda: plan.forward(bf["q"], bf["k"], bf["v"], o, lse, ws),
                 "quantize": quantize}
        res = {}
        for name, fn in calls.items():
            for _ in range(max(3, args.warmup)):
                if name == "fp8":
                    quantize()
                fn()
            n = max(5, min(args.steps, 10))
            ev = [(torch.cuda.Event(True), torch.cuda.Event(True)) for _ in range(n)]
            for e0, e1 in ev:
                e0.record()
                fn()
                e1.record()
            torch.cuda.synchronize()
            res[name] = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        plan.sync_status()
        qbytes = 2 * (T_q * Hq * d * 2 + 2 * T_kv * Hkv * d * 2) + T_q * Hq * d + 2 * T_kv * Hkv * d
        rows.append({"variant": variant, "flops": flops,
                     "fp8_ms": res["fp8"], "fp8_tflops": flops / (res["fp8"] * 1e-3) / 1e12,
                     "bf16_ms": res["bf16"], "bf16_tflops": flops / (res["bf16"] * 1e-3) / 1e12,
                     "quantize_ms": res["quantize"],
                     "quantize_gbs": qbytes / (res["quantize"] * 1e-3) / 1e9})
        del bf, q8, k8, vt8, o, lse, ws
        torch.cuda.empty_cache()
    print(json.dumps({"metric": "fp8 vs bf16 forward TFLOPS (unmasked FLOPs)",
                      "workload": f"{w.name}: {w.seq_len} new tokens after {w.kv_prefix_len} cached, "
                                  f"{w.n_q_heads}/{w.n_kv_heads} heads, d={w.head_dim}, "
                                  f"CP={w.cp} {w.layout}",
                      "fp8_peak_tflops": 2 * peaks["bf16_tflops"],
                      "bf16_peak_tflops": peaks["bf16_tflops"],
                      "peak_kind": f"bf16_tflops burst ({peak_kind}); fp8 = 2 x bf16 (nominal ratio)",
                      "hbm_gbs": peaks["hbm_gbs"], "rows": rows}), flush=True)


def run_e2e(args, plan, inp, dev, stream, flops, ws):
    """End to end through the public whole-op calls with host buffers. Every
    step copies its inputs from pinned host memory, runs the layout
    permutes, cp_attn_forward and cp_attn_backward, permutes the results back
    and reads them into pinned host memory. Steps are pipelined over two
    buffer sets: step i's copies (on a copy stream) overlap step i-1's and
    step i+1's compute; events order each step's copy-in, compute and
    copy-out, and a set is reused only after its previous copy-out."""
    import torch
    import context_causal_attention_ring_gb300 as cpa

    def pinned(bits):
        t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    hq, hk, hv, hdo = (pinned(x) for x in (inp.q, inp.k, inp.v, inp.dout))
    h2d_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)

    class BufSet:
        def __init__(self):
            self.d_nat = [torch.empty(x.shape, dtype=x.dtype, device=dev) for x in (hq, hk, hv, hdo)]
            self.d_rm = [torch.empty_like(x) for x in self.d_nat]
            self.o = torch.empty_like(self.d_rm[0])
            self.o_nat = torch.empty_like(self.o)
            self.lse = torch.empty((plan.Hq, plan.T_q), dtype=torch.float32, device=dev)
            self.dq = torch.empty((plan.T_q, plan.Hq, plan.d), dtype=torch.float32, device=dev)
            self.dk = torch.empty((plan.T_kv, plan.Hkv, plan.d), dtype=torch.float32, device=dev)
            self.dv = torch.empty_like(self.dk)
            self.g_nat = [torch.empty_like(x) for x in (self.dq, self.dk, self.dv)]
            self.h_out = [torch.empty(x.shape, dtype=x.dtype).pin_memory()
                          for x in (self.o_nat, self.lse, *self.g_nat)]
            self.ev_in = torch.cuda.Event()
            self.ev_done = torch.cuda.Event()
            self.ev_out = torch.cuda.Event()
            self.used = False

    sets = [BufSet(), BufSet()]
    ws_f = torch.empty(plan.workspace_size(cpa.OP_FORWARD), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(plan.workspace_size(cpa.OP_BACKWARD), dtype=torch.uint8, device=dev)
    h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hdo))
    d2h = sum(x.numel() * x.element_size() for x in sets[0].h_out)
    kinds = (cpa.TENSOR_Q, cpa.TENSOR_KV, cpa.TENSOR_KV, cpa.TENSOR_Q)

    def step(i):
        b = sets[i % 2]
        with torch.cuda.stream(h2d_stream):
            if b.used:
                h2d_stream.wait_event(b.ev_done)      # its inputs were consumed
            for h, dd in zip((hq, hk, hv, hdo), b.d_nat):
                dd.copy_(h, non_blocking=True)
            b.ev_in.record(h2d_stream)
        stream.wait_event(b.ev_in)
        if b.used:
            stream.wait_event(b.ev_out)               # its outputs were read back
        for kind, x, y in zip(kinds, b.d_nat, b.d_rm):
            plan.layout_apply(kind, cpa.TO_RANK_MAJOR, x, y, stream=stream)
        plan.forward(b.d_rm[0], b.d_rm[1], b.d_rm[2], b.o, b.lse, ws_f, stream=stream)
        plan.backward(b.d_rm[0], b.d_rm[1], b.d_rm[2], b.o, b.lse, b.d_rm[3], b.dq, b.dk, b.dv,
                      ws_b, o_f32=ws_f, stream=stream)
        plan.layout_apply(cpa.TENSOR_Q, cpa.TO_NATURAL, b.o, b.o_nat, stream=stream)
        plan.layout_apply(cpa.TENSOR_Q, cpa.TO_NATURAL, b.dq, b.g_nat[0], stream=stream)
        plan.layout_apply(cpa.TENSOR_KV, cpa.TO_NATURAL, b.dk, b.g_nat[1], stream=stream)
        plan.layout_apply(cpa.TENSOR_KV, cpa.TO_NATURAL, b.dv, b.g_nat[2], stream=stream)
        b.ev_done.record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(b.ev_done)
            for h, dd in zip(b.h_out, (b.o_nat, b.lse, *b.g_nat)):
                h.copy_(dd, non_blocking=True)
            b.ev_out.record(d2h_stream)
        b.used = True

    for i in range(max(1, args.warmup)):
        step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d_stream.wait_event(e0)
    d2h_stream.wait_event(e0)
    for i in range(args.steps):
        step(i)
    stream.wait_stream(h2d_stream)
    stream.wait_stream(d2h_stream)
    e1.record(stream)
    torch.cuda.synchronize()
    plan.sync_status(stream)
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    # latency of one call with host buffers, nothing overlapped: copy-in,
    # compute and copy-out of a single step with the device otherwise idle
    lat = []
    for i in range(3):
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        h2d_stream.wait_event(s0)
        step(i)
        stream.wait_stream(d2h_stream)
        s1.record(stream)
        torch.cuda.synchronize()
        lat.append(s0.elapsed_time(s1))
    lat_ms = max_over_ranks(statistics.median(lat), dev)
    return {"value": whole_job_tflops(ws, flops, ms), "unit": UNIT, "ms_per_step": ms,
            "latency_ms_unpipelined": lat_ms,
            "value_unpipelined": whole_job_tflops(ws, flops, lat_ms),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "pinned host -> device, layout to rank-major, cp_attn_forward, "
                    "cp_attn_backward, layout to natural, device -> pinned host; "
                    "copies on their own streams, pipelined over two buffer sets; "
                    "latency_ms_unpipelined: one step alone, copies not overlapped"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3_8b_layer", choices=sorted(WORKLOADS))
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' figures (tiny ring, packed documents)")
    ap.add_argument("--q-heads", type=int, default=0,
                    help="profiling aid: override the workload's query heads")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="profiling aid: override the workload's KV heads")
    ap.add_argument("--variant-sweep", action="store_true",
                    help="time Pass KV against Pass Q at several KV-cache hit rates")
    ap.add_argument("--usp-sweep", action="store_true",
                    help="time the layer as zigzag ring, USP and pure Ulysses arrangements")
    ap.add_argument("--graph", action="store_true",
                    help="time replays of the step captured as CUDA graphs (launch-bound shapes)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the FP8 (E4M3) forward against bf16 on the 405B-shaped prefill")
    ap.add_argument("--fp8-workload", default="prefill_405b_full", choices=sorted(WORKLOADS),
                    help="workload of --fp8")
    ap.add_argument("--clocks-csv", default=None,
                    help="where the nvidia-smi clock samples of the timed region go "
                         "('{rank}' is replaced by the rank); a temporary file by default")
    ap.add_argument("--decode", action="store_true",
                    help="time the one-row decode against the HBM roofline")
    args = ap.parse_args()
    if args.fp8:
        run_fp8_bench(args)
        return
    if args.decode:
        run_decode_bench(args)
        return
    if args.variant_sweep:
        run_variant_sweep(args)
        return
    if args.usp_sweep:
        run_usp_sweep(args)
        return
    w = WORKLOADS[args.workload]
    if args.q_heads or args.kv_heads:
        import dataclasses
        w = dataclasses.replace(w, n_q_heads=args.q_heads or w.n_q_heads,
                                n_kv_heads=args.kv_heads or w.n_kv_heads,
                                name=w.name + f"_h{args.q_heads or w.n_q_heads}"
                                     f"kv{args.kv_heads or w.n_kv_heads}")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
