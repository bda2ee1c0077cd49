#!/usr/bin/env python3
"""Benchmark of the Switch top-1 MoE layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config base]
    python bench.py --impl reference ...      # the CPU oracle, timed alone

One step = one switch_moe_forward() over one batch of the workload
(router, scan + L_aux, slot assignment + dispatch, expert GEMM 1, expert
GEMM 2, combine).  Prints ONE JSON line (rank 0):

  value      tokens/s of the whole job, inputs resident in HBM, timed with
             CUDA events over exactly K steps between barriers; each step
             replays the whole forward captured once into a CUDA graph (as
             a serving loop does; eager calls are timed too, reported in
             "timing", and are the fallback if capture fails; --eager
             times eager calls only)
  e2e        the same through switch_moe_forward_hostio(): x copied from
             pinned host memory and every output copied back inside the
             timed region
  roofline   the expert GEMMs (the dominant kernel) against the measured
             HBM copy bandwidth, from per-phase CUDA events on the stream
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload

With --gpus N > 1 (launched by torch.distributed.run) every rank runs an
independent replica of the layer on its own GPU: the forward has no data
exchange, so there is no collective on the data path; only the barriers and
the max-over-ranks of the timed region use the process group.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import CONFIGS, expert_weights, make_inputs, zipf_bias  # noqa: E402

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the dominant kernel, from the ncu captures summarised in profiles/: the
# one-launch expert FFN (ffn_tc_kernel) where the workload uses it, else the
# mean of the two gemm_tc_kernel launches.  Valid only for the kernel source
# it was taken on (sha256 of the .cu file); any other source reports null.
NCU_TRAFFIC = {
    "base": {"source": "ffn_tc.cu",
             "sha256": "f5ef46009d9600e77aafa2ed11ec17daa742959dc9f87abfb7f69c01b4afded6",
             "bytes_per_launch": (1266.399 + 87.187) * 1e6},
}
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
CPU_SAMPLE_EXPERTS = 16


def kernel_traffic(config: str):
    rec = NCU_TRAFFIC.get(config)
    if not rec:
        return None
    import hashlib
    src = os.path.join(ROOT, "switch_top_expert_router_b300", "csrc", rec["source"])
    with open(src, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != rec["sha256"]:
            return None
    return rec["bytes_per_launch"]


def gemm2_ksplit(w, C: int) -> int:
    """K splits of the second routed GEMM, by the library's rule: token
    tiles up to 128 take the one-launch FFN (no split); wider ones split the
    K = d_ff reduction (in powers of two, at most 8) only while there are
    fewer than two (expert, token tile, 128-row) tiles per SM of a 148-SM
    B300."""
    bn = min(-(-C // 16) * 16, 256)
    if bn <= 128:
        return 1
    tiles = w.N * -(-C // bn) * -(-w.d_model // 128)
    k_blocks = -(-w.d_ff // 64)
    s = 1
    while s < 8 and tiles * s < 2 * 148 and k_blocks % (2 * s) == 0:
        s *= 2
    return s


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of every rank's value (each rank's timed region); the
    job is as slow as its slowest replica.  Identity without a group."""
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(T: int, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank processed `steps` batches of T tokens
    within the (max-over-ranks) `ms` milliseconds."""
    return T * steps * world / (ms / 1e3)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ oracle sample
def oracle_sample_step(w, seed=0, expand=1, top_k=1, renormalize=0, expert_choice=0):
    """One bounded CPU-oracle step on the workload: route the whole batch
    (with Expanded Drop over `expand` candidates when > 1, or top-2), then the
    expert FFN and combine of the tokens processed by the first
    CPU_SAMPLE_EXPERTS experts (top-2: of the token-choice pairs, counted as
    half a token each).  Returns (tokens processed, seconds)."""
    import oracle
    inp = make_inputs(w, seed, device="cpu", with_experts=False)
    experts = {e: expert_weights(w, e, seed, "cpu") for e in range(min(CPU_SAMPLE_EXPERTS, w.N))}
    t0 = time.perf_counter()
    r = oracle.route(inp.x, inp.W_g, zipf_bias(w))
    C = oracle.capacity(w.T, w.N, w.capacity_factor)
    if expert_choice:
        chosen, gates = oracle.expert_choice(r["probs"], C)
        slots = 0
        for e in experts:
            oracle.forward_rows_expert_choice(chosen[e], inp.x, chosen[e:e + 1], gates[e:e + 1],
                                              w.gate_multiply, lambda i: experts[e])
            slots += chosen.shape[1]
        oracle.aux_loss(r["probs"], np.bincount(r["expert_id"], minlength=w.N))
        # a token holds N * k / T slots on average
        return slots * w.T / (w.N * chosen.shape[1]), time.perf_counter() - t0
    if top_k == 2:
        c = oracle.candidates(r["logits"], 2)
        g2 = oracle.top2_gates(r["probs"], c, renormalize)
        s2, _, _ = oracle.assign_slots_top2(c, w.N, C)
        pairs = 0
        for k in range(2):
            rows = np.nonzero(c[:, k] < len(experts))[0]
            oracle.forward_rows(rows, inp.x, c[:, k], g2[:, k], s2[:, k], w.gate_multiply,
                                lambda i: experts[i])
            pairs += int(rows.size)
        oracle.aux_loss(r["probs"], np.bincount(c[:, 0], minlength=w.N))
        return pairs / 2, time.perf_counter() - t0
    slot, drop, counts = oracle.assign_slots(r["expert_id"], r["gate"], w.N, C, w.priority_mode)
    e, g = r["expert_id"], r["gate"]
    if expand > 1:
        e, slot, drop, _ = oracle.assign_slots_expanded(oracle.candidates(r["logits"], expand),
                                                        w.N, C)
        g = r["probs"][np.arange(w.T), e]
    rows = np.nonzero(e < len(experts))[0]
    oracle.forward_rows(rows, inp.x, e, g, slot, w.gate_multiply,
                        lambda i: experts[i], inp.W1s, inp.W2s)
    oracle.aux_loss(r["probs"], counts)
    return int(rows.size), time.perf_counter() - t0


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_sample_desc(w):
    return (f"{w.name} layer: routing of all {w.T} tokens + expert FFN and combine of the "
            f"tokens routed to experts 0..{min(CPU_SAMPLE_EXPERTS, w.N) - 1} "
            f"(of {w.N}); value = those tokens / wall time")


def run_reference(args, rank, world):
    w = CONFIGS[args.config]
    if args.token_order:
        w = w.replace(priority_mode=0)
    if rank != 0:
        return
    kw = dict(expand=args.expand, top_k=args.top_k, renormalize=args.renormalize,
              expert_choice=args.expert_choice)
    for _ in range(args.warmup):
        oracle_sample_step(w, **kw)
    tok, sec = 0, 0.0
    for _ in range(args.steps):
        n, s = oracle_sample_step(w, **kw)
        tok += n
        sec += s
    value = tok / sec
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": "top-1 MoE layer tokens/sec", "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, args.expand, args.top_k, args.renormalize,
                                  args.expert_choice),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": cpu_sample_desc(w)},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w, expand=1, top_k=1, renormalize=0, expert_choice=0):
    route = ("top-2" + (" (gates renormalised over the pair)" if renormalize else "")
             if top_k == 2 else "Switch top-1")
    if expert_choice:
        route = "expert-choice"
    return {"workload": f"{w.name}: {route} MoE layer T={w.T} d_model={w.d_model} "
                        f"d_ff={w.d_ff} N={w.N} cf={w.capacity_factor} {w.dtype}"
                        f"{' +shared expert' if w.has_shared else ''}"
                        f"{f' +Expanded Drop over {expand} candidates' if expand > 1 else ''}",
            "expanded_drop_candidates": expand, "top_k": top_k, "expert_choice": expert_choice,
            "T": w.T, "d_model": w.d_model, "d_ff": w.d_ff, "N": w.N,
            "capacity_factor": w.capacity_factor,
            "priority": "gate" if w.priority_mode else "token-order",
            "gate_multiply": w.gate_multiply, "parallelism": "replicas",
            "l2": "inputs larger than L2: every step streams the active experts' weights "
                  "(far above the 126 MB L2) from HBM"}


FP32_FFMA_TFLOPS = 148 * 128 * 2 * 2.032 / 1e3   # B300: SMs x FP32 lanes x 2 flop x max GHz


def run_backward(args, sm, rank, world, local):
    """--backward: K calls of switch_moe_backward on the workload (the
    forward's routing computed once before), timed with CUDA events.  The
    backward runs on FFMA, so its roofline is the fp32 FMA peak (148 SMs x
    128 lanes x 2 flop at the 2032 MHz maximum clock); its algorithmic
    flops are 12 kept x d x F (six slot-sized contractions: the hidden
    activation, the expert output, dH, dX, dW1, dW2) + 6 T N d (router
    logits, dW_g, dx through W_g), shared expert extra."""
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    w = CONFIGS[args.config]
    if args.token_order:
        w = w.replace(priority_mode=0)
    inp = make_inputs(w, seed=0, device=dev)
    dy = torch.randn(w.T, w.d_model, generator=torch.Generator().manual_seed(7)).to(dev)
    alpha = 0.01
    fwd = sm.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, w.capacity_factor,
                                w.priority_mode, w.gate_multiply, b_g=inp.b_g, W1s=inp.W1s,
                                W2s=inp.W2s)
    p = sm.make_params(w.T, w.d_model, w.d_ff, w.N, w.capacity_factor, w.priority_mode,
                       w.gate_multiply, sm.BF16 if w.dtype == "bf16" else sm.F32, w.has_shared)
    ws = sm.workspace(sm.switch_moe_backward_workspace_bytes(p), dev)

    def step():
        sm.switch_moe_backward(inp.x, inp.W_g, inp.W1, inp.W2, w.capacity_factor, fwd, dy,
                               aux_coef=alpha, priority_mode=w.priority_mode,
                               gate_multiply=w.gate_multiply, b_g=inp.b_g, W1s=inp.W1s,
                               W2s=inp.W2s, ws=ws)

    for _ in range(args.warmup):
        step()
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1), pg, dev)
    clk = clocks.stop()
    rc = sm.switch_moe_sync_status()
    if rc != 0:
        raise RuntimeError(f"device status after timing: {sm.strerror(rc)}")
    C = sm.switch_moe_capacity(w.T, w.N, w.capacity_factor)
    kept = int(torch.clamp(fwd.expert_counts, max=C).sum())
    d, F = w.d_model, w.d_ff
    flops = (2.0 * kept * d * F * (6 if w.gate_multiply else 5) + 6.0 * w.T * w.N * w.d_model
             + (10.0 * w.T * d * F if w.has_shared else 0.0))
    achieved = flops / (ms / args.steps / 1e3) / 1e12
    if rank == 0:
        print(json.dumps({
            "metric": "top-1 MoE layer backward tokens/sec",
            "value": w.T * args.steps * world / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(w), pass_="backward"),
            "roofline": {"kernel": "bgemm_kernel (fp32 FFMA, every contraction of the backward)",
                         "bound": "alu", "achieved": achieved, "peak": FP32_FFMA_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / FP32_FFMA_TFLOPS,
                         "peak_kind": "derived: 148 SMs x 128 FP32 lanes x 2 flop x 2032 MHz",
                         "traffic": None, "algorithmic_flops_per_step": flops},
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": None, "clocks": clk}), flush=True)


# ------------------------------------------------------------------ GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--config", default="base", choices=sorted(CONFIGS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--expand", type=int, default=1,
                    help="Expanded Drop: candidates per token (1 = plain top-1)")
    ap.add_argument("--top-k", type=int, default=1, choices=[1, 2],
                    help="experts per token (2: top-2 token choice)")
    ap.add_argument("--renormalize", type=int, default=0, choices=[0, 1],
                    help="top-2 gates renormalised over the chosen pair")
    ap.add_argument("--expert-choice", type=int, default=0, choices=[0, 1],
                    help="expert-choice routing (each expert takes its C best tokens)")
    ap.add_argument("--backward", action="store_true",
                    help="time switch_moe_backward (gradients of <dy, y> + alpha L_aux) instead")
    ap.add_argument("--eager", action="store_true",
                    help="time eager calls only (no CUDA-graph replay)")
    ap.add_argument("--token-order", action="store_true",
                    help="token-order priority whatever the workload's (Expanded Drop "
                         "on the skewed shape)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import switch_top_expert_router_b300 as sm
    sm.load_library()
    torch.cuda.set_device(local)
    if args.backward:
        return run_backward(args, sm, rank, world, local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    w = CONFIGS[args.config]
    if args.token_order:
        w = w.replace(priority_mode=0)
    inp = make_inputs(w, seed=0, device=dev)
    p = sm.make_params(w.T, w.d_model, w.d_ff, w.N, w.capacity_factor, w.priority_mode,
                       w.gate_multiply, sm.BF16 if w.dtype == "bf16" else sm.F32, w.has_shared,
                       args.expand, args.top_k, args.renormalize, args.expert_choice)
    ws = sm.workspace(sm.switch_moe_workspace_bytes(p), dev)
    out = None
    stream = torch.cuda.current_stream(dev)

    def step():
        nonlocal out
        if args.expert_choice:
            out = sm.switch_moe_forward_expert_choice(inp.x, inp.W_g, inp.W1, inp.W2,
                                                      w.capacity_factor, w.gate_multiply,
                                                      b_g=inp.b_g, W1s=inp.W1s, W2s=inp.W2s,
                                                      ws=ws, out=out)
            return
        out = sm.switch_moe_forward(inp.x, inp.W_g, inp.W1, inp.W2, w.capacity_factor,
                                    w.priority_mode, w.gate_multiply, b_g=inp.b_g,
                                    W1s=inp.W1s, W2s=inp.W2s, ws=ws, out=out,
                                    expand=args.expand, top_k=args.top_k,
                                    renormalize=args.renormalize)

    for _ in range(args.warmup):
        step()
    rc = sm.switch_moe_sync_status()
    if rc != 0:
        raise RuntimeError(f"device status after warm-up: {sm.strerror(rc)}")

    # The whole forward captured once into a CUDA graph, as a serving loop
    # replays it (same kernels, same work every step); eager calls are timed
    # too, and are the fallback when capture is unavailable.
    graph, graph_note = None, None
    if not args.eager:
        try:
            cs = torch.cuda.Stream(dev)
            g = torch.cuda.CUDAGraph()
            torch.cuda.synchronize()
            with torch.cuda.stream(cs):
                with torch.cuda.graph(g, stream=cs):
                    step()
            torch.cuda.synchronize()
            for _ in range(args.warmup):
                g.replay()
            torch.cuda.synchronize()
            graph = g
        except Exception as exc:   # noqa: BLE001 -- reported in the JSON line
            graph_note = f"capture failed, eager timing: {exc!r}"[:200]

    # ---- timed region: exactly K steps
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def timed(fn):
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        return e0.elapsed_time(e1)

    ms = timed(graph.replay if graph else step)
    eager_ms = timed(step) if graph else ms
    clk = clocks.stop()
    rc = sm.switch_moe_sync_status()
    if rc != 0:
        raise RuntimeError(f"device status after timing: {sm.strerror(rc)}")
    ms = max_over_ranks(ms, pg, dev)
    eager_ms = max_over_ranks(eager_ms, pg, dev)
    value = job_tokens_per_s(w.T, args.steps, world, ms)

    # ---- per-phase times (same K steps, events at the phase boundaries)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(sm.NUM_PHASE_EVENTS)]
          for _ in range(args.steps)]
    for row in ev:
        for e in row:
            e.record(stream)       # materialise the CUDA event handles
    torch.cuda.synchronize()
    for row in ev:
        sm.switch_moe_set_phase_events(row)
        step()
    sm.switch_moe_set_phase_events(None)
    torch.cuda.synchronize()
    phase_ms = {name: statistics.mean(row[i].elapsed_time(row[i + 1]) for row in ev)
                for i, name in enumerate(sm.PHASES)}

    # ---- workload facts for the roofline
    C = sm.switch_moe_capacity(w.T, w.N, w.capacity_factor)
    # filled slots per expert (with Expanded Drop, re-routed tokens count
    # for the expert that runs them)
    if args.expert_choice:
        ch = out.chosen_token.cpu().numpy()
        kept = (ch >= 0).sum(axis=1).astype(np.int64)
        out_rows = int((out.experts_per_token.cpu().numpy() > 0).sum())   # y rows written
        n_choices = w.T   # "dropped" below: tokens no expert took
    else:
        eid, slt = out.expert_id.cpu().numpy(), out.slot.cpu().numpy()
        kept = np.bincount(eid[slt >= 0], minlength=w.N).astype(np.int64)
        out_rows = int((slt.reshape(w.T, -1) >= 0).any(axis=1).sum())   # y rows written
        n_choices = w.T * args.top_k
    active = int((kept > 0).sum())
    T_kept = int(kept.sum())   # filled slots (top-2: token-choice pairs)
    eb = 2 if w.dtype == "bf16" else 4
    d, F = w.d_model, w.d_ff
    wbytes_expert = d * F * eb
    g1_bytes = active * wbytes_expert + T_kept * d * eb + T_kept * F * eb
    g2_bytes = active * wbytes_expert + T_kept * F * eb + T_kept * d * 4
    gemm_ms = phase_ms["expert_gemm1"] + phase_ms["expert_gemm2"]
    tc_router = w.dtype == "bf16" and w.N <= 256
    fused = w.dtype == "bf16" and gemm2_ksplit(w, C) == 1
    ffn_one = fused and -(-C // 16) * 16 <= 128   # both routed GEMMs in one launch
    # algorithmic bytes of the dominant kernel per launch: the active experts'
    # weights, the dispatched tokens in and the expert outputs out -- and,
    # when GEMM 1 and GEMM 2 are separate launches, H out of one and into the
    # other (the mean of the two launches)
    ffn_bytes = (2 * active * wbytes_expert + T_kept * d * eb + out_rows * d * 4 if ffn_one
                 else (g1_bytes + g2_bytes) / 2)
    hbm, bf16_peak, peak_kind = peaks()
    achieved = ffn_bytes * (1 if ffn_one else 2) / (gemm_ms / 1e3) / 1e9
    layer_bytes = (w.T * d * eb + w.T * d * 4 + w.N * d * 4 + w.T * 13 * args.top_k + w.N * 4
                   + 2 * active * wbytes_expert + (2 * wbytes_expert if w.has_shared else 0))
    layer_flops = 4.0 * T_kept * d * F + (4.0 * w.T * d * F if w.has_shared else 0.0)
    t_roof = max(layer_flops / (bf16_peak * 1e12), layer_bytes / (hbm * 1e9))
    # kernels per forward: [split W_g +] router, scan, slots/dispatch [+ gate
    # ranking + dispatch], GEMM 1 [+ shared GEMMs], GEMM 2 [+ combine when the
    # second GEMM's epilogue cannot do it: fp32 layers, K-split GEMM 2]
    # [+ Expanded Drop passes and the moved rows' dispatch]
    # [+ the FFMA router kernel that adds the parts of a K-split
    # tensor-core router: few tokens (<= 8 tiles of 128), long d_model]
    tiles_r = -(-w.T // 128)
    router_split = (tc_router and w.N <= 128 and tiles_r <= 8
                    and -(-w.d_model // 64) >= 8 and tiles_r * 2 <= 148)
    launches = ((2 if tc_router else 1) + (1 if router_split else 0) + 2
                + (2 if w.priority_mode else 0)
                + (1 if ffn_one else 2) + (2 if w.has_shared else 0) + (0 if fused else 1)
                + (2 if args.expand > 1 else 0))

    # ---- end to end through the host-buffer entry point
    e2e = None
    if not args.no_e2e and not args.expert_choice:   # the host-buffer entry point is top-k only
        x_host = inp.x.cpu().pin_memory()
        hout = None
        hws = sm.workspace(sm.switch_moe_hostio_workspace_bytes(p), dev)

        def hstep():
            nonlocal hout
            hout = sm.switch_moe_forward_hostio(x_host, inp.W_g, inp.W1, inp.W2,
                                                w.capacity_factor, w.priority_mode,
                                                w.gate_multiply, b_g=inp.b_g, W1s=inp.W1s,
                                                W2s=inp.W2s, ws=hws, out=hout,
                                                expand=args.expand, top_k=args.top_k,
                                                renormalize=args.renormalize)
        for _ in range(args.warmup):
            hstep()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        h0.record(stream)
        for _ in range(args.steps):
            hstep()
        h1.record(stream)
        torch.cuda.synchronize()
        hms = max_over_ranks(h0.elapsed_time(h1), pg, dev)
        e2e = {"value": job_tokens_per_s(w.T, args.steps, world, hms), "unit": "tokens/s",
               "h2d_bytes_per_step": w.T * d * eb,
               "d2h_bytes_per_step": w.T * d * 4 + w.T * 13 * args.top_k + w.N * 4 + 4,
               "ms_per_step": hms / args.steps}
        if sm.switch_moe_sync_status() != 0:
            raise RuntimeError("device status after the host-IO run")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, sec = 0, 0.0
        while sec < 10.0:
            n, s = oracle_sample_step(w, expand=args.expand, top_k=args.top_k,
                                      renormalize=args.renormalize,
                                      expert_choice=args.expert_choice)
            tok += n
            sec += s
        cpu = {"value": tok / sec, "unit": "tokens/s", "cores": blas_threads(),
               "kind": "oracle", "sample": cpu_sample_desc(w)}

    if rank == 0:
        line = {
            "metric": "top-1 MoE layer tokens/sec", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": dict(workload_config(w, args.expand, args.top_k, args.renormalize,
                                           args.expert_choice),
                           launch=("CUDA-graph replay of the whole forward" if graph
                                   else "eager calls")),
            "timing": {"graph_replay": graph is not None, "eager_ms_per_step": eager_ms / args.steps,
                       "note": graph_note},
            "e2e": e2e,
            "roofline": {"kernel": ("ffn_tc_kernel (expert GEMM 1 + 2, one launch)" if ffn_one
                                    else "gemm_tc_kernel (expert GEMM 1 + 2)"),
                         "bound": "hbm",
                         "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm, "peak_kind": peak_kind,
                         # the ncu figure is for the plain top-1 workload only
                         "traffic": (kernel_traffic(args.config)
                                     if ffn_one and args.expand == 1 and args.top_k == 1
                                     and not args.expert_choice else None),
                         "algorithmic_bytes_per_launch": ffn_bytes},
            "layer_roofline": {"t_roof_us": t_roof * 1e6, "t_step_us": 1e3 * ms / args.steps,
                               "frac": t_roof / (ms / args.steps / 1e3),
                               "bytes": layer_bytes, "flops": layer_flops,
                               "peaks": {"hbm_gbs": hbm, "bf16_tflops": bf16_peak,
                                         "kind": peak_kind}},
            "phase_us": {k: 1e3 * v for k, v in phase_ms.items()},
            "routing": {"active_experts": active,
                        # top-2: token-choice pairs kept and dropped
                        "kept_tokens": T_kept,
                        "dropped": (int(w.T - out_rows) if args.expert_choice
                                    else int(n_choices - T_kept)),
                        "capacity": C,
                        "aux_loss": float(out.aux_loss.item())},
            "cpu_baseline": cpu,
            "gpu_launches": launches * args.steps,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
