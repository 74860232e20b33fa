#!/usr/bin/env python
"""Throughput of the LatentMoE layer forward (top-16 of 896 experts, SwiGLU
experts on MXFP4 weights) on GB300, one process per GPU.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload decode|decode1|decode16|tiny|prefill|skewed|block] [--no-cpu-baseline]

A step is one lmoe_forward call (route -> permute -> MXFP8 activations ->
gate/up GEMM + SwiGLU -> down GEMM -> combine) over one batch of seeded
synthetic tokens with the whole expert bank resident in HBM.  With N > 1
(torchrun) every rank runs its own replica of the layer on its own batch:
the layer has no exchange step on one node's replicas, so there is no
collective on the data path ("scaling": "weak").  Rank 0 prints one JSON line.

`--impl reference` times the CPU oracle (plain single-threaded C, fp64) on a
bounded sample of the same workload on the host cores; it is the only other
place besides the CPU-baseline leg where this script runs the oracle.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "LatentMoE layer tokens/s; % HBM BW (decode) / % block-scaled TC peak (prefill)"
UNIT = "tokens/s"
# MXFP4 bytes per weight element (4-bit code + one E8M0 byte per 32 elements)
MXFP4_B = 0.5 + 1.0 / 32


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-sample-tokens", type=int, default=16)
    # batches of up to this many pairs run the small-batch kernels (default: the library's)
    ap.add_argument("--small-batch-pairs", type=int, default=None)
    # the decode run also measures the prefill and batch-1 workloads on the
    # same resident bank (sub-records of its line); this skips them
    ap.add_argument("--no-side-workloads", action="store_true")
    # launcher check without a GPU: the ranks start, meet over gloo and
    # report; nothing is measured and no bench line is printed
    ap.add_argument("--launch-selftest", action="store_true", help=argparse.SUPPRESS)
    return ap.parse_args()


def spawn_ranks(n: int, argv) -> int:
    """Run this script as n local ranks (one per GPU) under
    torch.distributed.run when it was started as a single process with
    --gpus n > 1; returns the launcher's exit code.  Rank 0 prints the line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def launch_selftest(ws: int, rank: int) -> None:
    """Ranks meet over gloo, agree on the slowest rank's value with the same
    barrier / max-over-ranks code the bench uses, and rank 0 reports how many
    ranks took part."""
    import torch
    import torch.distributed as tdist
    tdist.init_process_group("gloo")
    try:
        barrier(ws)
        slowest = max_over_ranks(float(rank + 1), ws, torch.device("cpu"))
        seen = torch.tensor([1.0])
        tdist.all_reduce(seen)
        if rank == 0:
            print(json.dumps({"launch_selftest": True, "n_gpus": ws, "ranks_seen": int(seen.item()),
                              "slowest_rank_value": slowest}), flush=True)
    finally:
        tdist.destroy_process_group()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def gemm_source_hash() -> str:
    import hashlib
    csrc = os.path.join(ROOT, "top_routing_mxfp4_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("k_ffn_tc.cu", "tc_ptx.cuh", "lmoe_internal.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per step of the expert GEMMs (the fused kernel, or gate/up +
    down) from the committed ncu summary of this workload, or None when the
    GEMM source has changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"k_moe_gemm_{workload}.md")
    if not os.path.exists(path):
        return None
    meta = {}
    for line in open(path):
        if ":" in line and line.split(":")[0].strip() in ("gemm_source_sha256_16", "traffic_bytes_per_launch"):
            k, v = line.split(":", 1)
            meta[k.strip()] = v.strip()
    if meta.get("gemm_source_sha256_16") != gemm_source_hash():
        return None
    total = None
    for kv in meta.get("traffic_bytes_per_launch", "").split():
        key, _, val = kv.partition("=")
        if key in ("ffn", "gate_up", "down"):
            total = (total or 0) + int(val)
    return total


def barrier(ws: int) -> None:
    """All ranks meet (no-op for a single process)."""
    if ws > 1:
        import torch.distributed as tdist
        tdist.barrier()


def max_over_ranks(value: float, ws: int, device) -> float:
    """The largest of the ranks' values (the slowest rank's time): one
    all-reduce of a scalar on `device` (the GPU under NCCL, the CPU under gloo)."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as tdist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(tokens_per_rank: int, ws: int, ms_per_step: float) -> float:
    """Tokens per second of all ranks together: every rank processes its own
    batch (weak scaling, replicas), timed by the slowest rank."""
    return ws * tokens_per_rank / (ms_per_step / 1e3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid, self.proc, self.t0, self.t1 = uuid, None, None, None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [[c.strip() for c in l.split(",")] for l in out.strip().splitlines() if l.count(",") >= 8]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------

def setup_layer(wl, dev):
    import numpy as np
    import torch

    import lmoe_inputs as gen
    from top_routing_mxfp4_gb300 import lmoe
    bank = lmoe.ExpertBank(wl.E, wl.d, wl.I, dev)
    for e0 in range(0, wl.E, 32):
        e1 = min(wl.E, e0 + 32)
        for which in ("gate", "up", "down"):
            bank.load(which, e0, torch.from_numpy(gen.expert_f32(wl, which, e0, e1)).to(dev))
    bias = gen.router_bias(wl)
    layer = lmoe.Layer(torch.from_numpy(gen.router_f32(wl)).to(dev), bank, k=wl.k,
                       bias=None if bias is None else torch.from_numpy(bias).to(dev))
    x = gen.x_bf16(wl)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)
    torch.cuda.synchronize()
    return layer, x, xd, bank


def roofline_for(wl, touched: int, ms_per_step: float, stages: dict, peaks: dict, traffic=None) -> dict:
    """The roofline of the expert GEMMs (gate/up + down: one fused kernel for
    decode-sized token tiles, two kernels otherwise; their time from the
    stage events) and the layer's fraction for a workload: HBM-bound (the
    touched experts' weight bytes) below 16 pairs per expert, tensor-bound
    (FP8-rate block-scaled MMA) above."""
    per_expert_w = 3 * wl.I * wl.d * MXFP4_B
    P = wl.T * wl.k
    t_ffn = (stages["gate_up"] + stages["down"]) / 1e3
    kernel = "expert GEMMs (gate/up + down)"
    if P >= 16 * wl.E:
        # prefill-shaped: the expert GEMMs are compute-bound; the block-scaled
        # MMA (kind::mxf8f6f4) runs at the FP8 rate = 2 x the measured bf16 peak
        fp8_peak = 2.0 * peaks["bf16_tflops"]
        gu_flops = 2.0 * 2 * P * wl.d * wl.I            # gate + up GEMMs
        expert_flops = 2.0 * 3 * P * wl.d * wl.I        # gate + up + down
        proj_flops = 2.0 * 2 * wl.T * wl.d * wl.hidden  # block: the two bf16 projections
        ideal_s = expert_flops / (fp8_peak * 1e12) + proj_flops / (peaks["bf16_tflops"] * 1e12)
        t_gu = stages["gate_up"] / 1e3
        return {"bound": "tensor", "kernel": kernel, "achieved": expert_flops / t_ffn / 1e12,
                "peak": fp8_peak, "unit": "TFLOP/s", "frac": expert_flops / t_ffn / 1e12 / fp8_peak,
                "traffic": traffic, "traffic_unit": "DRAM bytes per step of the expert GEMMs (ncu)",
                "algorithmic_flops": expert_flops,
                "gate_up_frac": gu_flops / t_gu / 1e12 / fp8_peak,
                "peak_source": f"{peaks['source']} bf16 burst x 2 (nominal fp8 / bf16 ratio)",
                "layer_tflops": (expert_flops + proj_flops) / (ms_per_step / 1e3) / 1e12,
                "layer_frac": ideal_s / (ms_per_step / 1e3),
                "layer_frac_note": "expert FLOPs at the FP8-rate peak"
                                   + (" + projection FLOPs at the bf16 peak" if wl.hidden else "")
                                   + ", as ideal time / measured step"}
    weight_bytes = touched * per_expert_w  # weights the expert GEMMs must stream once
    achieved = weight_bytes / t_ffn / 1e9
    layer_weight_gbs = weight_bytes / (ms_per_step / 1e3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved,
            "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
            "traffic": traffic, "traffic_unit": "DRAM bytes per step of the expert GEMMs (ncu)",
            "algorithmic_bytes": weight_bytes, "peak_source": peaks["source"],
            "layer_weight_gbs": layer_weight_gbs, "layer_frac": layer_weight_gbs / peaks["hbm_gbs"]}


class L2Flush:
    """Overwrites L2 between timed steps: a buffer twice the L2 size is
    written, then a second one as large is read, so that L2 holds clean lines
    when the step starts (the dirty lines of the write are written back here,
    not during the timed step)."""

    def __init__(self, l2_bytes: int, dev):
        import torch
        self.w = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(2 * l2_bytes // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)
        self.bytes = self.w.numel() * 4

    def run(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.out)

    def describe(self) -> str:
        return f"{self.bytes / 1e6:.0f} MB written, then {self.bytes / 1e6:.0f} MB of another buffer read"


def scale_histogram_record(bank) -> dict:
    """The bank's E8M0 weight-scale histograms (lmoe_mxfp4_scale_histogram:
    256 bins per expert matrix, counted on the GPU), summed over the experts
    for each of gate, up and down, with each matrix's scale range."""
    rec = {}
    for w, h in bank.scale_histograms().items():
        h = h.cpu().long()                       # [E, 256]
        tot = h.sum(0)
        nz = [int(b) for b in (tot > 0).nonzero().flatten()]
        per_lo = [int((row > 0).nonzero().min()) for row in h]
        per_hi = [int((row > 0).nonzero().max()) for row in h]
        rec[w] = {"bins": {str(b): int(tot[b]) for b in nz},
                  "scale_exponent_range": [nz[0] - 127, nz[-1] - 127] if nz else None,
                  "per_matrix_exponent_span_max": max(hi - lo for lo, hi in zip(per_lo, per_hi)) if nz else 0}
    return rec


def time_steps(fwd, K: int, st, scrub=None) -> float:
    """Device time of K forward passes (ms): back to back, or, with `scrub`
    (an L2Flush), each step timed alone after the flush."""
    import torch
    if scrub is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(K):
            fwd()
        b.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in evs:
        scrub.run()
        a.record(st)
        fwd()
        b.record(st)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


def stage_times(lmoe, fwd, K: int, st, scrub=None) -> dict:
    """Mean stage times (ms) over K passes with CUDA events at lmoe_forward's
    stage boundaries (these serialise the launches)."""
    import torch
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(lmoe.NUM_STAGE_EVENTS)] for _ in range(K)]
    for row in evs:  # torch creates the CUDA event objects on first record
        for e in row:
            e.record(st)
    torch.cuda.synchronize()
    for i in range(K):
        if scrub is not None:
            scrub.run()
        lmoe.set_stage_events(evs[i])
        fwd()
    torch.cuda.synchronize()
    lmoe.set_stage_events(None)
    return {name: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / K for j, name in enumerate(lmoe.STAGES)}


def side_record(lmoe, name: str, bank, Wr_dev, dev, steps: int, warmup: int, peaks: dict, scrub) -> dict:
    """Another workload on the same resident expert bank, measured in the same
    run: its own batch and workspace, timed like the headline (each step
    alone after an L2 overwrite when its touched weights could stay in L2)."""
    import numpy as np
    import torch

    import lmoe_inputs as gen
    wl = gen.WORKLOADS[name]
    assert (wl.E, wl.d, wl.I) == (bank.E, bank.d, bank.I) and not wl.hidden
    bias = gen.router_bias(wl)
    layer = lmoe.Layer(Wr_dev, bank, k=wl.k, bias=None if bias is None else torch.from_numpy(bias).to(dev))
    x = torch.from_numpy(np.ascontiguousarray(gen.x_bf16(wl)).view(np.int16)).to(dev).view(torch.bfloat16)
    y = torch.empty((wl.T, wl.d), dtype=torch.bfloat16, device=dev)
    idx = torch.empty((wl.T, wl.k), dtype=torch.int32, device=dev)
    st = torch.cuda.current_stream()

    def fwd():
        layer.forward(x, y=y, topk_idx=idx)
    for _ in range(max(3, warmup)):
        fwd()
    torch.cuda.synchronize()
    assert layer.device_status() == 0
    touched = int((torch.bincount(idx.view(-1).long(), minlength=wl.E) > 0).sum())
    per_expert_w = 3 * wl.I * wl.d * MXFP4_B
    l2_bytes = scrub.bytes // 2
    flush = touched * per_expert_w < 2 * l2_bytes
    ms = time_steps(fwd, steps, st, scrub if flush else None) / steps
    stages = stage_times(lmoe, fwd, min(steps, 50), st, scrub if flush else None)
    small = lmoe.forward_workspace_views(wl.T, wl.d, wl.E, wl.k, wl.I).path == 1
    layer._ws = None
    roof = roofline_for(wl, touched, ms, stages, peaks, None if small else profiled_traffic(wl.name))
    if small:
        roof["kernel"] = "small-batch gate/up + down kernels (CUDA cores)"
    return {"workload": wl.name, "T": wl.T, "steps": steps, "ms_per_step": ms, "value": wl.T / (ms / 1e3),
            "unit": UNIT, "path": "small-batch kernels" if small else "tensor-core kernels",
            "l2": "flushed before every step" if flush else "inputs larger than L2", "touched_experts": touched,
            "roofline": roof, "stage_ms": stages}


def cpu_baseline(wl, ntok: int):
    """The oracle as it stands, on `ntok` tokens of the workload, one core."""
    import numpy as np

    import lmoe_inputs as gen
    import oracle
    ntok = min(ntok, wl.T)
    x = gen.x_bf16(wl, 0, ntok)
    Wr = gen.router_f32(wl)
    bias = gen.router_bias(wl)
    # weights of the experts these tokens route to, quantised by the oracle (not timed: load-time work)
    lg = oracle.router_logits(x, Wr, bias)
    idx, _ = oracle.topk_softmax(lg, wl.k)
    bank = oracle.quantize_experts(wl, experts=np.unique(idx))
    t0 = time.perf_counter()
    lg = oracle.router_logits(x, Wr, bias)
    idx, w = oracle.topk_softmax(lg, wl.k)
    oracle.permute(idx, wl.E)
    oracle.moe_tokens(x, idx, w, bank, wl.d, wl.E, wl.I)
    dt = time.perf_counter() - t0
    return {"value": ntok / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{ntok} of the {wl.T} tokens of the {wl.name} workload through the whole layer "
                      f"(routing over all {wl.E} experts, top-{wl.k}, permute, SwiGLU experts, combine); "
                      f"{dt:.1f} s of CPU time"}


def run_ours(args, ws, rank, local):
    import numpy as np
    import torch

    import lmoe_inputs as gen
    from top_routing_mxfp4_gb300 import build as lbuild
    lbuild.build()
    from top_routing_mxfp4_gb300 import lmoe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = gen.WORKLOADS[args.workload]
    if args.small_batch_pairs is not None:
        lmoe.set_small_batch_pairs(args.small_batch_pairs)
    small = lmoe.forward_workspace_views(wl.T, wl.d, wl.E, wl.k, wl.I).path == 1
    layer, x, xd, bank = setup_layer(wl, dev)
    T = wl.T
    st = torch.cuda.current_stream()
    idx = torch.empty((T, wl.k), dtype=torch.int32, device=dev)
    y = torch.empty((T, wl.d), dtype=torch.bfloat16, device=dev)
    if wl.hidden:
        # the block: bf16 hidden -> latent projection, the layer, latent -> hidden
        def dev_bf16(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
        blk = lmoe.Block(dev_bf16(gen.proj_in_bf16(wl)), layer, dev_bf16(gen.proj_out_bf16(wl)))
        x = gen.hidden_bf16(wl)
        xin = dev_bf16(x)
        out = torch.empty((T, wl.hidden), dtype=torch.bfloat16, device=dev)

        def fwd(xi):
            blk.forward(xi, out=out, topk_idx=idx)
    else:
        xin, out = xd, y

        def fwd(xi):
            layer.forward(xi, y=y, topk_idx=idx)
    for _ in range(max(3, args.warmup)):
        fwd(xin)
    torch.cuda.synchronize()
    if not wl.hidden:
        assert layer.device_status() == 0
    counts = torch.bincount(idx.view(-1).long(), minlength=wl.E)
    touched = int((counts > 0).sum())
    per_expert_w = 3 * wl.I * wl.d * MXFP4_B           # gate + up + down bytes of one expert
    # Batches whose touched weights could stay in L2 between steps (batch-1
    # decode: 16 experts = 47 MB) get L2 written over before every step, and
    # each step is timed alone with events after the flush.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 129 * 2 ** 20)
    flush = touched * per_expert_w < 2 * l2_bytes
    scrub = L2Flush(l2_bytes, dev) if flush else None

    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    time.sleep(0.3)
    K = args.steps
    # headline: K back-to-back forward passes, nothing else on the stream (the
    # kernels of consecutive stages overlap their launch through programmatic
    # dependent launch, which an event between them would serialise)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    if flush:
        step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b in step_ev:
            scrub.run()
            a.record(st)
            fwd(xin)
            b.record(st)
        torch.cuda.synchronize()
        barrier(ws)
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    else:
        t_start.record(st)
        for i in range(K):
            fwd(xin)
        t_end.record(st)
        torch.cuda.synchronize()
        barrier(ws)
        elapsed_ms = t_start.elapsed_time(t_end)
    # stage breakdown (and the gate/up GEMM time of the roofline): a second
    # live pass with CUDA events at the stage boundaries
    K2 = min(K, 50)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(lmoe.NUM_STAGE_EVENTS)] for _ in range(K2)]
    for row in evs:  # torch creates the CUDA event objects on first record
        for e in row:
            e.record(st)
    torch.cuda.synchronize()
    for i in range(K2):
        if flush:
            scrub.run()
        lmoe.set_stage_events(evs[i])
        fwd(xin)
    torch.cuda.synchronize()
    lmoe.set_stage_events(None)
    clocks = sampler.stop()
    stage_ms = {name: sum(e[j].elapsed_time(e[j + 1]) for e in evs) / K2 for j, name in enumerate(lmoe.STAGES)}
    elapsed_ms = max_over_ranks(elapsed_ms, ws, dev)
    ms_per_step = elapsed_ms / K
    value = whole_job_rate(T, ws, ms_per_step)

    # end to end through host buffers: H2D of the input from pinned memory, forward, D2H of the output
    xh = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).pin_memory()
    yh = torch.empty(tuple(out.shape), dtype=torch.bfloat16).pin_memory()
    xdev = torch.empty_like(xin)
    for _ in range(3):
        xdev.copy_(xh, non_blocking=True)
        fwd(xdev)
        yh.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    barrier(ws)
    if flush:
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for a, b in e2e_ev:
            scrub.run()
            a.record(st)
            xdev.copy_(xh, non_blocking=True)
            fwd(xdev)
            yh.copy_(out, non_blocking=True)
            b.record(st)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), ws, dev)
    else:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(K):
            xdev.copy_(xh, non_blocking=True)
            fwd(xdev)
            yh.copy_(out, non_blocking=True)
        e1.record(st)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    barrier(ws)

    peaks = load_peaks()
    launches_per_step = lmoe.forward_kernel_count(T, wl.d, wl.E, wl.k, wl.I) + (2 if wl.hidden else 0)
    roofline = roofline_for(wl, touched, ms_per_step, stage_ms, peaks, None if small else profiled_traffic(wl.name))
    if small:
        roofline["kernel"] = "small-batch gate/up + down kernels (CUDA cores)"
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "mxfp4 x mxfp8 -> f32 acc", "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": wl.name, "T": T, "d": wl.d, "E": wl.E, "k": wl.k, "I": wl.I, "hidden": wl.hidden,
                   "per_gpu_batch_tokens": T, "parallelism": f"replicas x{ws}",
                   "path": "small-batch kernels" if small else "tensor-core kernels",
                   "l2": (f"L2 flushed before every step ({scrub.describe()}, not timed); "
                          if flush else "inputs larger than L2: ")
                         + f"{touched} touched experts = {touched * per_expert_w / 1e9:.2f} GB of weights read "
                           f"per step (L2 {l2_bytes / 2 ** 20:.0f} MB)"},
        "roofline": roofline,
        "stage_ms": stage_ms,
        "stage_ms_note": f"second live pass of {K2} steps with CUDA events at the layer's stage boundaries (the "
                         "events serialise the launches, so the stages add up to more than the layer's share of "
                         "ms_per_step)" + ("; the block's two projections are not in these stages" if wl.hidden else ""),
        "touched_experts": touched,
        "e2e": {"value": whole_job_rate(T, ws, e2e_ms / K), "unit": UNIT, "h2d_bytes_per_step": xh.numel() * 2,
                "d2h_bytes_per_step": yh.numel() * 2},
        "gpu_launches": K * launches_per_step, "clocks": clocks,
        "weight_scale_histogram": scale_histogram_record(bank),
    }
    if ws == 1 and wl.name == "decode" and not args.no_side_workloads:
        # The same run, on the same resident expert bank: the headline re-timed
        # with L2 written over before every step, then the prefill (T = 8192)
        # and batch-1 (T = 1) workloads as sub-records with their own rooflines.
        scrub_all = scrub if scrub is not None else L2Flush(l2_bytes, dev)
        side_sampler = ClockSampler(uuid)
        side_sampler.start()
        time.sleep(0.3)
        K3 = min(K, 100)
        ms_fl = time_steps(lambda: fwd(xin), K3, st, scrub_all) / K3
        line["l2_flushed"] = {"ms_per_step": ms_fl, "value": whole_job_rate(T, ws, ms_fl), "unit": UNIT, "steps": K3,
                              "note": f"each step timed alone after an L2 flush ({scrub_all.describe()}), "
                                      "not timed"}
        line["side_workloads"] = [side_record(lmoe, "prefill", bank, layer.Wr, dev, 10, 3, peaks, scrub_all),
                                  side_record(lmoe, "decode1", bank, layer.Wr, dev, 100, 5, peaks, scrub_all)]
        line["side_workloads_clocks"] = side_sampler.stop()
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_sample_tokens)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------
# reference arm: the CPU oracle as it stands
# ---------------------------------------------------------------------------------

def run_reference(args, ws, rank):
    """The oracle as it stands on the host cores (one thread), rank 0 only.
    A step is one token of the workload through the whole layer (routing
    over all experts, top-k, permute, SwiGLU experts, combine); the tokens
    cycle over the batch's first REF_TOKENS, whose experts are quantised once
    before timing (load-time work).  Steps stop early once REF_BUDGET_S of
    timed CPU work is spent; the line reports the steps actually timed."""
    if rank != 0:
        return
    import lmoe_inputs as gen
    import oracle
    gen.build()
    oracle.build()
    wl = gen.WORKLOADS[args.workload]
    REF_TOKENS, REF_BUDGET_S = 8, 150.0
    ntok = min(REF_TOKENS, wl.T)
    x = gen.x_bf16(wl, 0, ntok)
    Wr = gen.router_f32(wl)
    bias = gen.router_bias(wl)
    lg = oracle.router_logits(x, Wr, bias)
    idx, _ = oracle.topk_softmax(lg, wl.k)
    bank = oracle.quantize_experts(wl, experts=np.unique(idx))

    def step(i):
        xt = x[i % ntok:i % ntok + 1]
        l = oracle.router_logits(xt, Wr, bias)
        ix, w = oracle.topk_softmax(l, wl.k)
        oracle.permute(ix, wl.E)
        oracle.moe_tokens(xt, ix, w, bank, wl.d, wl.E, wl.I)

    warm = min(args.warmup, 3)
    for i in range(warm):
        step(i)
    times = []
    for i in range(args.steps):
        t0 = time.perf_counter()
        step(i)
        times.append(time.perf_counter() - t0)
        if sum(times) > REF_BUDGET_S:
            break
    dt = sum(times) / len(times)
    value = 1.0 / dt
    sample = (f"{len(times)} steps of one token each (tokens 0..{ntok - 1} of the {wl.T}-token {wl.name} workload, "
              f"cycled) through the whole layer: routing over all {wl.E} experts, top-{wl.k}, permute, SwiGLU "
              f"experts, combine; {sum(times):.1f} s of CPU time")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": len(times),
            "steps_requested": args.steps, "warmup": warm, "warmup_requested": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic (seeded counter-based generator)",
            "config": {"workload": wl.name, "T": wl.T, "d": wl.d, "E": wl.E, "k": wl.k, "I": wl.I},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_env()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    if args.launch_selftest:
        launch_selftest(ws, rank)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    if ws > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    try:
        run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            import torch.distributed as tdist
            tdist.destroy_process_group()


if __name__ == "__main__":
    main()
