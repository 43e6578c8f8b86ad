#!/usr/bin/env python3
"""Throughput of one Hy3-style MoE FFN layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one whole layer forward (router GEMM + top-k, permutation, grouped
gate/up GEMM + SiLU, grouped down GEMM with the shared expert, combine) through
the C ABI on one batch of seeded synthetic input of the pages' shapes, with
weights resident in HBM.  The headline workload is the Hy3 decode batch
(T = 8 tokens, H = 4096, 192 routed experts top-8 + 1 shared, I = 1536); the
Hy3 prefill chunk (T = 4096) is measured too and reported in "prefill".

L2 is flushed between timed steps: a 256 MiB write, then a 256 MiB read of
another buffer, so that the write-back of the flush's dirty lines is over
before the step starts (left to the step it cost ~20 us of HBM time at
decode); each step is timed with CUDA events on the launching stream.  Under torchrun each rank runs its own
replica on its own tokens (weak scaling, no collective on the data path) and
the slowest rank's time is used.

--impl reference times the fp64 oracle (oracle/) on the host cores on the same
workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "MoE-layer tokens/s at Hy3 shape (T=8, T=4096); % of HBM or BF16 tensor roofline"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers

def log(*a):
    print(*a, file=sys.stderr, flush=True)


def peaks():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {  # the files that define each kernel's code
    "expert_ffn": ["expert_gemm.cu", "ptx.cuh"],
    "gate_up": ["expert_gemm.cu", "ptx.cuh"], "down": ["expert_gemm.cu", "ptx.cuh"],
    "route": ["router.cu", "ptx.cuh"], "permute": ["permute.cu", "ptx.cuh"], "combine": ["combine.cu", "ptx.cuh"],
}


def source_hash(kernel: str) -> str:
    """Hash of a kernel's sources: stored ncu counters are used only for the same code."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        f = ROOT / "expert_ffn_layer_gb300" / "csrc" / name
        h.update(name.encode())
        h.update(f.read_bytes())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """dram bytes per launch from a committed ncu summary, if it matches these sources."""
    p = ROOT / "profiles" / f"dram_traffic_{workload}.json"
    if not p.exists():
        return None
    d = json.loads(p.read_text())
    k = d.get("kernels", {}).get(kernel)
    if k is None or k.get("source_hash") != source_hash(kernel):
        return None
    return float(k["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait(timeout=5)

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = [r.split(", ") for r in Path(self.file.name).read_text().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------------------------------- multi-rank helpers

def replica_hidden(w, rank: int):
    """Tokens of one replica: rank 0 uses the workload's own hidden states (so a
    one-GPU run is the workload itself); rank r > 0 draws its own seeded batch."""
    import workloads as W

    if rank == 0:
        return W.router_inputs(w)[0]
    return W.normal_bf16(w.seed + 1000 * rank, W.TID_HIDDEN, (w.T, w.H), w.hidden_sigma)


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The slowest rank's time (all ranks get the same value)."""
    if world == 1:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def layer_launches(T: int, top_k: int) -> int:
    """Kernels one layer forward launches: router split, router GEMM, top-k, the
    permutation (one kernel up to 8192 routed slots, else count + scatter), the
    expert FFN, combine."""
    return 6 + (1 if T * top_k > 8192 else 0)


def job_throughput(world: int, tokens_per_step: int, steps: int, total_ms: float) -> float:
    """Whole-job tokens/s: every rank processes its own batch each step (weak scaling)."""
    return world * tokens_per_step * steps / (total_ms * 1e-3)


# ----------------------------------------------------------------------------- algorithmic work

def stage_work(w, n_active: int):
    """Algorithmic bytes and FLOPs of each kernel of one layer forward."""
    T, H, E, k, I = w.T, w.H, w.E, w.top_k, w.I
    S = T * k
    Is = w.I_shared if w.has_shared else 0
    Ts = T if w.has_shared else 0
    ns = 1 if w.has_shared else 0
    return {
        # route = split (E*H fp32 -> 2 x bf16) + router GEMM (x, W_high, W_low) + top-k
        "route": {"bytes": E * H * 4 + 2 * E * H * 2 + T * H * 2 + S * 8 + E * 4, "flops": 2 * 2 * T * H * E},
        "permute": {"bytes": S * 4 * 3 + (2 * E + 1) * 4, "flops": 0},
        "gate_up": {"bytes": (n_active * 2 * I + ns * 2 * Is) * H * 2 + (S + Ts) * H * 2 + (S * I + Ts * Is) * 2,
                    "flops": 4 * (S * H * I + Ts * H * Is)},
        "down": {"bytes": (n_active * I + ns * Is) * H * 2 + (S * I + Ts * Is) * 2 + (S + Ts) * H * 2,
                 "flops": 2 * (S * H * I + Ts * H * Is)},
        "combine": {"bytes": S * H * 2 + Ts * H * 2 + T * H * 2 + S * 8, "flops": 2 * S * H},
        # the fused persistent kernel (gate/up then down, one launch): every activated
        # expert's three weight matrices, token rows in, expert outputs out, and the
        # bf16 activations written and read back
        "expert_ffn": {"bytes": (n_active * 3 * I + ns * 3 * Is) * H * 2 + (S + Ts) * H * 2 + (S + Ts) * H * 2
                                + 2 * (S * I + Ts * Is) * 2,
                       "flops": 6 * (S * H * I + Ts * H * Is)},
    }


def roofline_for(stage: str, work: dict, ms: float, pk: dict, pk_kind: str, workload: str, bound: str | None = None):
    b, f = work[stage]["bytes"], work[stage]["flops"]
    t_mem = b / (pk["hbm_gbs"] * 1e9)
    t_tc = f / (pk["bf16_tflops"] * 1e12) if f else 0.0
    if bound is None:
        bound = "tensor" if t_tc > t_mem else "hbm"
    sec = ms * 1e-3
    if bound == "hbm":
        ach, peak, unit = b / sec / 1e9, pk["hbm_gbs"], "GB/s"
    else:
        ach, peak, unit = f / sec / 1e12, pk["bf16_tflops"], "TFLOP/s"
    return {"kernel": stage, "bound": bound, "achieved": round(ach, 1), "peak": peak, "unit": unit,
            "frac": round(ach / peak, 4), "peak_source": f"{pk_kind} (MEASURED_PEAKS.json)" if pk_kind == "measured"
            else "fallback", "traffic": stored_traffic(stage, workload), "algorithmic_bytes": b,
            "algorithmic_flops": f, "ms": round(ms, 4)}


# ----------------------------------------------------------------------------- our implementation

def run_ours(args, rank, world, local_rank):
    import torch

    import expert_ffn_layer_gb300 as moe
    import workloads as W
    import __graft_entry__

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    moe.load()
    pk, pk_kind = peaks()

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def f32(a):
        return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).to(dev)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def flush_l2(i):
        """Evict L2: write a buffer larger than L2, then read another one, so that
        L2 holds clean unrelated lines (no write-back left for the timed step)."""
        flush.fill_(i & 0xFF)
        flush_rd.sum()

    def setup(name, replica_seed):
        w = W.WORKLOADS[name]
        t0 = time.time()
        _, router_w, bias = W.router_inputs(w)
        hidden_np = replica_hidden(w, replica_seed)  # each rank has its own tokens, same weights
        gate, up, down = W.expert_weights(w)
        sg, su, sd = W.shared_weights(w)
        d = moe.dims(w.T, w.H, w.E, w.I, w.top_k, w.I_shared, w.score_mode, w.route_scale, w.renorm_eps,
                     w.has_shared)
        layer = moe.MoELayer(d, f32(router_w), f32(bias), bf(gate), bf(up), bf(down), bf(sg), bf(su), bf(sd))
        del gate, up, down
        hidden = bf(hidden_np)
        log(f"[rank {rank}] {name}: inputs ready in {time.time() - t0:.1f}s")
        return w, d, layer, hidden, hidden_np, (router_w, bias, sg, su, sd)

    def timed(fn, K, W_):
        for _ in range(W_):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        for i in range(K):
            flush_l2(i)
            ev[i][0].record()
            fn()
            ev[i][1].record()
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def graph_of(fn, reps):
        """A CUDA graph of `reps` back-to-back calls (no host gaps between kernels)."""
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()  # one eager call on the capture stream first
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            for _ in range(reps):
                fn()
        return g

    samples = {}  # workload -> the GPU's routing and sampled output rows, compared with the oracle at the end

    def take_sample(name, w, d, layer, hidden):
        """One untimed layer forward plus the router's logits: the GPU side of the
        parity report (sampled output rows, every row's selection, all logits)."""
        idx = torch.empty((w.T, w.top_k), dtype=torch.int32, device=dev)
        wts = torch.empty((w.T, w.top_k), dtype=torch.float32, device=dev)
        logits = torch.empty((w.T, w.E), dtype=torch.float32, device=dev)
        moe.moe_route(d, hidden, layer.router_w, layer.expert_bias, idx, wts, layer.ws, logits_out=logits)
        out = layer(hidden)
        torch.cuda.synchronize()
        rows = parity_rows(w.T)
        samples[name] = {"w": w, "rows": rows, "out_rows": out[torch.from_numpy(rows).to(dev)].float().cpu().numpy(),
                         "idx": idx.cpu().numpy(), "logits": logits.cpu().numpy(),
                         "device_error": moe.moe_ws_read_error(layer.ws)}

    def stage_times(w, d, layer, hidden, K):
        """Each kernel of the layer on its own: a graph of K back-to-back launches of
        that kernel, timed with events around the replay; ms per launch."""
        S = w.T * w.top_k
        idx = torch.empty((w.T, w.top_k), dtype=torch.int32, device=dev)
        wts = torch.empty((w.T, w.top_k), dtype=torch.float32, device=dev)
        counts = torch.empty(w.E, dtype=torch.int32, device=dev)
        offs = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
        perm = torch.empty(S, dtype=torch.int32, device=dev)
        inv = torch.empty(S, dtype=torch.int32, device=dev)
        y = torch.empty((S, w.H), dtype=torch.bfloat16, device=dev)
        z = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
        out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
        ws = layer.ws
        L = layer
        calls = {
            "route": lambda: moe.moe_route(d, hidden, L.router_w, L.expert_bias, idx, wts, ws),
            "permute": lambda: moe.moe_permute(d, idx, counts, offs, perm, inv, ws),
            "expert_ffn": lambda: moe.moe_expert_ffn(d, hidden, perm, offs, L.w_gate, L.w_up, L.w_down, L.ws_gate,
                                                     L.ws_up, L.ws_down, y, z, ws),
            "combine": lambda: moe.moe_combine(d, y, z, inv, wts, out),
            # the two phases of expert_ffn as separate launches, for reference
            "gate_up": lambda: moe.moe_expert_gate_up(d, hidden, perm, offs, L.w_gate, L.w_up, L.ws_gate, L.ws_up, ws),
            "down": lambda: moe.moe_expert_down(d, offs, L.w_down, L.ws_down, y, z, ws),
        }
        for name in calls:  # produce every intermediate once, in order
            calls[name]()
        torch.cuda.synchronize()
        times = {}
        for name, fn in calls.items():
            g = graph_of(fn, K)
            g.replay()
            flush_l2(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            times[name] = e0.elapsed_time(e1) / K
            del g
        n_active = int((counts > 0).sum().item())
        return times, n_active, counts.cpu().numpy()

    # ---------------- headline workload (decode, T = 8)
    name = args.workload
    w, d, layer, hidden, hidden_np, host = setup(name, rank)
    out = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
    if args.profile:
        if args.fp8 or args.w8a8:  # the layer with FP8 expert weights (quantised once, before the layers)
            q = moe.quantize_fp8_experts(layer.w_gate, layer.w_up, layer.w_down, layer.ws_gate, layer.ws_up,
                                         layer.ws_down)
            fwd = moe.moe_layer_forward_w8a8 if args.w8a8 else moe.moe_layer_forward_fp8
            for _ in range(args.warmup + 1):
                fwd(d, hidden, layer.router_w, layer.expert_bias, q, out, layer.ws)
        elif args.phases:
            # warm-up layers, then the expert FFN's two phases as separate launches
            # (gate/up, then down) so that counters can be taken per phase
            for _ in range(args.warmup):
                layer(hidden, out)
            S = w.T * w.top_k
            idx = torch.empty((w.T, w.top_k), dtype=torch.int32, device=dev)
            wts = torch.empty((w.T, w.top_k), dtype=torch.float32, device=dev)
            offs = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
            perm = torch.empty(S, dtype=torch.int32, device=dev)
            moe.moe_route(d, hidden, layer.router_w, layer.expert_bias, idx, wts, layer.ws)
            moe.moe_permute(d, idx, torch.empty(w.E, dtype=torch.int32, device=dev), offs, perm,
                            torch.empty(S, dtype=torch.int32, device=dev), layer.ws)
            y = torch.empty((S, w.H), dtype=torch.bfloat16, device=dev)
            z = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
            moe.moe_expert_gate_up(d, hidden, perm, offs, layer.w_gate, layer.w_up, layer.ws_gate, layer.ws_up,
                                   layer.ws)
            moe.moe_expert_down(d, offs, layer.w_down, layer.ws_down, y, z, layer.ws)
        else:
            for _ in range(args.warmup + 1):
                layer(hidden, out)
        torch.cuda.synchronize()
        return {"profile": name, "fp8": bool(args.fp8), "w8a8": bool(args.w8a8), "phases": bool(args.phases),
                "device_error": moe.moe_ws_read_error(layer.ws)}

    def eager_step():
        layer(hidden, out)

    # one layer forward captured as a CUDA graph (the library enqueues no host
    # synchronisation and allocates nothing, so the whole chain captures)
    layer_graph = graph_of(eager_step, 1)

    def step():
        layer_graph.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        per_step = timed(step, args.steps, 0)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = max_over_ranks(float(np.sum(per_step)), world, dev)
    err = moe.moe_ws_read_error(layer.ws)
    if err:
        raise RuntimeError(f"device error word {err:#x} after the timed steps")
    value = job_throughput(world, w.T, args.steps, total_ms)
    eager_ms = max_over_ranks(float(np.sum(timed(eager_step, args.steps, 1))), world, dev)

    if rank == 0 and world == 1:
        take_sample(name, w, d, layer, hidden)

    # ---------------- end to end through MoELayer with host buffers
    h_in = torch.from_numpy(np.ascontiguousarray(hidden_np).view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = torch.empty((w.T, w.H), dtype=torch.bfloat16).pin_memory()

    def e2e_step():
        hidden.copy_(h_in, non_blocking=True)
        layer(hidden, out)
        h_out.copy_(out, non_blocking=True)

    e2e_ms = max_over_ranks(float(np.sum(timed(e2e_step, args.steps, max(1, args.warmup)))), world, dev)
    e2e_value = job_throughput(world, w.T, args.steps, e2e_ms)

    # ---------------- per-kernel durations -> roofline of the dominant kernel
    st_ms, n_active, counts = stage_times(w, d, layer, hidden, args.steps)
    work = stage_work(w, n_active)
    in_layer = ("route", "permute", "expert_ffn", "combine")
    dominant = max(in_layer, key=st_ms.get)
    roof = roofline_for(dominant, work, st_ms[dominant], pk, pk_kind, f"{name}_T{w.T}", bound="hbm")
    kernels = {n: {"ms": round(v, 4), **{kk: vv for kk, vv in roofline_for(n, work, v, pk, pk_kind,
                                                                            f"{name}_T{w.T}").items()
                                          if kk in ("bound", "achieved", "unit", "frac")}}
               for n, v in st_ms.items()}

    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded N(0,1) hidden, N(0,0.02) bf16 expert weights, N(0,0.02) fp32 router, "
                "N(0,0.1) expert bias (the pages' shapes; no trained weights)",
        "config": {**w.describe(), "workload": f"hy3_{name}_T{w.T}", "l2": "flushed between steps (256 MiB write, then 256 MiB read of another buffer)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": f"CUDA graph of one layer forward ({layer_launches(w.T, w.top_k)} kernels, PDL-chained)",
                   "eager_ms_per_step": round(eager_ms / args.steps, 5),
                   "active_experts": n_active, "max_tokens_per_expert": int(counts.max())},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": w.T * w.H * 2,
                "d2h_bytes_per_step": w.T * w.H * 2, "ms_per_step": round(e2e_ms / args.steps, 5)},
        "gpu_launches": layer_launches(w.T, w.top_k) * args.steps,
        "roofline": roof,
        "kernels": kernels,
        "clocks": clk.summary(),
    }
    # ---------------- the same decode layer with FP8 (E4M3, one scale per row)
    # expert weights: quantised once on the device, then moe_layer_forward_fp8
    # as a graph; not the headline (the metric names bf16 weights)
    if world == 1 and not args.no_fp8:
        try:
            fp8 = moe.quantize_fp8_experts(layer.w_gate, layer.w_up, layer.w_down, layer.ws_gate, layer.ws_up,
                                           layer.ws_down)
            fout = torch.empty_like(out)

            def fp8_step():
                moe.moe_layer_forward_fp8(d, hidden, layer.router_w, layer.expert_bias, fp8, fout, layer.ws)

            fgraph = graph_of(fp8_step, 1)
            fms = float(np.sum(timed(fgraph.replay, args.steps, args.warmup))) / args.steps
            ferr = moe.moe_ws_read_error(layer.ws)
            S = w.T * w.top_k
            perm_s = torch.empty(S, dtype=torch.int32, device=dev)
            offs_s = torch.empty(w.E + 1, dtype=torch.int32, device=dev)
            idx_s = torch.empty((w.T, w.top_k), dtype=torch.int32, device=dev)
            wts_s = torch.empty((w.T, w.top_k), dtype=torch.float32, device=dev)
            moe.moe_route(d, hidden, layer.router_w, layer.expert_bias, idx_s, wts_s, layer.ws)
            moe.moe_permute(d, idx_s, torch.empty(w.E, dtype=torch.int32, device=dev), offs_s, perm_s,
                            torch.empty(S, dtype=torch.int32, device=dev), layer.ws)
            y_s = torch.empty((S, w.H), dtype=torch.bfloat16, device=dev)
            z_s = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev)
            eg = graph_of(lambda: moe.moe_expert_ffn_fp8(d, hidden, perm_s, offs_s, fp8, y_s, z_s, layer.ws),
                          args.steps)
            eg.replay()
            flush_l2(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            eg.replay()
            e1.record()
            torch.cuda.synchronize()
            ems = e0.elapsed_time(e1) / args.steps
            wbytes = (n_active * 3 * w.I + 3 * w.I_shared) * w.H          # one byte per code
            sbytes = (n_active * (2 * w.I + w.H) + 2 * w.I_shared + w.H) * 4
            result["fp8_decode"] = {
                "weights": "E4M3 codes, one fp32 scale per output row (moe_quantize_fp8_rows)",
                "value": round(w.T / (fms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(fms, 5),
                "expert_ffn_ms": round(ems, 4),
                "expert_ffn_code_bytes": wbytes + sbytes,
                "expert_ffn_gbs": round((wbytes + sbytes) / (ems * 1e-3) / 1e9, 1),
                "device_error": ferr,
            }
            # W8A8: the same codes, FP8 activations, 8-bit MMAs (moe_layer_forward_w8a8)
            wout = torch.empty_like(out)

            def w8a8_step():
                moe.moe_layer_forward_w8a8(d, hidden, layer.router_w, layer.expert_bias, fp8, wout, layer.ws)

            wgraph = graph_of(w8a8_step, 1)
            wms = float(np.sum(timed(wgraph.replay, args.steps, args.warmup))) / args.steps
            werr = moe.moe_ws_read_error(layer.ws)
            weg = graph_of(lambda: moe.moe_expert_ffn_w8a8(d, hidden, perm_s, offs_s, fp8, y_s, z_s, layer.ws),
                           args.steps)
            weg.replay()
            flush_l2(1)
            e0.record()
            weg.replay()
            e1.record()
            torch.cuda.synchronize()
            wems = e0.elapsed_time(e1) / args.steps  # the hidden-state quantiser plus the expert kernel
            result["w8a8_decode"] = {
                "weights": "E4M3 codes, one fp32 scale per output row; activations E4M3 with one scale per row "
                           "(hidden per token, SiLU*up per routed slot); kind::f8f6f4 MMAs",
                "value": round(w.T / (wms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(wms, 5),
                "expert_ffn_ms": round(wems, 4),
                "expert_ffn_code_bytes": wbytes + sbytes,
                "expert_ffn_gbs": round((wbytes + sbytes) / (wems * 1e-3) / 1e9, 1),
                "expert_ffn_hbm_frac": round((wbytes + sbytes) / (wems * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
                "launch": "CUDA graph of one layer forward (7 kernels: hidden quantiser first, PDL-chained)",
                "device_error": werr,
            }
            del fp8, fgraph, eg, wgraph, weg
        except Exception as e:  # an auxiliary measurement: record the failure, keep the headline
            result["fp8_decode"] = {"error": f"{type(e).__name__}: {e}"}
    del layer, hidden, layer_graph
    torch.cuda.empty_cache()

    # ---------------- the larger configurations, single GPU: the Hy3 prefill
    # chunk (T = 4096), the skewed long prefill (T = 16384) and the
    # HunyuanImage-style softmax layer (T = 8192)
    def big_layer(name):
        bw, bd, blayer, bhidden, _, _ = setup(name, 0)
        bout = torch.empty((bw.T, bw.H), dtype=torch.bfloat16, device=dev)
        bgraph = graph_of(lambda: blayer(bhidden, bout), 1)
        bst = timed(bgraph.replay, args.steps, args.warmup)
        bms = float(np.mean(bst))
        # clocks under this workload's load: one second of back-to-back layers
        with ClockSampler(local_rank) as bclk:
            for _ in range(max(1, int(1.0 / (bms * 1e-3)))):
                bgraph.replay()
            torch.cuda.synchronize()
        take_sample(name, bw, bd, blayer, bhidden)
        bst_ms, bact, bcounts = stage_times(bw, bd, blayer, bhidden, max(3, args.steps // 2))
        bwork = stage_work(bw, bact)
        flops = bwork["expert_ffn"]["flops"]
        wbytes = (bact * 3 * bw.I + 3 * bw.I_shared) * bw.H * 2
        bdom = max(("route", "permute", "expert_ffn", "combine"), key=bst_ms.get)
        res = {
            "workload": f"{'hy3_' if name != 'image' else 'hunyuanimage_'}{name}_T{bw.T}",
            "value": round(bw.T / (bms * 1e-3), 1), "unit": UNIT,
            "ms_per_step": round(bms, 5), "active_experts": bact, "max_tokens_per_expert": int(bcounts.max()),
            "layer_tensor_frac": round(flops / (bms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
            # the same against the sustained (power-capped, seconds-long) bf16 figure
            "layer_tensor_frac_sustained": (round(flops / (bms * 1e-3) / 1e12 / pk["bf16_tflops_sustained"], 4)
                                            if pk.get("bf16_tflops_sustained") else None),
            "layer_hbm_frac": round(wbytes / (bms * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
            "roofline": roofline_for(bdom, bwork, bst_ms[bdom], pk, pk_kind, f"{name}_T{bw.T}"),
            "kernels": {n: round(v, 4) for n, v in bst_ms.items()},
            "gpu_launches": layer_launches(bw.T, bw.top_k) * args.steps,
            "clocks_under_load": bclk.summary(),
        }
        if name == "prefill":
            # the same layer with W8A8 experts (E4M3 weights, quantised once, and
            # E4M3 activations; moe_layer_forward_w8a8), not the headline dtype
            q8 = moe.quantize_fp8_experts(blayer.w_gate, blayer.w_up, blayer.w_down, blayer.ws_gate, blayer.ws_up,
                                          blayer.ws_down)
            wout = torch.empty_like(bout)
            wg = graph_of(lambda: moe.moe_layer_forward_w8a8(bd, bhidden, blayer.router_w, blayer.expert_bias, q8,
                                                             wout, blayer.ws), 1)
            wms = float(np.mean(timed(wg.replay, args.steps, args.warmup)))
            res["w8a8"] = {"value": round(bw.T / (wms * 1e-3), 1), "unit": UNIT, "ms_per_step": round(wms, 5),
                           "device_error": moe.moe_ws_read_error(blayer.ws)}
            del q8, wg
        del blayer, bhidden, bgraph
        torch.cuda.empty_cache()
        return res

    if world == 1 and not args.no_prefill:
        result["prefill"] = big_layer("prefill")
    if world == 1 and not args.no_extra:
        result["prefill_u"] = big_layer("prefill_u")
        result["zipf"] = big_layer("zipf")
        result["image"] = big_layer("image")

    # ---------------- the oracle on the host cores (rank 0 only, N = 1): timed on
    # the headline batch, on one core for the tiny and decode batches, and run on
    # each workload's sampled rows to report parity beside that workload's numbers
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, hidden_np, budget_s=args.cpu_seconds)
        result["cpu_baseline"]["one_core"] = {n: oracle_one_core(n) for n in ("tiny", "decode")}
        for key, smp in samples.items():
            par = parity_vs_oracle(smp)
            if key == name:
                result["parity"] = par
            elif key in result:
                result[key]["parity"] = par
    return result


# ----------------------------------------------------------------------------- the oracle as a baseline

def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


_ORACLE_INPUTS = {}


def _oracle_inputs(w, hidden_np=None):
    """The workload's inputs for the oracle; only the experts the batch reaches
    are generated (the oracle touches no other expert)."""
    import oracle
    import workloads as W

    key = (w.name, None if hidden_np is None else hash(hidden_np.tobytes()))
    if key not in _ORACLE_INPUTS:
        hid, router_w, bias = W.router_inputs(w)
        if hidden_np is not None:
            hid = hidden_np
        logits = oracle.router_logits(hid, router_w)
        r = oracle.route_sigmoid(logits, bias, w.top_k, w.route_scale) if w.score_mode == "sigmoid" \
            else oracle.route_softmax(logits, w.top_k, w.renorm_eps)
        gate, up, down = W.expert_weights(w, experts=np.unique(r["idx"]))
        sg, su, sd = W.shared_weights(w)
        _ORACLE_INPUTS.clear()
        _ORACLE_INPUTS[key] = (hid, router_w, bias, gate, up, down, sg, su, sd)
    return _ORACLE_INPUTS[key]


def cpu_baseline(w, hidden_np=None, budget_s: float = 15.0, steps: int | None = None):
    """Time the fp64 oracle (as it stands) on the same workload: whole layers of
    the T-token batch, repeated until the time budget (or `steps` layers) is used."""
    import oracle

    hid, router_w, bias, gate, up, down, sg, su, sd = _oracle_inputs(w, hidden_np)
    runs, t0 = 0, time.perf_counter()
    while True:
        oracle.layer_forward(hid, router_w, bias, gate, up, down, sg, su, sd, top_k=w.top_k,
                             score_mode=w.score_mode, route_scale=w.route_scale, renorm_eps=w.renorm_eps)
        runs += 1
        el = time.perf_counter() - t0
        if (steps is not None and runs >= steps) or (steps is None and el >= budget_s):
            break
    return {"value": round(runs * w.T / el, 3), "unit": UNIT, "cores": _oracle_threads(), "kind": "oracle",
            "sample": f"{runs} whole layer forwards of the {w.T}-token batch (fp64 numpy oracle), {el:.1f}s",
            "seconds_per_layer": round(el / runs, 3)}


# ----------------------------------------------------------------------------- parity against the oracle

PARITY_TOL = {"layer_rel_l2": 5e-3, "layer_max_abs": 3e-2, "router_rel_l2": 1e-5, "near_tie": 1e-5}


def parity_rows(T: int, n: int = 24, seed: int = 11) -> np.ndarray:
    """Rows whose outputs the oracle recomputes: all of a small batch; else the
    first and last four and a seeded sample between them."""
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    mid = rng.choice(np.arange(4, T - 4), size=n - 8, replace=False)
    return np.unique(np.concatenate([np.arange(4), mid, np.arange(T - 4, T)]))


def parity_vs_oracle(smp: dict) -> dict:
    """The GPU's results on one workload against the fp64 oracle: router logits
    (relative L2 over all [T, E]), the selection of every row (equal to the
    oracle's, or a valid choice where the k-th and (k+1)-th keys are within
    1e-5: near ties are counted), and the layer output on the sampled rows
    (relative L2 and max |diff|), the oracle re-evaluated with the GPU's
    selection on near-tie rows."""
    import oracle
    import workloads as W

    w, rows = smp["w"], smp["rows"]
    t0 = time.perf_counter()
    hidden, router_w, bias = W.router_inputs(w)
    logits = oracle.router_logits(hidden, router_w)
    r_rel = float(np.linalg.norm(smp["logits"] - logits) / np.linalg.norm(logits))
    r = (oracle.route_sigmoid(logits, bias, w.top_k, w.route_scale) if w.score_mode == "sigmoid"
         else oracle.route_softmax(logits, w.top_k, w.renorm_eps))
    gsel = np.sort(smp["idx"], axis=1)
    osel = np.sort(r["idx"], axis=1)
    differs = ~(gsel == osel).all(axis=1)
    mand, cand = oracle.near_tie_alternatives(r["keys"], w.top_k, PARITY_TOL["near_tie"])
    T = w.T
    in_g = np.zeros((T, w.E), dtype=bool)
    np.put_along_axis(in_g, smp["idx"].astype(np.int64), True, axis=1)
    valid = (~mand | in_g).all(axis=1) & (~in_g | mand | cand).all(axis=1)
    violations = int((differs & ~(valid & (r["margin"] < PARITY_TOL["near_tie"]))).sum())
    use = np.where((differs & valid)[rows, None], smp["idx"][rows], r["idx"][rows])
    gate, up, down = W.expert_weights(w, experts=np.unique(use))
    sg, su, sd = W.shared_weights(w)
    ref = oracle.layer_forward(hidden[rows], router_w, bias, gate, up, down, sg, su, sd, top_k=w.top_k,
                               score_mode=w.score_mode, route_scale=w.route_scale, renorm_eps=w.renorm_eps,
                               topk_idx=use)["out"]
    got = smp["out_rows"].astype(np.float64)
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    mx = float(np.abs(got - ref).max())
    ok = (rel <= PARITY_TOL["layer_rel_l2"] and mx <= PARITY_TOL["layer_max_abs"]
          and r_rel <= PARITY_TOL["router_rel_l2"] and violations == 0 and smp["device_error"] == 0)
    return {"rows_compared": int(rows.size), "layer_rel_l2": rel, "layer_max_abs": mx, "router_rel_l2": r_rel,
            "near_tie_rows": int((r["margin"] < PARITY_TOL["near_tie"]).sum()),
            "gpu_selection_differs": int(differs.sum()), "selection_violations": violations,
            "max_abs_ref": float(np.abs(ref).max()), "device_error": smp["device_error"], "pass": bool(ok),
            "tolerance": PARITY_TOL, "oracle_seconds": round(time.perf_counter() - t0, 2)}


def oracle_one_core(name: str, steps: int | None = None) -> dict:
    """The oracle on one host core (BLAS threads pinned to 1 in a child process):
    whole layers of a workload's batch."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    n = steps if steps is not None else (20 if name == "tiny" else 1)
    code = ("import json, sys; sys.path.insert(0, %r); import bench, workloads as W; "
            "print(json.dumps(bench.cpu_baseline(W.WORKLOADS[%r], steps=%d)))" % (str(ROOT), name, n))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}"}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["value"], "unit": d["unit"], "cores": 1, "seconds_per_layer": d["seconds_per_layer"]}


def run_reference(args, world):
    import workloads as W

    w = W.WORKLOADS[args.workload]
    for _ in range(args.warmup):
        cpu_baseline(w, steps=1)
    t0 = time.perf_counter()
    cb = cpu_baseline(w, steps=args.steps)
    el = time.perf_counter() - t0
    value = cb["value"]
    ms = 1e3 * el / args.steps
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (same seeded workload as the GPU arm)",
        "config": {**w.describe(), "workload": f"hy3_{args.workload}_T{w.T}"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                         "sample": cb["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "prefill_u", "zipf", "image", "decode_e48", "prefill_e32"])
    ap.add_argument("--profile", action="store_true",
                    help="only run warm-up layer forwards and one more (for hardware-counter captures)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the T=4096 prefill measurement")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the skewed long-prefill (T=16384) and HunyuanImage (T=8192) measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8-weight decode measurement")
    ap.add_argument("--fp8", action="store_true", help="with --profile: run the layer with FP8 expert weights")
    ap.add_argument("--w8a8", action="store_true", help="with --profile: run the W8A8 layer (FP8 weights and activations)")
    ap.add_argument("--phases", action="store_true",
                    help="with --profile: after the warm-up layers, run the expert FFN's gate/up and down as two launches")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, world)), flush=True)
        return

    if world > 1:
        import torch

        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch

        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
