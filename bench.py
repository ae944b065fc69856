#!/usr/bin/env python
"""Benchmark of the W8A16 / W4A16 fused-MoE layer forward (tokens/s).

One step = one pass of the hot path over one synthetic batch, as one call of
moe_quant_forward_logits (router logits in: routing -- fused into the align
kernel for small batches --, align, gate/up GEMM with fused dequant and
SiLU-and-mul, down GEMM with fused dequant, weighted combine).  Weights
are quantised once before timing (load time, as on the experts_int8 page).

Default workload: the Mixtral-8x7B-shaped W8A16 layer (E=8, k=2, H=4096,
I=14336) at T=64 decode tokens.  Inputs live in HBM; the 1.41 GB of int8
weights exceed the 129 MB L2, so every step streams them from HBM.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--T T]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores

Prints exactly one JSON line (rank 0).
"""

from __future__ import annotations

import argparse
import hashlib
import json
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

from weight_quantized_moe_gb300 import synth  # noqa: E402

PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------- utils --
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="mixtral_decode", choices=sorted(synth.WORKLOADS))
    p.add_argument("--T", type=int, default=64)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--sweep", default="auto",
                   help="comma list of extra T values timed after the main run, 'auto' or 'none'")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--path", default="auto", choices=["auto", "tc", "decode"],
                   help="consumers of the expert GEMMs: by GEMM and batch size (auto), "
                        "tcgen05 for both (tc) or warp-level MMAs for both (decode)")
    return p.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cuda = torch.cuda.is_available()
    if world > 1:
        import torch.distributed as dist
        if cuda:
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if cuda else "gloo")
    elif cuda:
        torch.cuda.set_device(0)
    elif args.impl != "reference":
        raise RuntimeError("bench.py needs a CUDA device (only --impl reference runs on the CPU)")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(x, world, op, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(x, world, device="cuda"):
    """Slowest rank's value (the job's time is the slowest replica's)."""
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.MAX, device)


def sum_over_ranks(x, world, device="cuda"):
    """Whole-job total (tokens processed by all replicas)."""
    import torch.distributed as dist
    return _reduce(x, world, dist.ReduceOp.SUM, device)


def job_throughput(local_tokens, local_ms, world, device="cuda"):
    """Weak-scaling throughput of N independent replicas: all ranks' tokens
    over the slowest rank's time."""
    ms = max_over_ranks(local_ms, world, device)
    return sum_over_ranks(local_tokens, world, device) / (ms / 1e3), ms


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons, 100 ms period."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            uuid = getattr(torch.cuda.get_device_properties(self.dev), "uuid", None)
            ident = f"GPU-{uuid}" if uuid else str(self.dev)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, RuntimeError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workload --
class Problem:
    """One layer's weights (quantised on the device) and one batch."""

    def __init__(self, wl, T, seed, device="cuda", path="auto", weights=None):
        import weight_quantized_moe_gb300 as mq
        self.wl, self.T, self.seed, self.path = wl, T, seed, path
        E, H, I = wl.E, wl.H, wl.I
        self.x = synth.hidden_states(T, H, seed, device=device)
        self.logits = synth.router_logits(T, E, seed, bias=wl.bias, device=device)
        self.w = {} if weights is None else weights  # the same layer's weights, shared
        for which, (N, K) in (("w13", (2 * I, H)), ("w2", (H, I))):
            if which in self.w:
                continue
            bf = synth.expert_weights(E, N, K, seed, which, device=device)
            if wl.bits == 8:
                self.w[which] = mq.moe_quantize_int8_per_channel(bf) + (None,)
            else:
                q, s, z = mq.moe_quantize_uint4_group(bf, wl.group_size)
                self.w[which] = (q, s, z)
            del bf
        torch.cuda.synchronize()
        ws = mq.lib().moe_quant_forward_logits_workspace(T, H, I, E, wl.k, wl.bits, wl.group_size)
        self.ws = torch.empty(max(int(ws), 16), dtype=torch.uint8, device=device)
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        # the routing of this batch, for the touched-expert count (the step
        # routes inside the forward call)
        self.tw, self.tid = mq.moe_topk_route(self.logits, wl.k, wl.renormalize)

    def step(self, x=None, logits=None, out=None):
        import weight_quantized_moe_gb300 as mq
        wl = self.wl
        x = self.x if x is None else x
        logits = self.logits if logits is None else logits
        out = self.out if out is None else out
        (q13, s13, z13), (q2, s2, z2) = self.w["w13"], self.w["w2"]
        # ExpertsInt8MoEMethod.apply(x, router_logits, ...) as one call:
        # routing, align, both expert GEMMs and the combine
        mq.moe_quant_forward_logits(x, logits, q13, q2, s13, s2, wl.k, wl.renormalize,
                                    bits=wl.bits, group_size=wl.group_size, has_zp=wl.has_zp,
                                    z13=z13, z2=z2, workspace=self.ws, out=out, path=self.path)
        return out

    def touched_experts(self):
        return np.unique(self.tid.cpu().numpy())


class EndToEnd:
    """A serving loop through the public API with pinned host buffers: every
    step copies its x and router logits to the device, runs the forward and
    copies its output back to the host.  The copies run on their own streams
    with two device buffers of each, so step i+1's upload and step i's
    download overlap step i's kernels, as a server would pipeline them."""

    def __init__(self, prob):
        self.prob = prob
        T, H = prob.x.shape
        self.x_h = prob.x.cpu().pin_memory()
        self.lg_h = prob.logits.cpu().pin_memory()
        self.out_h = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        self.x_d = [torch.empty_like(prob.x) for _ in range(2)]
        self.lg_d = [torch.empty_like(prob.logits) for _ in range(2)]
        self.out_d = [torch.empty_like(prob.out) for _ in range(2)]
        self.h2d = torch.cuda.Stream()
        self.d2h = torch.cuda.Stream()
        ev = lambda: [torch.cuda.Event() for _ in range(2)]
        self.ev_in, self.ev_done, self.ev_down = ev(), ev(), ev()
        self.i = 0

    def step(self):
        s = self.i & 1
        comp = torch.cuda.current_stream()
        with torch.cuda.stream(self.h2d):  # after the forward that last read slot s
            self.h2d.wait_event(self.ev_done[s])
            self.x_d[s].copy_(self.x_h, non_blocking=True)
            self.lg_d[s].copy_(self.lg_h, non_blocking=True)
            self.ev_in[s].record(self.h2d)
        comp.wait_event(self.ev_in[s])
        comp.wait_event(self.ev_down[s])  # slot s's previous output is on the host
        self.prob.step(self.x_d[s], self.lg_d[s], out=self.out_d[s])
        self.ev_done[s].record(comp)
        with torch.cuda.stream(self.d2h):
            self.d2h.wait_event(self.ev_done[s])
            self.out_h[s].copy_(self.out_d[s], non_blocking=True)
            self.ev_down[s].record(self.d2h)
        self.i += 1

    def finish(self):
        """The last download belongs to the timed region."""
        torch.cuda.current_stream().wait_stream(self.d2h)


def algorithmic_work(wl, T, touched):
    """Per-launch algorithmic bytes and flops of the two expert GEMMs (and
    of the one-launch layer that runs both)."""
    S = T * wl.k
    n_touched = len(touched)
    H, I = wl.H, wl.I
    if wl.bits == 8:
        w13 = 2 * I * H + 4 * 2 * I
        w2 = H * I + 4 * H
    else:
        gs = wl.group_size
        w13 = I * H + 2 * 2 * I * (H // gs) + (I * (H // gs) if wl.has_zp else 0)
        w2 = H * I // 2 + 2 * H * (I // gs) + ((H // 2) * (I // gs) if wl.has_zp else 0)
    g1 = {"bytes": n_touched * w13 + T * H * 2 + S * I * 2, "flops": 4.0 * S * I * H}
    g2 = {"bytes": n_touched * w2 + S * I * 2 + S * H * 4, "flops": 2.0 * S * I * H}
    # the one-launch layer (8-bit, many experts) runs both GEMMs in one kernel
    layer = {"bytes": g1["bytes"] + g2["bytes"], "flops": g1["flops"] + g2["flops"]}
    return {"gemm1": g1, "gemm2": g2, "layer": layer}


def time_loop(fn, steps, warmup, world, finish=None):
    """Device time of `steps` calls of fn (ms), CUDA events on the current
    stream; `finish` joins any side streams into it before the end event."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(steps):
        fn()
    if finish is not None:
        finish()
    b.record(st)
    torch.cuda.synchronize()
    barrier(world)
    return a.elapsed_time(b)


def time_steps_flushed(fn, steps, warmup, flush):
    """Device time of `steps` calls of fn (ms), each preceded by a write of a
    buffer larger than L2 outside the timed part (for layers whose touched
    weights would otherwise stay resident in the 129 MB L2)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    evs = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        fn()
        b.record(st)
        evs.append((a, b))
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in evs)


L2_BYTES = 129 * 2 ** 20


def profile_kernels(fn, steps, world):
    """{kernel slot: (total ms, launches)} of a separate pass of `steps`
    calls, each kernel bracketed by events on its stream."""
    import weight_quantized_moe_gb300 as mq
    mq.mq_profile_enable(True)
    time_loop(fn, steps, 2, world)
    mq.mq_profile_enable(False)
    return mq.mq_profile_read()


def roofline_of(wl, T, prof, touched, peaks, long_run, traffic_key=None):
    """Roofline of the dominant expert GEMM: algorithmic bytes (decode) or
    flops (prefill) per launch over its mean launch time."""
    work = algorithmic_work(wl, T, touched)
    kern = max(("gemm1", "gemm2", "layer"), key=lambda k: prof.get(k, (0, 1))[0])
    k_ms, k_n = prof[kern]
    k_ms_launch = k_ms / max(k_n, 1)
    wk = work[kern]
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    if wk["flops"] / wk["bytes"] > ridge:
        achieved = wk["flops"] / (k_ms_launch / 1e3) / 1e12
        peak = peaks["bf16_tflops_sustained"] if long_run else peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "peak_kind": "sustained" if long_run else "burst"}
    else:
        achieved = wk["bytes"] / (k_ms_launch / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    roof.update({"kernel": kern,
                 "traffic": ncu_traffic(kern, traffic_key) if traffic_key else None,
                 "algorithmic_bytes_per_launch": wk["bytes"],
                 "algorithmic_flops_per_launch": wk["flops"],
                 "ms_per_launch": k_ms_launch,
                 "peak_source": peaks["source"] + " (MEASURED_PEAKS.json)"
                 if peaks["source"] == "measured" else "fallback",
                 "kernel_ms_per_step": {k: v[0] / v[1] for k, v in prof.items()}})
    return roof


def measure_entry(wl, T, seed, steps, world, peaks, path, weights=None, flush=None):
    """One extra workload of the line: whole-step tokens/s, the dominant
    kernel's roofline, the step's HBM fraction and the routing's load."""
    prob = Problem(wl, T, seed, path=path, weights=weights)
    touched = prob.touched_experts()
    bytes_touched = len(touched) * wl.bytes_per_expert()
    use_flush = flush is not None and bytes_touched < 2 * L2_BYTES
    if use_flush:
        ms = time_steps_flushed(prob.step, steps, 3, flush)
    else:
        ms = time_loop(prob.step, steps, 3, world)
    ms = max_over_ranks(ms, world)
    prof = profile_kernels(prob.step, steps, world)
    work = algorithmic_work(wl, T, touched)
    step_bytes = work["gemm1"]["bytes"] + work["gemm2"]["bytes"]
    ms_step = ms / steps
    ent = {"workload": f"{wl.name} T={T}", "T": T,
           "tokens_per_s": sum_over_ranks(T * steps, world) / (ms / 1e3),
           "ms_per_step": ms_step,
           "touched_experts": int(len(touched)),
           "zero_token_experts": int(wl.E - len(touched)),
           "hbm_frac_step": step_bytes / (ms_step / 1e3) / 1e9 / peaks["hbm_gbs"],
           "tflops_step": wl.flops(T) / (ms_step / 1e3) / 1e12,
           "roofline": roofline_of(wl, T, prof, touched, peaks, long_run=False,
                                   traffic_key=f"{wl.name}_T{T}"),
           "l2": "flushed between steps (touched weights < 2x L2)" if use_flush
           else "touched weights larger than L2 stream from HBM every step"}
    return ent, prob.w


def kernel_source_sha():
    import glob
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "weight_quantized_moe_gb300", "csrc", "*"))):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload_key):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    ent = d.get(f"{kernel}@{workload_key}")
    if not ent or ent.get("source_sha") != kernel_source_sha():
        return None
    return ent.get("dram_bytes_per_launch")


# ---------------------------------------------------------------- oracle --
def oracle_sample(wl, T, seed, n_tokens, device=None):
    """Inputs for timing the CPU oracle on a bounded token sample of the
    workload: the oracle quantises the touched experts itself (load time,
    untimed); the timed part is route + align + forward on the sample."""
    import oracle
    if device is None:  # the generators run on the GPU when there is one
        device = "cuda" if torch.cuda.is_available() else "cpu"
    x = synth.hidden_states(T, wl.H, seed, device=device).float().cpu().numpy()
    lg = synth.router_logits(T, wl.E, seed, bias=wl.bias, device=device).cpu().numpy()
    _, ids = oracle.topk_route(lg, wl.k, wl.renormalize)
    tokens = np.arange(min(n_tokens, T))
    touched = np.unique(ids[tokens])
    E, H, I = wl.E, wl.H, wl.I
    if wl.bits == 8:
        ex = oracle.Int8Experts(np.zeros((E, 2 * I, H), np.int8), np.zeros((E, 2 * I), np.float32),
                                np.zeros((E, H, I), np.int8), np.zeros((E, H), np.float32))
    else:
        gs = wl.group_size
        ex = oracle.Uint4Experts(
            np.zeros((E, 2 * I, H // 2), np.uint8), np.zeros((E, 2 * I, H // gs), np.float16),
            np.zeros((E, I, H // gs), np.uint8), np.zeros((E, H, I // 2), np.uint8),
            np.zeros((E, H, I // gs), np.float16), np.zeros((E, H // 2, I // gs), np.uint8),
            gs, wl.has_zp)
    for e in touched:
        for which, (N, K) in (("w13", (2 * I, H)), ("w2", (H, I))):
            w = synth.expert_weights(E, N, K, seed, which, device=device,
                                     experts=[int(e)])[0].float().cpu().numpy()
            if wl.bits == 8:
                q, s = oracle.quantize_int8_per_channel(w)
                if which == "w13":
                    ex.w13[e], ex.s13[e] = q, s
                else:
                    ex.w2[e], ex.s2[e] = q, s
            else:
                q, s, z = oracle.quantize_uint4_group(w, wl.group_size)
                packed = (oracle.pack_uint4_along_k(q), s, oracle.pack_uint4_along_n(z))
                if which == "w13":
                    ex.qw13[e], ex.sc13[e], ex.qz13[e] = packed
                else:
                    ex.qw2[e], ex.sc2[e], ex.qz2[e] = packed

    def run():
        w, ids = oracle.topk_route(lg, wl.k, wl.renormalize)
        oracle.align_block(ids, wl.E, 16)
        oracle.moe_forward(x, ex, w, ids, tokens=tokens)

    return run, len(tokens)


def oracle_tokens_for(wl):
    per_expert = wl.bytes_per_expert()
    # about 2-5 s of CPU work per step at ~1 GB/s of dequantised expert bytes
    return max(1, int(4e9 // (per_expert * wl.k * 8)))


def cpu_baseline(wl, T, seed, min_seconds=10.0, max_seconds=30.0):
    """The oracle, as it stands, on a bounded sample of the workload, repeated
    until at least `min_seconds` of CPU work have been timed."""
    n_tok = max(1, min(T, 4 * oracle_tokens_for(wl)))
    run, n = oracle_sample(wl, T, seed, n_tok)
    reps, dt = 0, 0.0
    t0 = time.perf_counter()
    while dt < min_seconds and (reps == 0 or dt + dt / reps < max_seconds):
        run()
        reps += 1
        dt = time.perf_counter() - t0
    return {"value": n * reps / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{reps} x (route+align of all {T} tokens, expert MLP of the first {n} tokens); "
                      f"oracle: numpy float64, BLAS matmuls threaded, dequant single-threaded",
            "seconds": dt}


def run_reference(args, world, rank):
    wl = synth.WORKLOADS[args.workload]
    if rank != 0:
        return
    n_tok = max(1, min(args.T, oracle_tokens_for(wl)))
    run, n = oracle_sample(wl, args.T, args.seed, n_tok)
    for _ in range(max(args.warmup, 0)):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "impl": "reference", "metric": "W8A16 fused-MoE layer tokens/s" if wl.bits == 8
        else "W4A16 fused-MoE layer tokens/s",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(wl, args.T),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"per step: route+align of {args.T} tokens, expert MLP of {n} tokens"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(wl, T):
    return {"workload": f"{wl.name} T={T}", "E": wl.E, "top_k": wl.k, "H": wl.H, "I": wl.I,
            "T": T, "renormalize": wl.renormalize, "weights": "int8 per-channel" if wl.bits == 8
            else f"uint4 gs={wl.group_size} zp={int(wl.has_zp)}", "activations": "bf16",
            "router_bias": wl.bias or "none",
            "l2": "weights larger than the 129 MB L2 stream from HBM every step"}


# ------------------------------------------------------------------ main --
def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    import weight_quantized_moe_gb300 as mq
    mq.lib()
    wl = synth.WORKLOADS[args.workload]
    T = args.T
    peaks = measured_peaks()
    prob = Problem(wl, T, args.seed + rank, path=args.path)

    clocks = ClockSampler(torch.cuda.current_device()).start()
    time.sleep(0.3)
    for _ in range(args.warmup):  # warm-up first, so that the count below is the timed steps'
        prob.step()
    launches0 = mq.mq_kernel_launch_count()
    ms = time_loop(prob.step, args.steps, 0, world)
    launches = mq.mq_kernel_launch_count() - launches0
    clk = clocks.stop()
    assert mq.mq_device_status() == 0, "device status flagged during the timed run"

    value, ms_max = job_throughput(T * args.steps, ms, world)
    tokens_all = sum_over_ranks(T * args.steps, world)

    # per-kernel device times (separate pass of the same steps, events on the
    # launching stream)
    prof = profile_kernels(prob.step, args.steps, world)
    touched = prob.touched_experts()
    roof = roofline_of(wl, T, prof, touched, peaks, long_run=ms_max > 1000.0,
                       traffic_key=f"{wl.name}_T{T}")
    roof["touched_experts"] = int(len(touched))

    # end to end through the public API with host buffers
    e2e_run = EndToEnd(prob)
    e2e_ms = max_over_ranks(time_loop(e2e_run.step, args.steps, args.warmup, world,
                                      finish=e2e_run.finish), world)
    e2e = {"value": tokens_all / (e2e_ms / 1e3), "unit": "tokens/s",
           "h2d_bytes_per_step": T * wl.H * 2 + T * wl.E * 4, "d2h_bytes_per_step": T * wl.H * 2}

    # the rest of the metric: the decode sweep of the same layer, the
    # prefill half (the same weights, routed with the prefill bias), and the
    # fine-grained and W4A16 layers
    steps_x = max(20, args.steps // 4)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    clocks_x = ClockSampler(torch.cuda.current_device()).start()
    sweep = []
    extra = []
    if args.sweep == "auto":
        extra = [(wl, t) for t in wl.Ts if t != T]
        if wl.name == "mixtral_decode":
            extra += [(synth.WORKLOADS["fine"], 64), (synth.WORKLOADS["fine"], 512),
                      (synth.WORKLOADS["w4a16"], 32)]
    elif args.sweep not in ("none", ""):
        extra = [(wl, int(t)) for t in args.sweep.split(",")]
    shared = {wl.name: prob.w}
    for wl2, t in extra:
        ent, w = measure_entry(wl2, t, args.seed + rank, steps_x, world, peaks, args.path,
                               weights=shared.get(wl2.name), flush=flush)
        shared[wl2.name] = w
        sweep.append(ent)
    prefill = None
    if args.sweep == "auto" and wl.name == "mixtral_decode":
        pwl = synth.WORKLOADS["mixtral_prefill"]
        prefill, _ = measure_entry(pwl, 4096, args.seed + rank, steps_x, world, peaks, args.path,
                                   weights=prob.w)
    shared.clear()
    del flush
    clk_x = clocks_x.stop()

    line = {
        "metric": "W8A16 fused-MoE layer tokens/s" if wl.bits == 8 else "W4A16 fused-MoE layer tokens/s",
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": ("bf16 activations in/out; int8 weight codes dequantised exactly to f16 "
                  "(gate/up, activations scaled exactly by a power of two per row) or bf16 "
                  "(down); float32 accumulation") if wl.bits == 8 else
                 ("bf16 activations in/out; uint4 codes with f16 group scales as f16 operands; "
                  "float32 accumulation"),
        "data": "synthetic (seeded N(0,1) activations/logits, N(0,0.02) weights quantised on device)",
        "config": workload_config(wl, T), "roofline": roof, "e2e": e2e,
        "gpu_launches": int(launches), "clocks": clk, "sweep": sweep, "prefill": prefill,
        "clocks_sweep": clk_x,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, T, args.seed)
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
