"""MoE decode throughput on GB300: tokens/s of the Granite-MoE-shaped 24-layer stack
(hidden 1024, 32 experts of FFN 512, top-8, q8_0, LRU slot pool holding 50% of the
experts), one decode step = every layer at batch T (router -> slot pool -> expert
GEMVs -> combine).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--batch T]

--impl reference times the fp64 CPU oracle on the same workload (bounded sample per
step) — the slow, obviously-correct program the GPU path is checked against.
Under torchrun (N > 1) each rank runs an independent replica (the path does not
shard; no collective on the data path), value = all ranks' tokens / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE decode tokens/s at batch 1/8/32 (1 GB300); % HBM roofline; cache hit %"
CONFIG_INDEX = 1


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def traffic_record(kernel: str):
    """ncu DRAM bytes per launch recorded in profiles/ncu_traffic.txt, if the kernel source
    is unchanged since the capture (its sha256 matches)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = os.path.join(ROOT, "routed_expert_ffn_gemv_gb300", "csrc", "moe_gemv.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == digest:
            return {"bytes_per_launch": float(parts[2]), "algorithmic_bytes_per_launch": float(parts[3])}
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    def __init__(self, index: int):
        self.proc = None
        self.path = os.path.join(ROOT, "gpurun_out", f"clocks_bench_{os.getpid()}.csv")
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [s.strip() for s in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------------- reference

def run_reference(args, world, rank):
    """The fp64 oracle on the host cores: each step = one layer of one decode step at batch T
    (layers cycled), scaled to a full 24-layer step."""
    if rank != 0:
        return 0
    import oracle
    from routed_expert_ffn_gemv_gb300 import synth
    cfg = synth.config(CONFIG_INDEX)
    T = args.batch
    cores = oracle.num_threads()
    times = []
    for i in range(args.warmup + args.steps):
        layer = i % cfg.L
        x = synth.tokens_x(cfg, 1000 + i, T).astype(np.float64)
        wr, b = synth.router_weights(cfg, layer), synth.router_bias(cfg, layer)
        ids, _, _ = oracle.topk_softmax(oracle.router_logits(x, wr, b), cfg.k)
        experts = {int(e): synth.expert_weights(cfg, layer, int(e)) for e in set(ids.reshape(-1).tolist())}
        t0 = time.perf_counter()
        oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x, wr, b, experts.__getitem__)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    layer_s = float(np.mean(times))
    step_s = layer_s * cfg.L
    tps = T / step_s
    sample = (f"{args.steps} single layers of a batch-{T} decode step (layers cycled), scaled by "
              f"{cfg.L} layers; expert weights generated outside the timed region")
    line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, T), "impl": "reference",
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def workload_config(cfg, T):
    g = cfg.groups[0]
    return {"workload": f"{cfg.name} decode, batch {T}", "layers": cfg.L, "hidden": cfg.H,
            "experts": cfg.E, "ffn": cfg.F, "top_k": cfg.k, "format": "q8_0",
            "pool_slots": g.n_slots, "pool_fraction": g.n_slots / (g.n_layers * cfg.E),
            "batch": T, "l2": "inputs larger than L2: each step streams > 129 MB of expert weights, no flush"}


# ----------------------------------------------------------------------------------- cpu baseline

def cpu_baseline(cfg, T, budget_s=12.0):
    import oracle
    from routed_expert_ffn_gemv_gb300 import synth
    times = []
    t_start = time.perf_counter()
    i = 0
    while time.perf_counter() - t_start < budget_s and i < cfg.L:
        layer = i
        x = synth.tokens_x(cfg, 5000 + i, T).astype(np.float64)
        experts = {}
        wr, b = synth.router_weights(cfg, layer), synth.router_bias(cfg, layer)

        def get(e):
            if e not in experts:
                experts[e] = synth.expert_weights(cfg, layer, e)
            return experts[e]
        # weights generated before the clock starts
        lg = oracle.router_logits(x, wr, b)
        ids, _, _ = oracle.topk_softmax(lg, cfg.k)
        for e in set(ids.reshape(-1).tolist()):
            get(int(e))
        t0 = time.perf_counter()
        oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x, wr, b, get)
        times.append(time.perf_counter() - t0)
        i += 1
    step_s = float(np.mean(times)) * cfg.L
    return {"value": T / step_s, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(times)} layers of one batch-{T} decode step (fp64 C oracle, OpenMP over "
                      f"rows), scaled by {cfg.L} layers"}


# ----------------------------------------------------------------------------------- GPU arm

def time_steps(stack, xs, T, steps, warmup, torch, stream):
    """Warm-up then `steps` decode steps bracketed by events on the launching stream."""
    y = torch.empty((T, stack.cfg.H), dtype=torch.float32, device=xs[0].device)
    for i in range(warmup):
        stack.decode(xs[i % len(xs)], y, stream=stream)
    torch.cuda.synchronize()
    stack.profile_reset()
    stats0 = stack.cache_stats()[0]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        stack.decode(xs[(warmup + i) % len(xs)], y, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    prof = stack.profile()
    stats1 = stack.cache_stats()[0]
    d = {k: (np.array(stats1[k]) - np.array(stats0[k])).tolist() for k in stats1}
    return ms, prof, d


def run_gpu(args, world, rank, local):
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from routed_expert_ffn_gemv_gb300 import _lib as L, synth
    from routed_expert_ffn_gemv_gb300.workload import Stack
    L.load()
    cfg = synth.config(CONFIG_INDEX)
    peaks = load_peaks()
    stack = Stack(cfg, max_T=max(max(cfg.tokens), args.batch), profile=1)
    stream = torch.cuda.Stream()
    batches = [args.batch] if args.lite else sorted(set(list(cfg.tokens) + [args.batch]))
    n_inputs = 64
    inputs = {T: [torch.from_numpy(synth.tokens_x(cfg, 3 + s, T)).cuda() for s in range(n_inputs)]
              for T in batches}
    expert_bytes = cfg.expert_bytes
    gate_up_bytes_per_expert = 2 * cfg.matrix_bytes(cfg.F, cfg.H)

    clocks = ClockSampler(local)
    results = {}
    main = None
    for T in batches:
        steps = args.steps if T == args.batch else max(20, args.steps // 2)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ms, prof, st = time_steps(stack, inputs[T], T, steps, args.warmup, torch, stream)
        if world > 1:
            t = torch.tensor([ms], device="cuda")
            torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
            ms = float(t.item())
        q = sum(st["queries"])
        hits = sum(st["hits"])
        bytes_per_step = q * expert_bytes / steps
        tps = T * steps / (ms / 1e3) * world
        roof8 = T / (bytes_per_step / 8e12)
        roofm = T / (bytes_per_step / (peaks["hbm_gbs"] * 1e9))
        gu_bw = prof["gateup_bytes"] / (prof["gateup_ms"] / 1e3) / 1e9 if prof["gateup_ms"] > 0 else None
        dn_bw = prof["down_bytes"] / (prof["down_ms"] / 1e3) / 1e9 if prof["down_ms"] > 0 else None
        results[T] = {
            "tokens_per_s": tps, "ms_per_step": ms / steps, "steps": steps,
            "hit_rate": hits / q if q else None,
            "route_hit_rate": st["route_hits"] / st["route_queries"] if st["route_queries"] else None,
            "expert_bytes_per_step": bytes_per_step,
            "hbm_roofline_tokens_per_s_8tbs": roof8, "frac_of_8tbs_roofline": tps / world / roof8,
            "frac_of_measured_hbm_roofline": tps / world / roofm,
            "gateup_gbs": gu_bw, "down_gbs": dn_bw,
            "gateup_ms_per_launch": prof["gateup_ms"] / max(1, prof["gateup_launches"]),
            "gateup_bytes_per_launch": prof["gateup_bytes"] / max(1, prof["gateup_launches"]),
            "gateup_ms_per_step": prof["gateup_ms"] / steps,
            "host_wait_ms_per_step": prof["host_wait_ms"] / steps,
            "h2d_bytes_per_step": st["h2d_bytes"] / steps,
            "kernel_launches_per_step": prof["kernel_launches"] / steps,
        }
        if T == args.batch:
            main = (ms, prof, st, steps)

    if args.lite:
        r = results[args.batch]
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["tokens_per_s"], "unit": "tokens/s",
                              "lite": True, "batch": args.batch, "result": r}), flush=True)
        clocks.stop()
        stack.close()
        return 0

    # per-kernel breakdown (events around every kernel; a separate, shorter loop)
    stack.set_profile(2)
    bsteps = max(20, args.steps // 4)
    _, bprof, _ = time_steps(stack, inputs[args.batch], args.batch, bsteps, 3, torch, stream)
    breakdown = {k + "_per_step": bprof[k] / bsteps for k in
                 ("router_ms", "permute_ms", "gateup_ms", "down_ms", "combine_ms", "host_wait_ms")}
    breakdown["down_gbs"] = (bprof["down_bytes"] / (bprof["down_ms"] / 1e3) / 1e9
                             if bprof["down_ms"] > 0 else None)
    breakdown["steps"] = bsteps
    stack.set_profile(0)

    # end-to-end: host (pinned) input -> decode -> host output, copies inside the timed region
    T = args.batch
    xh = [torch.from_numpy(synth.tokens_x(cfg, 900 + s, T)).pin_memory() for s in range(8)]
    yh = torch.empty((T, cfg.H), dtype=torch.float32).pin_memory()
    xd = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    yd = torch.empty_like(xd)
    e2e_steps = max(20, args.steps // 2)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            xd.copy_(xh[i % 8], non_blocking=True)
            stack.decode(xd, yd, stream=stream)
            yh.copy_(yd, non_blocking=True)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            xd.copy_(xh[i % 8], non_blocking=True)
            stack.decode(xd, yd, stream=stream)
            yh.copy_(yd, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    clk = clocks.stop()
    if world > 1:
        t = torch.tensor([e2e_ms], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        e2e_ms = float(t.item())
    e2e_tps = T * e2e_steps / (e2e_ms / 1e3) * world

    ms, prof, st, steps = main
    r = results[args.batch]
    gu_ms_launch = r["gateup_ms_per_launch"]
    gu_bytes_launch = r["gateup_bytes_per_launch"]
    achieved = gu_bytes_launch / (gu_ms_launch / 1e3) / 1e9 if gu_ms_launch > 0 else 0.0
    tr = traffic_record(f"gateup_q8_0_h{cfg.H}_t{T}")
    roofline = {"kernel": "gateup_kernel<q8_0> (dequantising gate/up GEMV)", "bound": "hbm",
                "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                "traffic": None if tr is None else tr["bytes_per_launch"],
                "algorithmic_bytes_per_launch": gu_bytes_launch,
                "launches": prof["gateup_launches"]}
    if rank == 0:
        cb = cpu_baseline(cfg, T) if world == 1 else None
        line = {"metric": METRIC, "value": r["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
                "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded q8_0 experts, N(0,1) activations; no datasets or trained weights)",
                "config": workload_config(cfg, T), "impl": "gb300",
                "hit_rate": r["hit_rate"], "frac_of_8tbs_roofline": r["frac_of_8tbs_roofline"],
                "frac_of_measured_hbm_roofline": r["frac_of_measured_hbm_roofline"],
                "batches": {str(b): results[b] for b in batches},
                "breakdown": breakdown,
                "roofline": roofline, "cpu_baseline": cb,
                "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": T * cfg.H * 4,
                        "d2h_bytes_per_step": T * cfg.H * 4, "steps": e2e_steps},
                "gpu_launches": int(prof["kernel_launches"]),
                "h2d_copies": int(prof["h2d_copies"]),
                "clocks": clk}
        print(json.dumps(line), flush=True)
    stack.close()
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--batch", type=int, default=8)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--lite", action="store_true",
                    help="only the timed loop at --batch (no other batches, breakdown, e2e or CPU "
                         "baseline); used as the ncu target")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
