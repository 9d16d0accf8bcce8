"""MoE decode throughput on GB300: tokens/s of the Granite-MoE-shaped 24-layer stack
(hidden 1024, 32 experts of FFN 512, top-8, q8_0, LRU slot pool holding 50% of the
experts), one decode step = every layer at batch T (router -> slot pool -> expert
GEMVs -> combine + pre-norm of the next layer).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--batch T] [--impl reference] [--lite]

The headline runs the device-managed pool (LRU planned on the GPU, missed experts read
from pinned host memory and written into their slots by the GEMV kernels themselves) with
the whole step replayed as a CUDA graph.  The host-managed pool (moe_cache_ensure + copy
engine uploads) is measured too; its profiled loop gives the gate/up GEMV roofline, since
there every GEMV byte comes from HBM.  The tcgen05 prefill grouped GEMM (Qwen-shaped layer,
512 and 4096 tokens) is measured against the dense tensor peak.

--impl reference times the fp64 CPU oracle on the same workload (bounded sample per step).
Under torchrun (N > 1) each rank runs an independent replica (the path does not shard; no
collective on the data path); value = all ranks' tokens / max time over ranks.
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
HEADLINE_PREFETCH = 1  # cross-layer speculative prefetch depth of the headline stack


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
    """ncu DRAM bytes per launch from profiles/ncu_traffic.txt, if the kernel source is unchanged
    since the capture (sha256 prefix of csrc/moe_gemv.cu matches)."""
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
    """nvidia-smi clock / throttle sampling during the timed regions."""

    def __init__(self, index: int):
        self.proc = None
        # the raw samples (the JSON line carries their summary); BENCH_LOG_DIR moves them
        log_dir = os.environ.get("BENCH_LOG_DIR", os.path.join(ROOT, "bench_logs"))
        self.path = os.path.join(log_dir, f"clocks_bench_{os.getpid()}.csv")
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


def dist_setup():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def workload_config(cfg, T):
    g = cfg.groups[0]
    return {"workload": f"{cfg.name} decode, batch {T}", "layers": cfg.L, "hidden": cfg.H,
            "experts": cfg.E, "ffn": cfg.F, "top_k": cfg.k, "format": "q8_0",
            "pool_slots": g.n_slots, "pool_fraction": g.n_slots / (g.n_layers * cfg.E),
            "batch": T, "stack": "h <- h + MoE(RMSNorm(h))",
            "l2": "inputs larger than L2: each step streams > 129 MB of expert weights, no flush"}


# ----------------------------------------------------------------------------------- CPU oracle

def _oracle_layer_time(cfg, layer, T, seed):
    """Times one oracle layer on T tokens (routed and shared experts); the experts are
    generated before the clock starts."""
    import oracle
    from routed_expert_ffn_gemv_gb300 import synth
    x = synth.tokens_x(cfg, seed, T).astype(np.float64)
    wr, b = synth.router_weights(cfg, layer), synth.router_bias(cfg, layer)
    ids, _, _ = oracle.topk_softmax(oracle.router_logits(x, wr, b), cfg.k)
    experts = {int(e): synth.expert_weights(cfg, layer, int(e)) for e in set(ids.reshape(-1).tolist())}
    shared = [synth.expert_weights(cfg, layer, cfg.E + s) for s in range(cfg.n_shared)]
    t0 = time.perf_counter()
    oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x, wr, b, experts.__getitem__, shared=shared)
    return time.perf_counter() - t0


def cpu_sample(cfg, T, budget_s):
    """The fp64 oracle (every host thread) on a bounded sample of one batch-T decode step's
    layers, scaled to the whole step."""
    import oracle
    times, t_start = [], time.perf_counter()
    while (time.perf_counter() - t_start < budget_s or not times) and len(times) < cfg.L:
        times.append(_oracle_layer_time(cfg, len(times), T, 6000 + len(times)))
    step_s = float(np.mean(times)) * cfg.L
    return {"value": T / step_s, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(times)} of {cfg.L} layers of one batch-{T} step, scaled to the step"}


def cpu_baseline(cfg, T, budget_s=12.0, budget_1t_s=4.0):
    """The fp64 C oracle on the host cores: a bounded sample of the layers of one batch-T
    decode step with every thread (OpenMP over the expert rows), scaled to the step; then a
    smaller sample with one thread."""
    import oracle
    from oracle import build as obuild
    times, t_start, i = [], time.perf_counter(), 0
    while time.perf_counter() - t_start < budget_s and i < cfg.L:
        times.append(_oracle_layer_time(cfg, i, T, 5000 + i))
        i += 1
    step_s = float(np.mean(times)) * cfg.L
    cores = oracle.num_threads()
    t1, t_start = [], time.perf_counter()
    oracle.set_num_threads(1)
    try:
        while (time.perf_counter() - t_start < budget_1t_s or not t1) and len(t1) < cfg.L:
            t1.append(_oracle_layer_time(cfg, len(t1), T, 7000 + len(t1)))
    finally:
        oracle.set_num_threads(cores)
    step1_s = float(np.mean(t1)) * cfg.L
    return {"value": T / step_s, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{len(times)} layers of one batch-{T} decode step (fp64 C oracle, OpenMP over "
                      f"rows), scaled by {cfg.L} layers",
            "s_per_token": step_s / T, "one_thread": {"value": T / step1_s, "s_per_token": step1_s / T,
                                                     "sample": f"{len(t1)} layers, scaled by {cfg.L}"},
            "affinity_cpus": len(os.sched_getaffinity(0)), "compiler": "gcc " + " ".join(obuild.CFLAGS)}


def run_reference(args, world, rank):
    """The fp64 oracle on the host cores: each step = one layer of a batch-T decode step
    (layers cycled), scaled to a full step."""
    if rank != 0:
        return 0
    import oracle
    from routed_expert_ffn_gemv_gb300 import synth
    cfg = synth.config(CONFIG_INDEX)
    T = args.batch
    times = []
    for i in range(args.warmup + args.steps):
        dt = _oracle_layer_time(cfg, i % cfg.L, T, 1000 + i)
        if i >= args.warmup:
            times.append(dt)
    step_s = float(np.mean(times)) * cfg.L
    tps = T / step_s
    sample = (f"{args.steps} single layers of a batch-{T} decode step (layers cycled), scaled by "
              f"{cfg.L} layers; expert weights generated outside the timed region")
    line = {"metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, T), "impl": "reference",
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------------- GPU arm

def time_steps(stack, xs, T, steps, warmup, torch, stream):
    """Warm-up, then `steps` decode steps bracketed by events on the launching stream."""
    y = torch.empty((T, stack.cfg.H), dtype=torch.float32, device=xs[0].device)
    for i in range(warmup):
        stack.decode(xs[i % len(xs)], y, stream=stream)
    torch.cuda.synchronize()
    stack.profile_reset()
    stats0 = stack.cache_stats()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        stack.decode(xs[(warmup + i) % len(xs)], y, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    prof = stack.profile()
    stats1 = stack.cache_stats()
    d = {}
    for k in stats1[0]:
        d[k] = (sum(np.array(s1[k]) - np.array(s0[k]) for s0, s1 in zip(stats0, stats1))).tolist()
    return ms, prof, d


def time_window(stack, xs, T, total, warmup, torch, stream):
    """From an empty pool: `warmup` untimed steps, then `total - warmup` steps bracketed by
    events on the launching stream.  Returns (ms, statistics of the timed steps, statistics
    of all `total` steps from the cold start)."""
    y = torch.empty((T, stack.cfg.H), dtype=torch.float32, device=xs[0].device)
    stack.reset_caches()
    for i in range(warmup):
        stack.decode(xs[i % len(xs)], y, stream=stream)
    torch.cuda.synchronize()
    stats0 = stack.cache_stats()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(warmup, total):
        stack.decode(xs[i % len(xs)], y, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    stats1 = stack.cache_stats()
    timed, cold = {}, {}
    for k in (stats1[0] if stats1 else {}):
        timed[k] = (sum(np.array(s1[k]) - np.array(s0[k]) for s0, s1 in zip(stats0, stats1))).tolist()
        cold[k] = (sum(np.array(s1[k]) for s1 in stats1)).tolist()
    return e0.elapsed_time(e1), timed, cold


def hit_fields(st, prefix=""):
    """Hit rates of a statistics dict: per distinct (layer, expert) query, per route, and by
    ubatch bucket (<= 8 tokens, 9..32 tokens)."""
    q, h = st["queries"], st["hits"]
    out = {prefix + "hit_rate": sum(h) / sum(q) if sum(q) else None,
           prefix + "route_hit_rate": st["route_hits"] / st["route_queries"] if st["route_queries"] else None}
    for i, name in enumerate(("le8", "9to32")):
        if q[i]:
            out[prefix + f"hit_rate_{name}"] = h[i] / q[i]
    return out


def run_config(ci, Ts, torch, stream, peaks, link_gbs, warmup, total=256, stack=None, cpu_budget_s=4.0,
               world=1, rank=0, resident=True):
    """One decode configuration at each batch size in Ts: the device-managed pool (the
    configuration's slot counts, LRU on the GPU, misses read over the CPU-GPU link),
    `total` steps from a cold pool of which the last total - warmup are timed, whole steps
    replayed as CUDA graphs; then the same timed steps with every expert resident in HBM
    (the HBM ceiling of the step); and the fp64 oracle on a bounded sample."""
    from routed_expert_ffn_gemv_gb300 import synth
    from routed_expert_ffn_gemv_gb300.workload import PinnedImages, Stack
    cfg = synth.config(ci)
    own = stack is None
    if own:
        images = PinnedImages(cfg, range(cfg.L), range(cfg.E))
        stack = Stack(cfg, max_T=max(Ts), device_managed=True, use_graph=True, images=images)
    images = stack.images
    out = {}
    xs = {T: [torch.from_numpy(synth.tokens_x(cfg, 3 + s, T)).cuda() for s in range(total)] for T in Ts}
    shared_bytes = cfg.L * cfg.n_shared * cfg.expert_bytes
    for T in Ts:
        ms, st, cold = time_window(stack, xs[T], T, total, warmup, torch, stream)
        ms = max_over_ranks(ms, world, torch)
        steps = total - warmup
        bytes_step = sum(st["queries"]) * cfg.expert_bytes / steps + shared_bytes
        tps = T * steps / (ms / 1e3)
        roof8 = T / (bytes_step / 8e12)
        e = {"workload": f"{cfg.name} decode, batch {T}", "tokens_per_s": tps * world,
             "ms_per_step": ms / steps, "steps_timed": steps, "steps_from_cold": total,
             "pool": "+".join(str(g.n_slots) for g in cfg.groups) + " slots of "
                     + "+".join(str(g.n_layers * cfg.E) for g in cfg.groups) + " experts",
             "expert_bytes_per_step": bytes_step, "miss_bytes_per_step": st["h2d_bytes"] / steps,
             "frac_of_8tbs_roofline": tps / roof8, "frac_of_measured_hbm_roofline":
                 tps / (T / (bytes_step / (peaks["hbm_gbs"] * 1e9)))}
        e.update(hit_fields(st))
        e.update(hit_fields(cold, "from_cold_"))
        miss_b = st["h2d_bytes"] / steps
        t_att = miss_b / (link_gbs * 1e9) + (bytes_step - miss_b) / (peaks["hbm_gbs"] * 1e9)
        e["frac_of_link_aware_attainable"] = tps / (T / t_att)
        out[T] = e
    stack.close()
    if not resident:
        del images
        torch.cuda.empty_cache()
        return out
    # every expert resident in HBM, the same inputs (the same routing, so the same bytes)
    res = Stack(cfg, max_T=max(Ts), resident=True, use_graph=True, images=images)
    for T in Ts:
        ms, _, _ = time_window(res, xs[T], T, total, warmup, torch, stream)
        ms = max_over_ranks(ms, world, torch)
        steps = total - warmup
        tps = T * steps / (ms / 1e3)
        b = out[T]["expert_bytes_per_step"]
        out[T].update({"resident_tokens_per_s": tps * world, "resident_ms_per_step": ms / steps,
                       "resident_frac_of_8tbs_roofline": tps / (T / (b / 8e12)),
                       "resident_frac_of_measured_hbm_roofline": tps / (T / (b / (peaks["hbm_gbs"] * 1e9)))})
    res.close()
    del res, images
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and cpu_budget_s > 0:
        for T in Ts:
            out[T]["cpu_baseline"] = cpu_sample(cfg, T, cpu_budget_s)
    return out


POLICIES = (
    # name, pool mode, Stack options (page 3 section 2.2: frequency admission; page 1 section 4.3:
    # --moe-lru-window 15 and --moe-expert-load-threshold 0.05)
    ("lru_device", dict(device_managed=True, use_graph=True)),
    ("admit2_device", dict(device_managed=True, use_graph=True, admit_after=2)),
    ("admit4_device", dict(device_managed=True, use_graph=True, admit_after=4)),
    ("load_threshold_0.05_device", dict(device_managed=True, use_graph=True, load_threshold=0.05)),
    # page 3 sections 2.3 / 4.3: cross-layer speculative prefetch, depth 1 and 2
    ("prefetch1_device", dict(device_managed=True, use_graph=True, prefetch_depth=1)),
    ("prefetch2_device", dict(device_managed=True, use_graph=True, prefetch_depth=2)),
    ("lru_host", dict()),
    ("window15_host", dict(lru_window=15)),
)


def run_policies(torch, stream, peaks, link_gbs, warmup, total=128, T=8):
    """The Granite-shaped stack at batch 8 (where plain LRU hits nothing: the 24 layers' ~720
    distinct experts per step cycle through 384 slots) under each pool policy: tokens/s, hit
    rates, bypassed misses and window evictions over `total - warmup` timed steps from a cold
    pool.  The load threshold changes the routing (fewer routes, a different result); the
    other policies only change where the weights are read from."""
    from routed_expert_ffn_gemv_gb300 import synth
    from routed_expert_ffn_gemv_gb300.workload import PinnedImages, Stack
    cfg = synth.config(1)
    images = PinnedImages(cfg, range(cfg.L), range(cfg.E))
    xs = [torch.from_numpy(synth.tokens_x(cfg, 3 + s, T)).cuda() for s in range(total)]
    out = {}
    for name, kw in POLICIES:
        st = Stack(cfg, max_T=T, images=images, **kw)
        ms, tst, cold = time_window(st, xs, T, total, warmup, torch, stream)
        steps = total - warmup
        e = {"tokens_per_s": T * steps / (ms / 1e3), "ms_per_step": ms / steps,
             "miss_bytes_per_step": tst["h2d_bytes"] / steps,
             "routes_per_step": tst["route_queries"] / steps,
             "bypassed_per_step": tst["bypassed"] / steps,
             "window_evictions_per_step": tst["window_evictions"] / steps,
             "prefetch_fills_per_step": tst["prefetch_fills"] / steps,
             "prefetch_hits_per_step": tst["prefetch_hits"] / steps}
        e.update(hit_fields(tst))
        out[name] = e
        st.close()
    del images
    torch.cuda.empty_cache()
    return out


def gemv_roofline(cfg, T, torch, stream, steps=40, warmup=5):
    """The decode GEMV kernels on HBM-resident weights: every layer's experts resident (24 x 32
    images, 1.28 GB, far above L2); every layer's router and permute run first, then rounds of
    the gate/up GEMV of all layers are launched back to back on `stream` between two CUDA
    events (so no launch finds its weights in L2 and no event sits between launches), then of
    the down GEMV, then of each layer's whole chain (permute, the GEMVs).
    Bytes per launch are the active experts' quantised blocks, counted on the device.
    `steps` rounds are timed after `warmup` untimed ones (at least 3 each)."""
    from routed_expert_ffn_gemv_gb300 import _lib as L, synth
    from routed_expert_ffn_gemv_gb300.workload import Stack
    st = Stack(cfg, max_T=T, resident=True, profile=0)
    x = torch.from_numpy(synth.tokens_x(cfg, 500, T)).cuda()
    with torch.cuda.stream(stream):
        st.gemv_timing(x, max(3, warmup), stream=stream)
        r = st.gemv_timing(x, max(3, steps), stream=stream)
    st.close()
    return {"gateup_ms_per_launch": r["gateup_us"] / 1e3, "gateup_bytes_per_launch": r["gateup_bytes"],
            "down_ms_per_launch": r["down_us"] / 1e3, "down_bytes_per_launch": r["down_bytes"],
            "reduce_ms_per_launch": r["reduce_us"] / 1e3,
            "gemv_ms_per_launch": r["gemv_us"] / 1e3, "fused": bool(r["fused"]),
            "launches": int(r["launches"]), "steps": steps}


def gemv_roofline_block(gv, cfg, T, peaks):
    """The roofline object of the JSON line: the decode path's dominant kernel, the gate/up
    GEMV (ffn_warp_kernel, two thirds of the weight bytes), timed in rounds of its own launches
    back to back; beside it the down GEMV and the K-split reduce timed the same way, and one
    layer's whole chain (permute, gate/up, reduce, down; or the fused launch when the library
    runs it) with the selected experts' bytes of all three matrices."""
    def gbs(b, ms):
        return b / (ms / 1e3) / 1e9 if ms > 0 else 0.0
    hbm = peaks["hbm_gbs"]
    gu_ms, gu_b = gv["gateup_ms_per_launch"], gv["gateup_bytes_per_launch"]
    dn_ms, dn_b = gv["down_ms_per_launch"], gv["down_bytes_per_launch"]
    ch_ms, ch_b = gv["gemv_ms_per_launch"], gu_b + dn_b
    tr = traffic_record(f"gateup_q8_0_h{cfg.H}_t{T}")
    chain = ("permute_kernel -> ffn_fused_kernel (gate/up + reduce + down in one launch)" if gv["fused"] else
             "permute_kernel -> ffn_warp_kernel<gate/up> -> ks_reduce_kernel -> ffn_warp_kernel<down>")
    return {"kernel": "ffn_warp_kernel<q8_0, gate/up> (dequantising gate/up GEMV + SwiGLU)", "bound": "hbm",
            "achieved": gbs(gu_b, gu_ms), "peak": hbm, "unit": "GB/s", "frac": gbs(gu_b, gu_ms) / hbm,
            "peak_source": peaks["source"], "traffic": None if tr is None else tr["bytes_per_launch"],
            "algorithmic_bytes_per_launch": gu_b, "ms_per_launch": gu_ms, "launches": gv["launches"],
            "down_achieved_gbs": gbs(dn_b, dn_ms), "down_frac": gbs(dn_b, dn_ms) / hbm,
            "down_ms_per_launch": dn_ms, "down_algorithmic_bytes_per_launch": dn_b,
            "ks_reduce_kernel_ms_per_launch": gv["reduce_ms_per_launch"],
            "layer_chain_kernels": chain, "layer_chain_achieved_gbs": gbs(ch_b, ch_ms),
            "layer_chain_frac": gbs(ch_b, ch_ms) / hbm, "layer_chain_ms_per_layer": ch_ms,
            "layer_chain_algorithmic_bytes_per_layer": ch_b,
            "measured_in": ("HBM-resident stack (all %d x %d expert images in HBM, above L2), batch %d; "
                            "each kernel (and each layer's chain) launched back to back over all layers in "
                            "rounds, CUDA events on the launching stream around the rounds (launch gaps "
                            "included)" % (cfg.L, cfg.E, T))}


def max_over_ranks(v, world, torch):
    """The largest of the ranks' values (the job's time is its slowest rank's): an all-reduce
    on the process group, on the GPU under NCCL and on the host under gloo."""
    if world <= 1:
        return v
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def h2d_bandwidth(torch, nbytes=1 << 30, reps=3):
    """Measured host->device copy bandwidth of this machine's CPU-GPU link (pinned source)."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9)
    del h, d
    return best


def batch_result(cfg, T, steps, ms, st, world, peaks, link_gbs):
    q, hits = sum(st["queries"]), sum(st["hits"])
    bytes_per_step = q * cfg.expert_bytes / steps
    miss_bytes_per_step = st["h2d_bytes"] / steps
    tps = T * steps / (ms / 1e3) * world
    roof8 = T / (bytes_per_step / 8e12)
    roofm = T / (bytes_per_step / (peaks["hbm_gbs"] * 1e9))
    # attainable with the misses crossing the CPU-GPU link and the hits read from HBM
    t_attain = miss_bytes_per_step / (link_gbs * 1e9) + (bytes_per_step - miss_bytes_per_step) / (peaks["hbm_gbs"] * 1e9)
    attain = T / t_attain if t_attain > 0 else None
    return {"tokens_per_s": tps, "ms_per_step": ms / steps, "steps": steps,
            "hit_rate": hits / q if q else None,
            "route_hit_rate": st["route_hits"] / st["route_queries"] if st["route_queries"] else None,
            "expert_bytes_per_step": bytes_per_step, "miss_bytes_per_step": miss_bytes_per_step,
            "hbm_roofline_tokens_per_s_8tbs": roof8, "frac_of_8tbs_roofline": tps / world / roof8,
            "frac_of_measured_hbm_roofline": tps / world / roofm,
            "link_aware_attainable_tokens_per_s": attain,
            "frac_of_link_aware_attainable": (tps / world / attain) if attain else None}


def run_prefill(torch, peaks, steps=10, warmup=3):
    """Qwen-shaped prefill layer (bf16 x, 128 resident 4-bit experts, top-8): router + grouped
    GEMM (tcgen05) + combine, and the two GEMM kernels alone (events around them)."""
    from routed_expert_ffn_gemv_gb300 import _lib as L, synth
    from routed_expert_ffn_gemv_gb300.workload import PinnedImages, slot_stride
    cfg = synth.config(4)
    imgs = PinnedImages(cfg, [0], range(cfg.E))
    pool = imgs.buf.cuda()
    stride = slot_stride(cfg)
    wr = torch.from_numpy(synth.router_weights(cfg, 0).view(np.int16)).cuda()
    b = torch.from_numpy(synth.router_bias(cfg, 0)).cuda()
    out = {}
    for T in cfg.tokens:
        x = torch.from_numpy(synth.tokens_x(cfg, 0, T).view(np.int16)).cuda()
        ids = torch.empty((T, cfg.k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, cfg.k), dtype=torch.float32, device="cuda")
        ws_bytes = L.moe_expert_ffn_workspace(T, cfg.H, cfg.F, cfg.qtype, 1, cfg.E, cfg.k)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        partial = torch.empty((T, cfg.k, cfg.H), dtype=torch.float32, device="cuda")
        y = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")

        def layer():
            L.moe_router_topk(x, 1, T, cfg.H, wr, b, cfg.E, cfg.k, ids, w)
            L.moe_expert_ffn(x, 1, T, cfg.H, cfg.F, cfg.qtype, cfg.E, cfg.k, ids, w, None, cfg.E, pool, stride,
                             None, 0, partial, ws, ws_bytes)
            L.moe_combine(partial, T, cfg.k, cfg.H, None, y)
        for _ in range(warmup):
            layer()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            layer()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        # the FFN alone (route + gather + two tcgen05 GEMMs)
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record()
        for _ in range(steps):
            L.moe_expert_ffn(x, 1, T, cfg.H, cfg.F, cfg.qtype, cfg.E, cfg.k, ids, w, None, cfg.E, pool, stride,
                             None, 0, partial, ws, ws_bytes)
        f1.record()
        torch.cuda.synchronize()
        ffn_ms = f0.elapsed_time(f1) / steps
        flops = T * cfg.k * 6.0 * cfg.H * cfg.F
        tflops = flops / (ffn_ms / 1e3) / 1e12
        out[str(T)] = {"layer_ms": ms, "tokens_per_s": T / (ms / 1e3), "ffn_ms": ffn_ms,
                       "ffn_tflops": tflops, "frac_of_dense_peak": tflops / peaks["bf16_tflops"],
                       "peak": "measured dense bf16 burst (fp16 tcgen05 runs at the same rate)",
                       "operands": "fp16 (bf16 x exact in fp16), fp32 accumulate"}
    return out


def flat_prefill(pf, peaks):
    """The prefill results as flat scalars (t<T>_<field>)."""
    out = {"peak_tflops": peaks["bf16_tflops"], "peak": "measured dense bf16 burst (fp16 tcgen05 runs at "
           "the same rate)", "operands": "fp16 (bf16 x exact in fp16), fp32 accumulate"}
    for T, r in pf.items():
        for k, v in r.items():
            if isinstance(v, (int, float)):
                out[f"t{T}_{k}"] = v
    return out


def summary_lines(line):
    """A compact human-readable table of the run (printed to stderr)."""
    rows = [f"headline {line['config']['workload']}: {line['value']:.1f} tok/s "
            f"({line['ms_per_step']:.3f} ms/step), e2e {line['e2e']['value']:.1f} tok/s"]
    r = line["roofline"]
    rows.append(f"gate/up GEMV {r['achieved']:.0f} GB/s = {r['frac']:.3f} of measured HBM; down "
                f"{r['down_frac']:.3f}; layer chain {r['layer_chain_frac']:.3f}")
    for name, e in line.get("configs", {}).items():
        rows.append(f"{name}: {e['tokens_per_s']:.1f} tok/s ({e['frac_of_8tbs_roofline']:.3f} of 8 TB/s), "
                    f"hit {e.get('hit_rate') or 0:.3f} (from cold {e.get('from_cold_hit_rate') or 0:.3f}); "
                    f"resident {e['resident_tokens_per_s']:.1f} tok/s "
                    f"({e['resident_frac_of_8tbs_roofline']:.3f} of 8 TB/s); "
                    f"oracle {e.get('cpu_baseline', {}).get('value', float('nan')):.2f} tok/s")
    for name, e in line.get("policies_granite_b8", {}).items():
        rows.append(f"policy {name}: {e['tokens_per_s']:.1f} tok/s, hit {e.get('hit_rate') or 0:.3f}, "
                    f"{e['routes_per_step']:.0f} routes/step, {e['miss_bytes_per_step'] / 1e6:.0f} MB from host/step")
    for name, e in line.get("batch_growth_qwen3", {}).items():
        rows.append(f"qwen3 batch {name[1:]}: {e['tokens_per_s']:.1f} tok/s, hit {e.get('hit_rate') or 0:.3f}")
    pf = line.get("prefill", {})
    for T in ("512", "4096"):
        if f"t{T}_ffn_ms" in pf:
            rows.append(f"prefill {T}: FFN {pf[f't{T}_ffn_ms']:.3f} ms, {pf[f't{T}_ffn_tflops']:.1f} TFLOP/s "
                        f"= {pf[f't{T}_frac_of_dense_peak']:.3f} of dense peak")
    return rows


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
    T = args.batch
    max_T = max(max(cfg.tokens), T)
    link_gbs = h2d_bandwidth(torch)
    # the headline stack: device-managed pool, graph replay, cross-layer prefetch of depth 1
    # (outputs identical to the plain pool; the fills of the next layer's misses start while
    # this layer computes)
    dev_stack = Stack(cfg, max_T=max_T, device_managed=True, use_graph=True, prefetch_depth=HEADLINE_PREFETCH)
    stream = torch.cuda.Stream()
    inputs = [torch.from_numpy(synth.tokens_x(cfg, 3 + s, T)).cuda() for s in range(64)]

    clocks = ClockSampler(local)
    # the headline: W warm-up steps, then exactly K timed steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ms, prof, st = time_steps(dev_stack, inputs, T, args.steps, args.warmup, torch, stream)
    ms = max_over_ranks(ms, world, torch)
    r = batch_result(cfg, T, args.steps, ms, st, world, peaks, link_gbs)
    r["kernel_launches_per_step"] = prof["kernel_launches"] / args.steps
    if args.lite:
        clocks.stop()
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": r["tokens_per_s"], "unit": "tokens/s",
                              "lite": True, "batch": T, "result": r}), flush=True)
        dev_stack.close()
        return 0

    # per-kernel breakdown of the device-managed step (eager launches, events around every kernel)
    dev_stack.set_profile(2)
    bsteps = max(20, args.steps // 4)
    _, bprof, bst = time_steps(dev_stack, inputs, T, bsteps, 3, torch, stream)
    breakdown = {k + "_per_step": bprof[k] / bsteps for k in
                 ("router_ms", "permute_ms", "gateup_ms", "down_ms", "combine_ms")}
    breakdown["steps"] = bsteps
    breakdown["note"] = ("device-managed pool, eager launches with events around every kernel; the "
                         "gate/up and down kernels also read missed experts over the CPU-GPU link"
                         + ("; the GEMVs run as one fused launch, all counted under gateup_ms"
                            if L.moe_get_decode_fused() else ""))
    dev_stack.set_profile(0)

    # host-managed pool (moe_cache_ensure + copy-engine uploads)
    host_stack = Stack(cfg, max_T=max_T, profile=1, images=dev_stack.images)
    hsteps = max(20, args.steps // 2)
    hms, hprof, hst = time_steps(host_stack, inputs, T, hsteps, args.warmup, torch, stream)
    hms = max_over_ranks(hms, world, torch)
    host_res = batch_result(cfg, T, hsteps, hms, hst, world, peaks, link_gbs)
    host_res["host_wait_ms_per_step"] = hprof["host_wait_ms"] / hsteps
    host_res["kernel_launches_per_step"] = hprof["kernel_launches"] / hsteps
    host_stack.close()

    # end to end through the public API: pinned host input -> decode -> pinned host output
    xh = [torch.from_numpy(synth.tokens_x(cfg, 900 + s, T)).pin_memory() for s in range(8)]
    yh = torch.empty((T, cfg.H), dtype=torch.float32).pin_memory()
    xd = torch.empty((T, cfg.H), dtype=torch.float32, device="cuda")
    yd = torch.empty_like(xd)
    e2e_steps = max(20, args.steps // 2)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            xd.copy_(xh[i % 8], non_blocking=True)
            dev_stack.decode(xd, yd, stream=stream)
            yh.copy_(yd, non_blocking=True)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(e2e_steps):
            xd.copy_(xh[i % 8], non_blocking=True)
            dev_stack.decode(xd, yd, stream=stream)
            yh.copy_(yd, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, torch)
    e2e_tps = T * e2e_steps / (e2e_ms / 1e3) * world

    # every decode configuration at the metric's batch sizes (256 steps from a cold pool each)
    configs = {}
    cpu_budget = 0.0 if args.no_cpu else 4.0
    # (the plain LRU pool, as on the pages; the headline's images are shared)
    plain = Stack(cfg, max_T=max_T, device_managed=True, use_graph=True, images=dev_stack.images)
    dev_stack.close()
    for ci, Ts, stk in ((1, (1, 4, 8), plain), (2, (1,), None), (3, (1, 32), None)):
        if args.configs is not None and ci not in args.configs:
            if stk is not None:
                stk.close()
            continue
        res = run_config(ci, Ts, torch, stream, peaks, link_gbs, args.warmup, total=args.config_steps,
                         stack=stk, cpu_budget_s=cpu_budget, world=world, rank=rank)
        short = {1: "granite", 2: "qwen3", 3: "deepseek"}[ci]
        for Tb, e in res.items():
            configs[f"{short}_b{Tb}"] = e

    # pool policy variants, and batch growth on the Qwen-shaped stack (the pages' model)
    policies = run_policies(torch, stream, peaks, link_gbs, args.warmup) if not args.lite else {}
    growth = {}
    if args.configs is None or 2 in args.configs:
        g = run_config(2, (2, 4, 8, 16, 32), torch, stream, peaks, link_gbs, args.warmup, total=64,
                       cpu_budget_s=0.0, world=world, rank=rank, resident=False)
        growth = {f"t{Tb}": {k: v for k, v in e.items() if k in (
            "tokens_per_s", "ms_per_step", "hit_rate", "route_hit_rate", "hit_rate_le8", "hit_rate_9to32",
            "miss_bytes_per_step", "expert_bytes_per_step", "frac_of_8tbs_roofline")} for Tb, e in g.items()}
        if "qwen3_b1" in configs:
            growth["t1"] = {k: configs["qwen3_b1"][k] for k in growth["t2"] if k in configs["qwen3_b1"]}
    prefill = run_prefill(torch, peaks)
    gv = gemv_roofline(cfg, T, torch, stream, steps=20, warmup=3)
    clk = clocks.stop()

    roofline = gemv_roofline_block(gv, cfg, T, peaks)
    if rank == 0:
        cb = cpu_baseline(cfg, T) if world == 1 and not args.no_cpu else None
        line = {"metric": METRIC, "value": r["tokens_per_s"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic (seeded q8_0 / 4-bit experts, N(0,1) activations; no datasets or trained weights)",
                "config": workload_config(cfg, T), "impl": "gb300",
                "mode": "device-managed pool, whole step replayed as a CUDA graph, cross-layer speculative "
                        "prefetch of depth %d (the real plans' hits include prefetched experts; the plain "
                        "LRU pool is policies_granite_b8.lru_device and configs.granite_b8)" % HEADLINE_PREFETCH,
                "hit_rate": r["hit_rate"], "frac_of_8tbs_roofline": r["frac_of_8tbs_roofline"],
                "frac_of_measured_hbm_roofline": r["frac_of_measured_hbm_roofline"],
                "h2d_link_gbs_measured": link_gbs,
                "frac_of_link_aware_attainable": r["frac_of_link_aware_attainable"],
                "headline": r, "host_managed": host_res, "breakdown": breakdown,
                "cpu_baseline": cb,
                "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": T * cfg.H * 4,
                        "d2h_bytes_per_step": T * cfg.H * 4, "steps": e2e_steps},
                "gpu_launches": int(prof["kernel_launches"]),
                "clocks": clk, "prefill": flat_prefill(prefill, peaks), "roofline": roofline,
                "policies_granite_b8": policies, "batch_growth_qwen3": growth,
                "configs": configs}
        print(json.dumps(line), flush=True)
        for row in summary_lines(line):
            print(row, file=sys.stderr)
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
                    help="only the device-managed timed loop at --batch (the ncu target)")
    ap.add_argument("--configs", type=lambda v: [int(c) for c in v.split(",")], default=None,
                    help="decode configurations of the configs block (default 1,2,3)")
    ap.add_argument("--config-steps", type=int, default=256,
                    help="decode steps per configuration entry, from a cold pool (warm-up included)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU samples")
    ap.add_argument("--only", choices=["host", "gemv", "prefill"], default=None,
                    help="profiling targets: 'host' = host-managed pool loop at --batch, 'gemv' = the "
                         "decode GEMVs on an HBM-resident stack at --batch, 'prefill' = the prefill "
                         "layer at 512 and 4096 tokens")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.only:
        return run_only(args)
    return run_gpu(args, world, rank, local)


def run_only(args):
    """Short single-purpose runs used as ncu targets (one JSON line, no headline)."""
    import torch
    torch.cuda.set_device(0)
    from routed_expert_ffn_gemv_gb300 import _lib as L, synth
    from routed_expert_ffn_gemv_gb300.workload import Stack
    L.load()
    peaks = load_peaks()
    if args.only == "prefill":
        print(json.dumps({"only": "prefill", "prefill": run_prefill(torch, peaks, steps=args.steps,
                                                                   warmup=args.warmup)}), flush=True)
        return 0
    cfg = synth.config(CONFIG_INDEX)
    T = args.batch
    if args.only == "gemv":
        gv = gemv_roofline(cfg, T, torch, torch.cuda.Stream(), steps=args.steps, warmup=args.warmup)
        gv.update({"only": "gemv", "batch": T,
                   "roofline": gemv_roofline_block(gv, cfg, T, peaks)})
        print(json.dumps(gv), flush=True)
        return 0
    stack = Stack(cfg, max_T=T, profile=1)
    xs = [torch.from_numpy(synth.tokens_x(cfg, 3 + s, T)).cuda() for s in range(16)]
    ms, prof, st = time_steps(stack, xs, T, args.steps, args.warmup, torch, torch.cuda.Stream())
    gl = max(1, prof["gateup_launches"])
    print(json.dumps({"only": "host", "batch": T, "ms_per_step": ms / args.steps,
                      "gateup_ms_per_launch": prof["gateup_ms"] / gl,
                      "gateup_bytes_per_launch": prof["gateup_bytes"] / gl,
                      "gateup_gbs": prof["gateup_bytes"] / max(1e-9, prof["gateup_ms"] / 1e3) / 1e9}),
          flush=True)
    stack.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
