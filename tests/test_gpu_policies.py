"""Slot-pool policy variants on the GPU, against the LRU simulator's model of each.

* Frequency admission (page 3, tiered MoE scheduling note, section "2.2 第二层专家缓存层":
  an expert moves into VRAM once its access count passes a threshold): host-managed pools
  and the device-managed plan kernel; a bypassed miss gets no slot and is read from its
  pinned host image.
* LRU window (page 1, section "4.3 运行时配置bat脚本里的魔鬼参数", --moe-lru-window: an
  expert unused for W tokens is unloaded): host-managed pools.
Slots, bypass decisions and statistics are compared bit-exact with oracle/lru_sim.py; a
policy never changes values, so stacks with a policy give bit-identical outputs to the
plain-LRU stack.
"""
import ctypes

import numpy as np
import pytest

from oracle.lru_sim import LRUSim
from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def dev():
    return torch.device("cuda", 0)


class Pool:
    """A slot pool over pinned images of a small configuration, with a policy."""

    def __init__(self, cfg, n_layers, n_slots, device_managed, admit_after=0, lru_window=0):
        self.cfg = cfg
        self.stride = (L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F) + 255) // 256 * 256
        self.img_bytes = L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F)
        self.host = torch.empty(n_layers * cfg.E * self.stride, dtype=torch.uint8, pin_memory=True)
        for l in range(n_layers):
            for e in range(cfg.E):
                g, u, d = synth.expert_weights(cfg, l, e)
                L.moe_pack_expert(cfg.qtype, cfg.H, cfg.F, g.ctypes.data, u.ctypes.data, d.ctypes.data,
                                  self.ptr(l, e))
        self.pool = torch.zeros(n_slots * self.stride, dtype=torch.uint8, device=dev())
        self.cs = torch.cuda.Stream()
        self.imgs = (ctypes.c_void_p * (n_layers * cfg.E))(
            *[self.ptr(l, e) for l in range(n_layers) for e in range(cfg.E)])
        sb = L.moe_cache_state_bytes(n_layers, cfg.E, n_slots) if device_managed else 0
        self.state = torch.empty(max(sb, 1), dtype=torch.uint8, device=dev())
        desc = L.CacheDesc(qtype=cfg.qtype, H=cfg.H, F=cfg.F, n_layers=n_layers, n_experts=cfg.E,
                           first_layer=0, n_slots=n_slots, slot_bytes=self.stride,
                           device_pool=self.pool.data_ptr(),
                           host_images=ctypes.cast(self.imgs, ctypes.POINTER(ctypes.c_void_p)),
                           copy_stream=self.cs.cuda_stream, device_managed=int(device_managed),
                           device_state=self.state.data_ptr() if device_managed else None,
                           device_state_bytes=sb, admit_after=admit_after, lru_window=lru_window)
        self.cache = L.moe_cache_create(desc)
        self.table = torch.empty(cfg.E, dtype=torch.int32, device=dev())
        self.fill = torch.empty(cfg.E, dtype=torch.int64, device=dev())

    def ptr(self, l, e):
        return self.host.data_ptr() + (l * self.cfg.E + e) * self.stride


def _requests(rng, E, n_layers, steps):
    """Decode-like traffic: every layer of a step in order, 1-4 tokens, top-2 with a skew."""
    p = 1.0 / np.arange(1, E + 1)
    p /= p.sum()
    for step in range(steps):
        T = int(rng.integers(1, 5))
        for layer in range(n_layers):
            yield step, layer, np.stack([rng.choice(E, size=2, replace=False, p=p) for _ in range(T)]).astype(np.int32)


# (slot counts chosen with the simulator so that each trace also has LRU evictions)
@pytest.mark.parametrize("admit_after,lru_window,n_slots", [(3, 0, 12), (1, 4, 20), (2, 3, 16)])
def test_host_pool_policies_match_simulator(admit_after, lru_window, n_slots):
    cfg = synth.small_config(0, H=64, F=64, E=16, k=2, seed_cfg=840)
    n_layers = 3
    fx = Pool(cfg, n_layers, n_slots, False, admit_after, lru_window)
    sim = LRUSim(n_slots, admit_after=max(1, admit_after), window=lru_window, first_layer=0)
    host_view = fx.host.numpy()
    for step, layer, ids in _requests(np.random.default_rng(9), cfg.E, n_layers, 40):
        slots = np.empty(ids.size, dtype=np.int32)
        mask = np.zeros(cfg.E, dtype=np.uint8)
        n_miss = L.moe_cache_ensure(fx.cache, layer, ids.ctypes.data, ids.shape[0], ids.shape[1],
                                    slots.ctypes.data, mask.ctypes.data, fx.table)
        res, hit_ids, miss_ids = sim.ensure(layer, ids.reshape(-1), n_tokens=ids.shape[0])
        uploaded = [e for e in miss_ids if res[e] >= 0]
        assert n_miss == len(uploaded), (step, layer)
        assert sorted(np.nonzero(mask)[0].tolist()) == uploaded
        for i, e in enumerate(ids.reshape(-1)):
            assert slots[i] == res[int(e)], (step, layer, e)
        L.moe_cache_wait_uploads(fx.cache)
        L.moe_cache_release(fx.cache)
        torch.cuda.synchronize()
        pool = fx.pool.cpu().numpy()
        for e, s in res.items():
            if s >= 0:
                off = (layer * cfg.E + e) * fx.stride
                assert np.array_equal(pool[s * fx.stride: s * fx.stride + fx.img_bytes],
                                      host_view[off: off + fx.img_bytes])
    for layer in range(n_layers):
        for e in range(cfg.E):
            assert L.moe_cache_lookup(fx.cache, layer, e) == sim.where.get((layer, e), -1)
    st = L.moe_cache_stats_get(fx.cache)
    assert sum(st["hits"]) == sim.hits and sum(st["misses"]) == sim.misses
    assert st["evictions"] == sim.evictions and st["bypassed"] == sim.bypassed
    assert st["window_evictions"] == sim.window_evictions
    assert st["h2d_bytes"] == sim.misses * fx.img_bytes
    assert (sim.bypassed > 0) == (admit_after > 1) and (sim.window_evictions > 0) == (lru_window > 0)
    assert sim.evictions > 0
    L.moe_cache_destroy(fx.cache)


def test_device_plan_admission_matches_simulator():
    cfg = synth.small_config(0, H=64, F=64, E=16, k=2, seed_cfg=841)
    n_layers, n_slots = 3, 10
    fx = Pool(cfg, n_layers, n_slots, True, admit_after=3)
    sim = LRUSim(n_slots, admit_after=3)
    for step, layer, ids in _requests(np.random.default_rng(10), cfg.E, n_layers, 40):
        ids_d = torch.from_numpy(ids).to(dev())
        L.moe_cache_plan(fx.cache, layer, ids_d, ids.shape[0], ids.shape[1], fx.table, fx.fill)
        res, hit_ids, miss_ids = sim.ensure(layer, ids.reshape(-1), n_tokens=ids.shape[0])
        table = fx.table.cpu().numpy()
        fill = fx.fill.cpu().numpy().astype(np.uint64)
        for e in range(cfg.E):
            if e in res:
                assert table[e] == res[e], (step, layer, e)
            expect = fx.ptr(layer, e) if e in miss_ids else 0   # admitted or bypassed: read host
            assert int(fill[e]) == expect, (step, layer, e)
    assert L.moe_device_status(clear=True) == 0
    st = L.moe_cache_stats_get(fx.cache)
    assert sum(st["hits"]) == sim.hits and sum(st["misses"]) == sim.misses
    assert st["evictions"] == sim.evictions and st["bypassed"] == sim.bypassed > 0
    L.moe_cache_destroy(fx.cache)


def test_device_managed_window_is_unsupported():
    cfg = synth.small_config(0, H=32, F=32, E=4, k=1, seed_cfg=842)
    with pytest.raises(L.MoeError) as ei:
        Pool(cfg, 1, 2, True, lru_window=4)
    assert ei.value.status == L.MOE_ERR_UNSUPPORTED


def _stack(*a, **kw):
    from routed_expert_ffn_gemv_gb300.workload import Stack
    return Stack(*a, **kw)


@pytest.mark.parametrize("mode", ["device_admit", "host_admit_window"])
def test_policy_stack_outputs_equal_plain_lru_and_pools_follow_simulator(mode):
    """The Granite-shaped stack (24 layers, 384 slots) for 12 batch-8 steps: the policy
    stack's outputs are bit-identical to the plain stack's, and its pool ends in the state,
    with the statistics, the simulator predicts for the same routing."""
    cfg = synth.config(1)
    plain = _stack(cfg, max_T=8)
    if mode == "device_admit":
        pol = _stack(cfg, max_T=8, device_managed=True, use_graph=True, images=plain.images, admit_after=2)
        sim = LRUSim(cfg.groups[0].n_slots, admit_after=2)
    else:
        pol = _stack(cfg, max_T=8, images=plain.images, admit_after=2, lru_window=3)
        sim = LRUSim(cfg.groups[0].n_slots, admit_after=2, window=3, first_layer=0)
    for step in range(12):
        x = torch.from_numpy(synth.tokens_x(cfg, 600 + step, 8)).to(dev())
        ya, yb = torch.empty_like(x), torch.empty_like(x)
        ids = np.empty((cfg.L, 8, cfg.k), dtype=np.int32)
        plain.decode(x, ya, ids_out=ids)
        pol.decode(x, yb)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), step
        for layer in range(cfg.L):
            sim.ensure(layer, ids[layer].reshape(-1), n_tokens=8)
    assert L.moe_device_status(clear=True) == 0
    st = pol.cache_stats()[0]
    assert sum(st["hits"]) == sim.hits and sum(st["misses"]) == sim.misses
    assert st["evictions"] == sim.evictions and st["bypassed"] == sim.bypassed
    assert st["window_evictions"] == sim.window_evictions
    c = pol.caches[0]
    for layer in range(cfg.L):
        for e in range(cfg.E):
            assert L.moe_cache_lookup(c, layer, e) == sim.where.get((layer, e), -1)
    pol.close()
    plain.close()


def test_load_threshold_stack_layers_match_oracle():
    """Routes whose weight is below 0.05 are dropped (page 1, section 4.3): the Granite-shaped
    stack (device-managed pool) layer by layer on its own hidden state for 3 batch-8 steps.
    The kept routes equal the oracle's (routes whose oracle weight is within 1e-5 of the
    threshold, and near-tie tokens, may go either way), the layer outputs equal the oracle's
    thresholded layer within 2e-3 (evaluated on the GPU's kept routes for undecided tokens),
    and the pool follows the simulator fed the kept routes."""
    import oracle
    from tests.gpu_helpers import GAP, TOL, layer_oracle, rel_err
    th = 0.05
    cfg = synth.config(1)
    st = _stack(cfg, max_T=8, device_managed=True, load_threshold=th)
    sim = LRUSim(cfg.groups[0].n_slots)
    dropped = kept = 0
    for step in range(3):
        h = torch.from_numpy(synth.tokens_x(cfg, 700 + step, 8)).to(dev())
        for layer in range(cfg.L):
            out = torch.empty_like(h)
            ids = np.empty((8, cfg.k), dtype=np.int32)
            w = np.empty((8, cfg.k), dtype=np.float32)
            st.layer(layer, h, out, ids, w)
            torch.cuda.synchronize()
            h64 = h.cpu().numpy().astype(np.float64)
            x64 = oracle.rmsnorm(h64)
            full = layer_oracle(cfg, layer, x64)          # no threshold: the top-k and its weights
            ref = np.zeros((8, cfg.H))
            undecided = []
            for t in range(8):
                l = full.logits[t]
                order = np.lexsort((np.arange(l.size), -l))
                near_tie = l[order[cfg.k - 1]] - l[order[cfg.k]] < GAP
                sure = {int(e) for e, wt in zip(full.ids[t], full.weights[t]) if wt >= th + 1e-5}
                maybe = {int(e) for e, wt in zip(full.ids[t], full.weights[t]) if abs(wt - th) <= 1e-5}
                got = {int(e) for e in ids[t] if e >= 0}
                assert all((e >= 0) == (wt > 0) for e, wt in zip(ids[t], w[t]))   # id -1 <=> weight 0
                if near_tie or maybe:
                    undecided.append(t)
                else:
                    assert got == sure, (step, layer, t, got, sure)
                dropped += int(np.sum(ids[t] < 0))
                kept += int(np.sum(ids[t] >= 0))
            decided = [t for t in range(8) if t not in undecided]
            if decided:
                ref[decided] = oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x64[decided],
                                                synth.router_weights(cfg, layer), synth.router_bias(cfg, layer),
                                                lambda e: synth.expert_weights(cfg, layer, e), load_threshold=th).y
            if undecided:  # the GPU's kept routes with the oracle's weights for them
                wt = np.zeros((len(undecided), cfg.k))
                for i, t in enumerate(undecided):
                    for j, e in enumerate(ids[t]):
                        if e >= 0:
                            pos = np.nonzero(full.ids[t] == e)[0]
                            wt[i, j] = full.weights[t, pos[0]] if pos.size else 0.0
                ref[undecided] = oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x64[undecided],
                                                  synth.router_weights(cfg, layer), synth.router_bias(cfg, layer),
                                                  lambda e: synth.expert_weights(cfg, layer, e),
                                                  route_override=(ids[undecided], wt)).y
            err = rel_err(out.cpu().numpy().astype(np.float64) - h64, ref)
            assert err.max() <= TOL, (step, layer, err)
            res, _, _ = sim.ensure(layer, ids[ids >= 0], n_tokens=8)
            for e, s in res.items():
                assert L.moe_cache_lookup(st.caches[0], layer, e) == s
            h = out
    assert L.moe_device_status(clear=True) == 0
    assert dropped > 0 and kept > 0
    stt = st.cache_stats()[0]
    assert sum(stt["hits"]) == sim.hits and sum(stt["misses"]) == sim.misses
    assert stt["route_queries"] == kept
    print(f"load threshold {th}: {dropped} of {dropped + kept} routes dropped")
    st.close()


@pytest.mark.parametrize("depth,admit", [(2, 1), (1, 1), (1, 2)])
def test_cross_layer_prefetch_follows_simulator_and_keeps_values(depth, admit):
    """Cross-layer speculative prefetch (page 3, sections 2.3 and 4.3, depth 1 or 2, with plain
    LRU or frequency admission) on the
    Granite-shaped stack, device-managed pool, batch 8, layer by layer for 3 steps: outputs
    bit-identical to the plain device-managed stack; the pool bit-exact against the simulator
    fed each layer's real ids and the predicted ids of the next two layers (the next layers'
    routers on this layer's normalised input, recomputed here with the same kernels); then
    the same steps as graph-replayed decode steps from an empty pool end in the same state."""
    cfg = synth.config(1)
    T = 8
    plain = _stack(cfg, max_T=T, device_managed=True)
    pf = _stack(cfg, max_T=T, device_managed=True, images=plain.images, prefetch_depth=depth, admit_after=admit)
    sim = LRUSim(cfg.groups[0].n_slots, admit_after=admit)
    xn = torch.empty((T, cfg.H), dtype=torch.float32, device=dev())
    pid = torch.empty((T, cfg.k), dtype=torch.int32, device=dev())
    pw = torch.empty((T, cfg.k), dtype=torch.float32, device=dev())
    finals = []
    for step in range(3):
        h = torch.from_numpy(synth.tokens_x(cfg, 800 + step, T)).to(dev())
        for layer in range(cfg.L):
            ya, yb = torch.empty_like(h), torch.empty_like(h)
            ids = np.empty((T, cfg.k), dtype=np.int32)
            plain.layer(layer, h, ya)
            pf.layer(layer, h, yb, ids)
            torch.cuda.synchronize()
            assert torch.equal(ya, yb), (step, layer)
            sim.ensure(layer, ids.reshape(-1), n_tokens=T)
            L.moe_combine_rmsnorm(None, T, 0, cfg.H, h, None, xn)   # the stack's pre-norm of h
            for dd in range(1, depth + 1):
                l2 = layer + dd
                if l2 >= cfg.L:
                    break
                L.moe_router_topk(xn, 0, T, cfg.H, pf.w_router[l2], pf.bias[l2], cfg.E, cfg.k, pid, pw)
                torch.cuda.synchronize()
                sim.prefetch(l2, pid.cpu().numpy().reshape(-1))
            c = pf.caches[0]
            for e in set(ids.reshape(-1).tolist()):
                assert L.moe_cache_lookup(c, layer, e) == sim.where.get((layer, e), -1), (step, layer, e)
            h = yb
        finals.append(h.clone())
    assert L.moe_device_status(clear=True) == 0
    st = pf.cache_stats()[0]
    assert sum(st["hits"]) == sim.hits and sum(st["misses"]) == sim.misses and st["evictions"] == sim.evictions
    assert (st["prefetch_queries"], st["prefetch_hits"], st["prefetch_fills"], st["prefetch_aborts"]) == \
        (sim.pf_queries, sim.pf_hits, sim.pf_fills, sim.pf_aborts)
    assert sim.pf_fills > 0
    for layer in range(cfg.L):
        for e in range(cfg.E):
            assert L.moe_cache_lookup(pf.caches[0], layer, e) == sim.where.get((layer, e), -1)
    print(f"prefetch: {sim.pf_queries} predicted, {sim.pf_hits} already resident, {sim.pf_fills} copied, "
          f"{sim.pf_aborts} abandoned; real hits {sim.hits} of {sim.hits + sim.misses}")
    # the same steps as decode steps (eager first, then graph replay) from an empty pool
    g = _stack(cfg, max_T=T, device_managed=True, use_graph=True, images=plain.images, prefetch_depth=depth,
               admit_after=admit)
    y = torch.empty((T, cfg.H), dtype=torch.float32, device=dev())
    for step in range(3):
        g.decode(torch.from_numpy(synth.tokens_x(cfg, 800 + step, T)).to(dev()), y)
        torch.cuda.synchronize()
        assert torch.equal(y, finals[step]), step
    assert g.cache_stats() == pf.cache_stats()
    assert L.moe_device_status(clear=True) == 0
    for s_ in (g, pf, plain):
        s_.close()
