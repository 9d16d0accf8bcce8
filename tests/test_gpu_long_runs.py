"""Whole-length decode runs at full size, in the headline pool mode.

Each configuration's decode workload runs its full 256 steps from an empty pool, so that
the slot pools reach steady-state eviction (the Qwen-shaped groups hold 1,834 slots each,
page 4 "MoE缓存到底缓存了什么": one LRU per type/shape group shared by its layers):

A. device-managed pools (the LRU on the GPU, missed experts read over the CPU-GPU link and
   written into their slots by the GEMVs), the layers run one by one through
   moe_stack_layer on the GPU's own hidden state.  At EVERY layer of EVERY step:
     * the routed ids equal the oracle's top-k of the oracle router on the layer's input
       (bit-exact; tokens whose k-th / (k+1)-th margin is below 1e-5 excluded);
     * the slot of every requested expert equals the LRU simulator's.
   On a sample of (step, layer) pairs the layer's MoE output is compared with the fp64
   oracle on the same input (2e-3 per token, normwise).
B. the same steps through moe_stack_decode replayed as a CUDA graph, from an empty pool:
   every step's output is bit-identical to run A's and the pool statistics are equal.
C. (pool configurations 2 and 3) the host-managed pool (LRU on the host, copy-engine
   uploads): again bit-identical outputs and equal statistics.
At the end the whole device table equals the simulator's, and evictions did happen.
"""
import concurrent.futures as cf

import numpy as np
import pytest

import oracle
from oracle.lru_sim import LRUSim
from tests.gpu_helpers import TOL, ids_match, rel_err
from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]

STEPS = 256


def dev():
    return torch.device("cuda", 0)


def _experts(cfg, layer, ids):
    """Canonical blocks of the given experts of a layer (generated in parallel threads)."""
    ids = sorted(set(int(e) for e in ids))
    with cf.ThreadPoolExecutor(max_workers=16) as ex:
        blocks = list(ex.map(lambda e: synth.expert_weights(cfg, layer, e), ids))
    return dict(zip(ids, blocks))


def _oracle_layer(cfg, layer, x64, wr, b, route_override=None):
    """The oracle layer on x64; the experts it needs are generated first (ids of the oracle's
    own routing, or of the override)."""
    if route_override is not None:
        need = route_override[0].reshape(-1)
    else:
        need = oracle.topk_softmax(oracle.router_logits(x64, wr, b), cfg.k)[0].reshape(-1)
    ex = _experts(cfg, layer, need)
    shared = list(_experts(cfg, layer, range(cfg.E, cfg.E + cfg.n_shared)).values())
    return oracle.moe_layer(cfg.qtype, cfg.H, cfg.F, cfg.k, x64, wr, b, ex.__getitem__, shared=shared,
                            route_override=route_override)


_IMAGES = {}


def _images(cfg):
    """The pinned expert images of one configuration, kept for the next test of the same one
    (the parametrisations below are grouped by configuration)."""
    from routed_expert_ffn_gemv_gb300.workload import PinnedImages
    if cfg.index not in _IMAGES:
        _IMAGES.clear()
        _IMAGES[cfg.index] = PinnedImages(cfg, range(cfg.L), range(cfg.E))
    return _IMAGES[cfg.index]


class Run:
    def __init__(self, cfg, T):
        self.cfg, self.T = cfg, T
        self.images = _images(cfg)
        self.wr = [synth.router_weights(cfg, l) for l in range(cfg.L)]
        self.b = [synth.router_bias(cfg, l) for l in range(cfg.L)]
        self.xs = [synth.tokens_x(cfg, 7000 + s, T) for s in range(STEPS)]
        self.group = []
        for l in range(cfg.L):
            self.group.append(next(i for i, g in enumerate(cfg.groups)
                                   if g.first_layer <= l < g.first_layer + g.n_layers))

    def stack(self, **kw):
        from routed_expert_ffn_gemv_gb300.workload import Stack
        return Stack(self.cfg, max_T=self.T, images=self.images, **kw)


def _layer_by_layer(run, sample):
    """Run A: device-managed pools, layer by layer; returns the outputs, stats and counts."""
    cfg, T = run.cfg, run.T
    st = run.stack(device_managed=True)
    sims = [LRUSim(g.n_slots) for g in cfg.groups]
    outs, compared, excluded, worst = [], 0, 0, 0.0
    for step in range(STEPS):
        h = torch.from_numpy(run.xs[step]).to(dev())
        for layer in range(cfg.L):
            out = torch.empty_like(h)
            ids = np.empty((T, cfg.k), dtype=np.int32)
            w = np.empty((T, cfg.k), dtype=np.float32)
            st.layer(layer, h, out, ids, w)
            torch.cuda.synchronize()
            h64 = h.cpu().numpy().astype(np.float64)
            x64 = oracle.rmsnorm(h64)  # the layer's MoE input (pre-norm)
            logits = oracle.router_logits(x64, run.wr[layer], run.b[layer])
            oids, _, _ = oracle.topk_softmax(logits, cfg.k)
            m = ids_match(ids, logits, oids, cfg.k)
            assert all(v is not False for v in m), (step, layer, ids, oids)
            g = run.group[layer]
            res, _, _ = sims[g].ensure(layer, ids.reshape(-1))
            c = st.caches[g]
            for e, s in res.items():
                assert L.moe_cache_lookup(c, layer, e) == s, (step, layer, e)
            if sample(step, layer):
                near = [t for t, v in enumerate(m) if v is None]
                ref = _oracle_layer(cfg, layer, x64, run.wr[layer], run.b[layer]).y
                if near:  # the oracle on the route the GPU took, weights from the oracle logits
                    sel = np.take_along_axis(logits[near], ids[near].astype(np.int64), axis=1)
                    ww = np.exp(sel - sel.max(axis=1, keepdims=True))
                    ww /= ww.sum(axis=1, keepdims=True)
                    ref[near] = _oracle_layer(cfg, layer, x64[near], run.wr[layer], run.b[layer],
                                              route_override=(ids[near], ww)).y
                delta = out.cpu().numpy().astype(np.float64) - h64
                err = rel_err(delta, ref)
                assert err.max() <= TOL, (step, layer, err)
                worst = max(worst, float(err.max()))
                compared += T
                excluded += len(near)
            h = out
        outs.append(h.clone())
    torch.cuda.synchronize()
    assert L.moe_device_status(clear=True) == 0
    # the whole table at the end: every (layer, expert) where the simulator has it, else -1
    for gi, grp in enumerate(cfg.groups):
        c = st.caches[gi]
        for layer in range(grp.first_layer, grp.first_layer + grp.n_layers):
            for e in range(cfg.E):
                assert L.moe_cache_lookup(c, layer, e) == sims[gi].where.get((layer, e), -1), (layer, e)
    stats = st.cache_stats()
    for gi, sim in enumerate(sims):
        assert sum(stats[gi]["hits"]) == sim.hits and sum(stats[gi]["misses"]) == sim.misses
        assert stats[gi]["evictions"] == sim.evictions
    evictions = [sim.evictions for sim in sims]
    st.close()
    return outs, stats, evictions, compared, excluded, worst


def _replay(run, outs, stats, **kw):
    """Runs B / C: whole steps from an empty pool; bit-identical outputs, equal statistics."""
    st = run.stack(**kw)
    y = torch.empty((run.T, run.cfg.H), dtype=torch.float32, device=dev())
    for step in range(STEPS):
        x = torch.from_numpy(run.xs[step]).to(dev())
        st.decode(x, y)
        torch.cuda.synchronize()
        assert torch.equal(y, outs[step]), (kw, step)
    assert L.moe_device_status(clear=True) == 0
    assert st.cache_stats() == stats, kw
    st.close()


@pytest.mark.parametrize("ci,T,every,lstride", [
    (2, 1, 16, 6),    # Qwen3-30B-A3B-shaped: two 24-layer groups of 1,834 slots, batch 1
    (3, 1, 16, 6),    # DeepSeek-MoE-16B-shaped: 224 slots + 2 resident shared experts, batch 1
    (3, 32, 64, 14),  # the same at batch 32 (4 sequences x 8 tokens)
    (1, 1, 32, 6),    # Granite-shaped: 384 slots, batch 1 / 4 / 8
    (1, 4, 32, 6),
    (1, 8, 32, 6),
])
def test_full_length_decode(ci, T, every, lstride):
    cfg = synth.config(ci)
    run = Run(cfg, T)
    # outputs on every `every`-th step, at every `lstride`-th layer from an offset that moves
    sample = lambda step, layer: step % every == 0 and (layer - step // every) % lstride == 0
    outs, stats, ev, compared, excluded, worst = _layer_by_layer(run, sample)
    print(f"config {ci} T={T}: {STEPS} steps x {cfg.L} layers, evictions per group {ev}, "
          f"hits {[sum(s['hits']) for s in stats]} misses {[sum(s['misses']) for s in stats]}, "
          f"outputs compared on {compared} token-layers (worst {worst:.2e}, near ties {excluded})")
    assert all(e > 0 for e in ev), ev   # the pools reached eviction
    assert compared >= STEPS // every * (cfg.L // lstride) * T
    _replay(run, outs, stats, device_managed=True, use_graph=True)
    if ci in (2, 3):
        _replay(run, outs, stats)
