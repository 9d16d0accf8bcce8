"""Device-managed slot pools: the LRU run on the GPU (moe_cache_plan) must assign exactly the
slots the LRU simulator assigns; the fill path (moe_expert_ffn_fill) must compute the same
outputs as the oracle while writing each missed expert's image into its slot; a
device-managed stack must give bit-identical results to the host-managed one, and its
CUDA-graph replay bit-identical results to eager launches."""
import ctypes

import numpy as np
import pytest

import oracle
from oracle.lru_sim import LRUSim
from tests.gpu_helpers import TOL, rel_err
from tests.test_gpu_stack import run_steps
from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def dev():
    return torch.device("cuda", 0)


class DevicePool:
    def __init__(self, cfg, n_layers, n_slots):
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
        sb = L.moe_cache_state_bytes(n_layers, cfg.E, n_slots)
        self.state = torch.empty(sb, dtype=torch.uint8, device=dev())
        self.imgs = (ctypes.c_void_p * (n_layers * cfg.E))(
            *[self.ptr(l, e) for l in range(n_layers) for e in range(cfg.E)])
        desc = L.CacheDesc(qtype=cfg.qtype, H=cfg.H, F=cfg.F, n_layers=n_layers, n_experts=cfg.E,
                           first_layer=0, n_slots=n_slots, slot_bytes=self.stride,
                           device_pool=self.pool.data_ptr(),
                           host_images=ctypes.cast(self.imgs, ctypes.POINTER(ctypes.c_void_p)),
                           copy_stream=None, device_managed=1, device_state=self.state.data_ptr(),
                           device_state_bytes=sb)
        self.cache = L.moe_cache_create(desc)
        self.table = torch.empty(cfg.E, dtype=torch.int32, device=dev())
        self.fill = torch.empty(cfg.E, dtype=torch.int64, device=dev())

    def ptr(self, l, e):
        return self.host.data_ptr() + (l * self.cfg.E + e) * self.stride

    def plan(self, layer, ids):
        ids_d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).to(dev())
        L.moe_cache_plan(self.cache, layer, ids_d, ids.shape[0], ids.shape[1], self.table, self.fill)
        return ids_d


def test_device_plan_matches_lru_simulator():
    cfg = synth.small_config(0, H=64, F=64, E=16, k=2, seed_cfg=870)
    n_layers, n_slots = 3, 10
    fx = DevicePool(cfg, n_layers, n_slots)
    sim = LRUSim(n_slots)
    rng = np.random.default_rng(21)
    for step in range(80):
        layer = int(rng.integers(0, n_layers))
        T = int(rng.integers(1, 5))
        ids = np.stack([rng.choice(cfg.E, size=2, replace=False) for _ in range(T)]).astype(np.int32)
        fx.plan(layer, ids)
        res, hit_ids, miss_ids = sim.ensure(layer, ids.reshape(-1))
        table = fx.table.cpu().numpy()
        fill = fx.fill.cpu().numpy().astype(np.uint64)
        for e, s in res.items():
            assert table[e] == s, (step, e)
        for e in range(cfg.E):
            expect = fx.ptr(layer, e) if e in miss_ids else 0
            assert int(fill[e]) == expect, (step, e)
            if e not in res:
                assert table[e] == L.moe_cache_lookup(fx.cache, layer, e)
    st = L.moe_cache_stats_get(fx.cache)
    assert sum(st["hits"]) == sim.hits and sum(st["misses"]) == sim.misses
    assert st["evictions"] == sim.evictions
    assert L.moe_device_status(clear=True) == 0
    # reset empties the pool
    L.moe_cache_reset(fx.cache)
    assert all(L.moe_cache_lookup(fx.cache, l, e) == -1 for l in range(n_layers) for e in range(cfg.E))
    L.moe_cache_destroy(fx.cache)


def test_device_plan_capacity_is_recorded():
    cfg = synth.small_config(0, H=32, F=32, E=8, k=2, seed_cfg=871)
    fx = DevicePool(cfg, 1, 3)
    fx.plan(0, np.array([[0, 1], [2, 3]], dtype=np.int32))   # 4 distinct > 3 slots
    torch.cuda.synchronize()
    assert L.moe_device_status(clear=True) == L.MOE_ERR_CAPACITY
    assert np.all(fx.table.cpu().numpy() == -1) and np.all(fx.fill.cpu().numpy() == 0)
    L.moe_cache_destroy(fx.cache)


@pytest.mark.parametrize("qtype", [0, 1])
def test_fill_ffn_matches_oracle_and_fills_slots(qtype):
    cfg = synth.small_config(qtype, H=256, F=128, E=12, k=2, seed_cfg=872 + qtype)
    fx = DevicePool(cfg, 2, 7)
    rng = np.random.default_rng(22 + qtype)
    host = fx.host.numpy()
    for step in range(12):
        layer = step % 2
        T = int(rng.integers(1, 4))
        ids = np.stack([rng.choice(cfg.E, size=2, replace=False) for _ in range(T)]).astype(np.int32)
        w = rng.uniform(0.1, 1.0, size=(T, 2)).astype(np.float32)
        x = rng.standard_normal((T, cfg.H), dtype=np.float32)
        ids_d = fx.plan(layer, ids)
        ws_bytes = L.moe_expert_ffn_workspace(T, cfg.H, cfg.F, qtype, 0, cfg.E, 2)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev())
        partial = torch.full((T, 2, cfg.H), float("nan"), dtype=torch.float32, device=dev())
        L.moe_expert_ffn_fill(torch.from_numpy(x).to(dev()), 0, T, cfg.H, cfg.F, qtype, cfg.E, 2, ids_d,
                              torch.from_numpy(w).to(dev()), fx.table, 7, fx.pool, fx.stride, fx.fill,
                              partial, ws, ws_bytes)
        torch.cuda.synchronize()
        assert L.moe_device_status(clear=True) == 0
        got = partial.cpu().numpy()
        for t in range(T):
            for j in range(2):
                g, u, d = synth.expert_weights(cfg, layer, int(ids[t, j]))
                ref = float(w[t, j]) * oracle.expert_ffn(qtype, cfg.H, cfg.F, g, u, d, x[t].astype(np.float64))
                assert rel_err(got[t, j][None], ref[None])[0] <= TOL
        pool = fx.pool.cpu().numpy()
        table = fx.table.cpu().numpy()
        for e in set(ids.reshape(-1).tolist()):
            s = table[e]
            off = (layer * cfg.E + e) * fx.stride
            assert np.array_equal(pool[s * fx.stride: s * fx.stride + fx.img_bytes],
                                  host[off: off + fx.img_bytes]), (step, e)
    L.moe_cache_destroy(fx.cache)


@pytest.mark.parametrize("qtype,H,T,k,E", [
    (0, 256, 8, 4, 6),    # about 5 routes per expert: two virtual experts per missed expert
    (1, 512, 16, 6, 8),   # 4-bit, 12 routes per expert on average: three or four groups
    (0, 1024, 1, 2, 12),  # one token: the gate/up K split reaches its maximum
])
def test_fill_ffn_with_several_groups_per_missed_expert(qtype, H, T, k, E):
    """A missed expert routed by more than 4 routes is split into several virtual experts: all
    read the pinned host image, the first writes it through to the slot."""
    cfg = synth.small_config(qtype, H=H, F=96, E=E, k=k, seed_cfg=890 + qtype + H)
    fx = DevicePool(cfg, 1, E)
    rng = np.random.default_rng(H + T)
    host = fx.host.numpy()
    ids = np.stack([rng.choice(cfg.E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    w = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
    x = rng.standard_normal((T, cfg.H), dtype=np.float32)
    ids_d = fx.plan(0, ids)
    ws_bytes = L.moe_expert_ffn_workspace(T, cfg.H, cfg.F, qtype, 0, cfg.E, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev())
    partial = torch.full((T, k, cfg.H), float("nan"), dtype=torch.float32, device=dev())
    L.moe_expert_ffn_fill(torch.from_numpy(x).to(dev()), 0, T, cfg.H, cfg.F, qtype, cfg.E, k, ids_d,
                          torch.from_numpy(w).to(dev()), fx.table, E, fx.pool, fx.stride, fx.fill,
                          partial, ws, ws_bytes)
    torch.cuda.synchronize()
    assert L.moe_device_status(clear=True) == 0
    got = partial.cpu().numpy()
    for t in range(T):
        for j in range(k):
            g, u, d = synth.expert_weights(cfg, 0, int(ids[t, j]))
            ref = float(w[t, j]) * oracle.expert_ffn(qtype, cfg.H, cfg.F, g, u, d, x[t].astype(np.float64))
            assert rel_err(got[t, j][None], ref[None])[0] <= TOL
    pool, table = fx.pool.cpu().numpy(), fx.table.cpu().numpy()
    for e in set(ids.reshape(-1).tolist()):
        s = table[e]
        assert np.array_equal(pool[s * fx.stride: s * fx.stride + fx.img_bytes],
                              host[e * fx.stride: e * fx.stride + fx.img_bytes]), e
    L.moe_cache_destroy(fx.cache)


def _stack(*a, **kw):
    from routed_expert_ffn_gemv_gb300.workload import Stack
    return Stack(*a, **kw)


def test_device_managed_stack_teacher_forced_small():
    import dataclasses
    cfg0 = synth.small_config(0, H=256, F=128, E=24, k=2, L=4, n_shared=2, bias_a=1.0, seed_cfg=830,
                              groups=(synth.PoolGroup(0, 2, 18), synth.PoolGroup(2, 2, 16)))
    cfg = dataclasses.replace(cfg0, tokens=(1, 3, 8))
    st = _stack(cfg, max_T=8, device_managed=True)
    for T in (1, 3, 8):
        run_steps(st, cfg, T, 3, step0=20 * T)
    st.close()


def test_device_managed_stack_equals_host_managed():
    cfg = synth.config(1)
    a = _stack(cfg, max_T=8)
    b = _stack(cfg, max_T=8, device_managed=True)
    for step in range(4):
        for T in (1, 8):
            x = torch.from_numpy(synth.tokens_x(cfg, 300 + step, T)).to(dev())
            ya, yb = torch.empty_like(x), torch.empty_like(x)
            a.decode(x, ya)
            b.decode(x, yb)
            torch.cuda.synchronize()
            assert torch.equal(ya, yb), (step, T)
    assert a.cache_stats() == b.cache_stats()
    assert L.moe_device_status(clear=True) == 0
    a.close()
    b.close()


def test_graph_replay_equals_eager():
    cfg = synth.config(1)
    a = _stack(cfg, max_T=8, device_managed=True, use_graph=True)
    b = _stack(cfg, max_T=8, device_managed=True)
    for step in range(5):
        x = torch.from_numpy(synth.tokens_x(cfg, 400 + step, 8)).to(dev())
        ya, yb = torch.empty_like(x), torch.empty_like(x)
        a.decode(x, ya)
        b.decode(x, yb)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), step
    assert a.cache_stats() == b.cache_stats()
    a.close()
    b.close()
