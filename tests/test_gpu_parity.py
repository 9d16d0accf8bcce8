"""GPU parity of every hot-path step against the fp64 oracle, through the C-ABI."""
import ctypes

import numpy as np
import pytest

import oracle
from oracle.lru_sim import LRUSim
from tests.gpu_helpers import GAP, TOL, ids_match, layer_oracle, random_routes, rel_err
from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def dev():
    return torch.device("cuda", 0)


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def status_clear():
    assert L.moe_device_status(clear=True) == 0


# ------------------------------------------------------------------------------------ router

ROUTER_CASES = [
    # H, E, k, T, xtype, bias_a
    (256, 8, 2, 1, 0, 0.0),        # tiny layer shape, one token
    (1024, 32, 8, 8, 0, 1.0),      # Granite-shaped, batch 8
    (2048, 128, 8, 1, 0, 1.1),     # Qwen-shaped, batch 1
    (2048, 64, 2, 32, 0, 1.2),     # DeepSeek-shaped, batch 32
    (2048, 128, 8, 100, 1, 1.1),   # bf16 prefill tokens: 4 clusters with a ragged tail
    (96, 5, 3, 7, 0, 0.7),         # odd E, H with 12 rows per cluster CTA
    # above 32 tokens: the tiled router (32-token CTAs, 32-row chunks of W_r)
    (1024, 32, 8, 33, 0, 1.0),     # one token past the decode limit: a 1-token second tile
    (96, 5, 3, 70, 0, 0.7),        # odd E (padded expert columns), 3 chunks
    (2048, 256, 8, 64, 1, 1.0),    # E = 256: 8 experts per thread
    (64, 200, 6, 45, 0, 0.5),      # E = 200, 2 chunks
    (2048, 128, 8, 300, 0, 1.1),   # Qwen-shaped, fp32 tokens, ragged last tile
    # bf16 tokens above 32 with E a multiple of 32 (at most 128): the tensor-core router
    (1024, 64, 6, 77, 1, 1.0),     # 2 n-tiles per warp, ragged last tile
    (512, 96, 4, 40, 1, 0.8),      # 3 n-tiles per warp
    (2048, 32, 2, 520, 1, 1.2),    # 1 n-tile per warp, many tiles
]


@pytest.mark.parametrize("H,E,k,T,xtype,bias_a", ROUTER_CASES)
def test_router_topk_parity(H, E, k, T, xtype, bias_a):
    cfg = synth.small_config(0, H=H, F=32, E=E, k=k, bias_a=bias_a, seed_cfg=700 + E)
    wr = synth.router_weights(cfg, 0)
    b = synth.router_bias(cfg, 0)
    rng = np.random.default_rng(H + E + T)
    x = rng.standard_normal((T, H), dtype=np.float32)
    if xtype == 1:
        xb = synth.f32_to_bf16_bits(x)
        x_d = to_dev(xb.view(np.int16))
        x64 = oracle.x_to_double(xb, 1)
    else:
        x_d = to_dev(x)
        x64 = oracle.x_to_double(x, 0)
    ids = torch.empty((T, k), dtype=torch.int32, device=dev())
    w = torch.empty((T, k), dtype=torch.float32, device=dev())
    lg = torch.empty((T, E), dtype=torch.float32, device=dev())
    L.moe_router_topk(x_d, xtype, T, H, to_dev(wr.view(np.int16)), None if b is None else to_dev(b),
                      E, k, ids, w, lg)
    torch.cuda.synchronize()
    status_clear()
    lo = oracle.router_logits(x64, wr, b)
    io, wo, gap = oracle.topk_softmax(lo, k)
    lg_h = lg.cpu().numpy().astype(np.float64)
    # fp32 accumulation keeps the logits far inside the exclusion margin
    assert np.max(np.abs(lg_h - lo)) < 2e-6 * max(1.0, np.max(np.abs(lo)))
    m = ids_match(ids.cpu().numpy(), lo, io, k)
    assert all(v is not False for v in m), m
    cmp = [t for t, v in enumerate(m) if v]
    assert len(cmp) >= T - 1
    # softmax over the selected logits moves each weight by at most 2*w*max|dl| for logit
    # errors dl (plus a few fp32 ulps of exp and the division)
    dl = np.max(np.abs(lg_h - lo), axis=1, keepdims=True)
    tol = 2.0 * dl * wo + 4e-7
    assert np.all(np.abs(w.cpu().numpy()[cmp] - wo[cmp]) <= tol[cmp])
    assert np.allclose(w.cpu().numpy().sum(axis=1), 1.0, atol=1e-6)


# ------------------------------------------------------------------------------------ expert FFN

def make_pool(cfg, layer, experts, random_scales=False):
    stride = (L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F) + 255) // 256 * 256
    host = torch.empty(len(experts) * stride, dtype=torch.uint8, pin_memory=True)
    for i, e in enumerate(experts):
        g, u, d = synth.expert_weights(cfg, layer, e, random_scales)
        L.moe_pack_expert(cfg.qtype, cfg.H, cfg.F, g.ctypes.data, u.ctypes.data, d.ctypes.data,
                          host.data_ptr() + i * stride)
    return host.to(dev()), stride


def run_ffn(cfg, pool, stride, x_d, xtype, ids, w, subset=None, partial=None, table=None, n_slots=None):
    T, k = ids.shape
    ws_bytes = L.moe_expert_ffn_workspace(T, cfg.H, cfg.F, cfg.qtype, xtype, cfg.E, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev())
    if partial is None:
        partial = torch.full((T, k, cfg.H), float("nan"), dtype=torch.float32, device=dev())
    sub = None if subset is None else to_dev(np.asarray(subset, dtype=np.int32))
    L.moe_expert_ffn(x_d, xtype, T, cfg.H, cfg.F, cfg.qtype, cfg.E, k, to_dev(ids), to_dev(w),
                     table, n_slots or cfg.E, pool, stride, sub, 0 if subset is None else len(subset),
                     partial, ws, ws_bytes)
    torch.cuda.synchronize()
    return partial


FFN_CASES = [
    # qtype, H, F, E, k, T, random_scales, xtype
    (0, 256, 512, 8, 2, 1, False, 0),     # the tiny layer shape
    (0, 64, 96, 4, 2, 3, True, 0),        # 3 row tiles, 2 blocks per row, per-block scales
    (1, 64, 96, 4, 2, 3, True, 0),
    (0, 1024, 512, 32, 8, 8, False, 0),   # Granite-shaped, K split in 2
    (1, 2048, 768, 16, 8, 4, True, 0),    # Qwen-shaped, 4-bit
    (1, 2048, 768, 32, 8, 32, False, 0),  # Qwen-shaped at batch 32: the K split grows until the
                                          # staged activations fit beside the ring
    (0, 2048, 1408, 8, 2, 32, False, 0),  # DeepSeek-shaped at batch 32: >8 tokens per expert
    (1, 256, 160, 6, 3, 13, True, 0),     # 5 row tiles, 13 tokens
    (0, 128, 64, 4, 4, 9, True, 1),       # bf16 activations, k = E
    (1, 96, 32, 3, 1, 2, True, 0),        # one row tile, three blocks over four warps
]


@pytest.fixture(params=[True, False], ids=["fused", "separate"])
def gemv_mode(request):
    """Runs a test with the decode GEMVs as one fused launch, then as three kernels."""
    before = L.moe_get_decode_fused()
    L.moe_set_decode_fused(request.param)
    yield request.param
    L.moe_set_decode_fused(before)


@pytest.mark.parametrize("qtype,H,F,E,k,T,rs,xtype", FFN_CASES)
def test_expert_ffn_parity(qtype, H, F, E, k, T, rs, xtype, gemv_mode):
    cfg = synth.small_config(qtype, H=H, F=F, E=E, k=k, seed_cfg=800 + H + F)
    pool, stride = make_pool(cfg, 0, range(E), rs)
    rng = np.random.default_rng(T * 31 + E)
    x = rng.standard_normal((T, H), dtype=np.float32)
    if xtype == 1:
        xb = synth.f32_to_bf16_bits(x)
        x_d, x64 = to_dev(xb.view(np.int16)), oracle.x_to_double(xb, 1)
    else:
        x_d, x64 = to_dev(x), oracle.x_to_double(x, 0)
    ids, w = random_routes(rng, T, E, k)
    partial = run_ffn(cfg, pool, stride, x_d, xtype, ids, w).cpu().numpy()
    status_clear()
    worst = 0.0
    for t in range(T):
        for j in range(k):
            g, u, d = synth.expert_weights(cfg, 0, int(ids[t, j]), rs)
            ref = float(w[t, j]) * oracle.expert_ffn(qtype, H, F, g, u, d, x64[t])
            err = rel_err(partial[t, j][None], ref[None])[0]
            worst = max(worst, err)
    assert worst <= TOL, worst
    assert worst <= 1e-4, worst  # fp32 accumulation of exact products stays far below 2e-3


@pytest.mark.parametrize("qtype,H,F,E,k,T,rs,xtype", FFN_CASES)
def test_fused_and_separate_gemvs_agree_bit_for_bit(qtype, H, F, E, k, T, rs, xtype):
    """The fused launch and the three separate kernels do the same arithmetic in the same order."""
    cfg = synth.small_config(qtype, H=H, F=F, E=E, k=k, seed_cfg=900 + H + F)
    pool, stride = make_pool(cfg, 0, range(E), rs)
    rng = np.random.default_rng(T * 17 + E)
    x = rng.standard_normal((T, H), dtype=np.float32)
    x_d = to_dev(synth.f32_to_bf16_bits(x).view(np.int16)) if xtype == 1 else to_dev(x)
    ids, w = random_routes(rng, T, E, k)
    before = L.moe_get_decode_fused()
    try:
        out = {}
        for mode in (True, False):
            L.moe_set_decode_fused(mode)
            out[mode] = run_ffn(cfg, pool, stride, x_d, xtype, ids, w).cpu().numpy()
    finally:
        L.moe_set_decode_fused(before)
    status_clear()
    assert np.all(np.isfinite(out[True]))
    assert np.array_equal(out[True].view(np.uint32), out[False].view(np.uint32))


def test_expert_ffn_subset_and_slot_table():
    cfg = synth.small_config(0, H=256, F=128, E=6, k=2, seed_cfg=811)
    # pool holds the experts in reverse order: slot = 5 - e
    pool, stride = make_pool(cfg, 0, [5, 4, 3, 2, 1, 0])
    table = to_dev(np.array([5 - e for e in range(6)], dtype=np.int32))
    rng = np.random.default_rng(3)
    T = 5
    x = rng.standard_normal((T, 256), dtype=np.float32)
    ids, w = random_routes(rng, T, 6, 2)
    subset = [0, 2, 3]
    partial = run_ffn(cfg, pool, stride, to_dev(x), 0, ids, w, subset=subset, table=table).cpu().numpy()
    status_clear()
    for t in range(T):
        for j in range(2):
            e = int(ids[t, j])
            if e in subset:
                g, u, d = synth.expert_weights(cfg, 0, e)
                ref = float(w[t, j]) * oracle.expert_ffn(0, 256, 128, g, u, d, x[t].astype(np.float64))
                assert rel_err(partial[t, j][None], ref[None])[0] <= TOL
            else:
                assert np.all(np.isnan(partial[t, j]))  # untouched


def test_out_of_range_ids_and_slots_are_recorded_not_read():
    cfg = synth.small_config(0, H=64, F=64, E=4, k=2, seed_cfg=812)
    pool, stride = make_pool(cfg, 0, range(4))
    x = to_dev(np.ones((2, 64), dtype=np.float32))
    ids = np.array([[0, 9], [1, 2]], dtype=np.int32)     # 9 is outside [0, E)
    w = np.full((2, 2), 0.5, dtype=np.float32)
    status_clear()
    partial = run_ffn(cfg, pool, stride, x, 0, ids, w).cpu().numpy()
    assert L.moe_device_status(clear=True) == L.MOE_ERR_INVALID
    assert np.all(np.isnan(partial[0, 1])) and np.all(np.isfinite(partial[1]))
    # a slot table entry outside the pool: the unit is skipped and recorded
    table = to_dev(np.array([0, 1, 7, 3], dtype=np.int32))
    ids2 = np.array([[0, 2]], dtype=np.int32)
    partial = run_ffn(cfg, pool, stride, x[:1], 0, ids2, w[:1], table=table).cpu().numpy()
    assert L.moe_device_status(clear=True) == L.MOE_ERR_INVALID
    assert np.all(np.isfinite(partial[0, 0])) and np.all(np.isnan(partial[0, 1]))


def test_combine_order_and_extra():
    rng = np.random.default_rng(4)
    T, k, H = 3, 5, 96
    p = rng.standard_normal((T, k, H), dtype=np.float32)
    e = rng.standard_normal((T, H), dtype=np.float32)
    y = torch.empty((T, H), dtype=torch.float32, device=dev())
    L.moe_combine(to_dev(p), T, k, H, to_dev(e), y)
    ref = e.copy()
    for j in range(k):
        ref = ref + p[:, j]
    assert np.array_equal(y.cpu().numpy(), ref)  # same fp32 order: bit-identical
    L.moe_combine(to_dev(p), T, k, H, None, y)
    ref = np.zeros_like(e)
    for j in range(k):
        ref = ref + p[:, j]
    assert np.array_equal(y.cpu().numpy(), ref)


def test_combine_rmsnorm_matches_fp64():
    rng = np.random.default_rng(15)
    T, k, H = 5, 3, 1024
    p = rng.standard_normal((T, k, H), dtype=np.float32)
    e = (rng.standard_normal((T, H)) * 3).astype(np.float32)
    y = torch.empty((T, H), dtype=torch.float32, device=dev())
    xn = torch.empty((T, H), dtype=torch.float32, device=dev())
    L.moe_combine_rmsnorm(to_dev(p), T, k, H, to_dev(e), y, xn)
    ref_y = e.copy()
    for j in range(k):
        ref_y = ref_y + p[:, j]
    assert np.array_equal(y.cpu().numpy(), ref_y)
    np.testing.assert_allclose(xn.cpu().numpy(), oracle.rmsnorm(ref_y.astype(np.float64)), rtol=2e-6, atol=1e-6)
    # k = 0 and no y: normalise the extra only
    L.moe_combine_rmsnorm(None, T, 0, H, to_dev(e), None, xn)
    np.testing.assert_allclose(xn.cpu().numpy(), oracle.rmsnorm(e.astype(np.float64)), rtol=2e-6, atol=1e-6)


# ------------------------------------------------------------------------------------ slot pool

class PoolFixture:
    def __init__(self, cfg, n_layers, n_slots, first_layer=0):
        self.cfg = cfg
        self.stride = (L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F) + 255) // 256 * 256
        self.host = torch.empty(n_layers * cfg.E * self.stride, dtype=torch.uint8, pin_memory=True)
        for l in range(n_layers):
            for e in range(cfg.E):
                g, u, d = synth.expert_weights(cfg, first_layer + l, e)
                L.moe_pack_expert(cfg.qtype, cfg.H, cfg.F, g.ctypes.data, u.ctypes.data, d.ctypes.data,
                                  self.ptr(l, e))
        self.pool = torch.zeros(n_slots * self.stride, dtype=torch.uint8, device=dev())
        self.cs = torch.cuda.Stream()
        self.imgs = (ctypes.c_void_p * (n_layers * cfg.E))(
            *[self.ptr(l, e) for l in range(n_layers) for e in range(cfg.E)])
        desc = L.CacheDesc(qtype=cfg.qtype, H=cfg.H, F=cfg.F, n_layers=n_layers, n_experts=cfg.E,
                           first_layer=first_layer, n_slots=n_slots, slot_bytes=self.stride,
                           device_pool=self.pool.data_ptr(),
                           host_images=ctypes.cast(self.imgs, ctypes.POINTER(ctypes.c_void_p)),
                           copy_stream=self.cs.cuda_stream)
        self.cache = L.moe_cache_create(desc)
        self.table = torch.empty(cfg.E, dtype=torch.int32, device=dev())
        self.img_bytes = L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F)

    def ptr(self, l, e):
        return self.host.data_ptr() + (l * self.cfg.E + e) * self.stride

    def ensure(self, layer, ids):
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        slots = np.empty(ids.size, dtype=np.int32)
        mask = np.zeros(self.cfg.E, dtype=np.uint8)
        n_miss = L.moe_cache_ensure(self.cache, layer, ids.ctypes.data, ids.shape[0], ids.shape[1],
                                    slots.ctypes.data, mask.ctypes.data, self.table)
        return slots, n_miss, mask


def test_slot_pool_matches_lru_simulator_and_uploads_images():
    cfg = synth.small_config(0, H=64, F=64, E=16, k=2, seed_cfg=820)
    n_layers, n_slots = 3, 10
    fx = PoolFixture(cfg, n_layers, n_slots)
    sim = LRUSim(n_slots)
    rng = np.random.default_rng(5)
    host_view = fx.host.numpy()
    for step in range(60):
        layer = int(rng.integers(0, n_layers))
        T = int(rng.integers(1, 5))
        ids = np.stack([rng.choice(cfg.E, size=2, replace=False) for _ in range(T)]).astype(np.int32)
        slots, n_miss, mask = fx.ensure(layer, ids)
        res, hit_ids, miss_ids = sim.ensure(layer, ids.reshape(-1))
        assert n_miss == len(miss_ids)
        assert sorted(np.nonzero(mask)[0].tolist()) == miss_ids
        for i, e in enumerate(ids.reshape(-1)):
            assert slots[i] == res[int(e)]
        L.moe_cache_wait_uploads(fx.cache)
        L.moe_cache_release(fx.cache)
        torch.cuda.synchronize()
        pool = fx.pool.cpu().numpy()
        table = fx.table.cpu().numpy()
        for e, s in res.items():
            assert table[e] == s
            got = pool[s * fx.stride: s * fx.stride + fx.img_bytes]
            off = (layer * cfg.E + e) * fx.stride
            assert np.array_equal(got, host_view[off: off + fx.img_bytes])
        for e in range(cfg.E):
            if e not in res:
                assert table[e] == L.moe_cache_lookup(fx.cache, layer, e)
    st = L.moe_cache_stats_get(fx.cache)
    assert sum(st["hits"]) == sim.hits and sum(st["misses"]) == sim.misses
    assert st["evictions"] == sim.evictions
    assert st["h2d_bytes"] == sim.misses * fx.img_bytes
    L.moe_cache_destroy(fx.cache)


def test_slot_pool_capacity_error_and_fault_injection():
    cfg = synth.small_config(0, H=32, F=32, E=8, k=2, seed_cfg=821)
    fx = PoolFixture(cfg, 1, 3)
    slots, n_miss, _ = fx.ensure(0, [[0, 1]])
    assert n_miss == 2
    ids = np.array([[2, 3], [4, 5]], dtype=np.int32)
    sl = np.empty(4, dtype=np.int32)
    rc = L.moe_cache_ensure_status(fx.cache, 0, ids.ctypes.data, 2, 2, sl.ctypes.data)
    assert rc == L.MOE_ERR_CAPACITY
    assert L.moe_cache_lookup(fx.cache, 0, 0) == 0 and L.moe_cache_lookup(fx.cache, 0, 2) == -1
    before = L.moe_cache_stats_get(fx.cache)
    # the second upload of the next request fails on the host
    L.moe_debug_inject_fault(1, 1)
    ids = np.array([[5, 6]], dtype=np.int32)
    rc = L.moe_cache_ensure_status(fx.cache, 0, ids.ctypes.data, 1, 2, sl.ctypes.data)
    L.moe_debug_inject_fault(0, 0)
    assert rc == L.MOE_ERR_CUDA
    assert L.moe_cache_lookup(fx.cache, 0, 6) == -1          # the failed slot stays empty
    s5 = L.moe_cache_lookup(fx.cache, 0, 5)
    assert s5 >= 0                                            # the earlier upload stands
    assert L.moe_cache_stats_get(fx.cache) == before          # stats unchanged
    # a retry completes, and every resident expert holds its image
    slots, n_miss, _ = fx.ensure(0, [[5, 6]])
    L.moe_cache_wait_uploads(fx.cache)
    L.moe_cache_release(fx.cache)
    torch.cuda.synchronize()
    pool = fx.pool.cpu().numpy()
    host = fx.host.numpy()
    for e in range(cfg.E):
        s = L.moe_cache_lookup(fx.cache, 0, e)
        if s >= 0:
            assert np.array_equal(pool[s * fx.stride: s * fx.stride + fx.img_bytes],
                                  host[e * fx.stride: e * fx.stride + fx.img_bytes])
    L.moe_cache_destroy(fx.cache)


def test_slot_pool_rejects_pageable_images():
    cfg = synth.small_config(0, H=32, F=32, E=2, k=1, seed_cfg=822)
    stride = (L.moe_slot_image_bytes(0, 32, 32) + 255) // 256 * 256
    pageable = np.zeros(2 * stride + 256, dtype=np.uint8)
    pool = torch.zeros(2 * stride, dtype=torch.uint8, device=dev())
    imgs = (ctypes.c_void_p * 2)(pageable.ctypes.data, pageable.ctypes.data + stride)
    desc = L.CacheDesc(qtype=0, H=32, F=32, n_layers=1, n_experts=2, first_layer=0, n_slots=2,
                       slot_bytes=stride, device_pool=pool.data_ptr(),
                       host_images=ctypes.cast(imgs, ctypes.POINTER(ctypes.c_void_p)), copy_stream=None)
    with pytest.raises(L.MoeError) as ei:
        L.moe_cache_create(desc)
    assert ei.value.status == L.MOE_ERR_INVALID


# ------------------------------------------------------------------------------------ bounded waits

@pytest.mark.parametrize("T", [8, 1])
def test_grid_barrier_wait_runs_out_and_is_reported(T):
    """A bounded device-side wait that runs out: the fused GEMV launch's grid barrier is made to
    wait for one arrival more than the grid has (host-armed fault injection, 20 ms bound).  The
    kernel records MOE_ERR_TIMEOUT and returns; the context stays usable and the next call
    (disarmed) gives the same bits as the separate kernels."""
    cfg = synth.small_config(0, H=1024, F=512, E=32, k=8, seed_cfg=960)
    pool, stride = make_pool(cfg, 0, range(cfg.E), False)
    rng = np.random.default_rng(61 + T)
    x_d = to_dev(rng.standard_normal((T, cfg.H), dtype=np.float32))
    ids, w = random_routes(rng, T, cfg.E, cfg.k)
    before = L.moe_get_decode_fused()
    status_clear()
    try:
        L.moe_set_decode_fused(True)
        L.moe_debug_inject_fault(2, 0)
        run_ffn(cfg, pool, stride, x_d, 0, ids, w)
        torch.cuda.synchronize()
        assert L.moe_device_status(clear=True) == L.MOE_ERR_TIMEOUT
        assert L.moe_device_status(clear=False) == 0   # cleared
        fused = run_ffn(cfg, pool, stride, x_d, 0, ids, w).cpu().numpy()   # disarmed again
        status_clear()
        L.moe_set_decode_fused(False)
        sep = run_ffn(cfg, pool, stride, x_d, 0, ids, w).cpu().numpy()
        status_clear()
    finally:
        L.moe_debug_inject_fault(0, 0)
        L.moe_set_decode_fused(before)
    assert np.array_equal(fused.view(np.uint32), sep.view(np.uint32))
