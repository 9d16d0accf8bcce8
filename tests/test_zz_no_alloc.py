"""The no-allocation expert FFN entry point (moe_expert_ffn_noalloc).

Some callers of this library cannot allocate device memory: a plugin inside a host
framework that owns all device allocations and passes it only input and output
buffers, or a latency-critical decode loop where cudaMalloc/cudaFree (which can
synchronise the whole device) is forbidden.  For them the library keeps the expert
FFN's scratch in a fixed-size device array of its own.  This file checks, through the
C-ABI, that the variant gives bit-identical partial outputs to moe_expert_ffn with a
caller-provided workspace (both run the same kernels on the same inputs) on calls in a
row that reuse the array: a larger call first, then smaller ones of another activation
type, so that contents left over from an earlier call must go unread; one call takes the
tensor-core prefill path through the array.  A request too large for the array is refused.
It is collected last on purpose, and passes alone or after the other tests.
"""
import numpy as np
import pytest

from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _pool(cfg):
    stride = (L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F) + 255) // 256 * 256
    host = torch.empty(cfg.E * stride, dtype=torch.uint8, pin_memory=True)
    for e in range(cfg.E):
        g, u, d = synth.expert_weights(cfg, 0, e, random_scales=True)
        L.moe_pack_expert(cfg.qtype, cfg.H, cfg.F, g.ctypes.data, u.ctypes.data, d.ctypes.data,
                          host.data_ptr() + e * stride)
    return host.cuda(), stride


def _x(rng, T, H, xtype):
    xf = rng.standard_normal((T, H), dtype=np.float32)
    if xtype == 0:
        return torch.from_numpy(xf).cuda()
    bits = (xf.view(np.uint32) >> 16).astype(np.uint16)  # bf16 by truncation: any pattern will do
    return torch.from_numpy(bits.view(np.int16)).cuda()


def _compare_calls(cfg, pool, stride, calls, seed):
    """Each (T, xtype) call through both entry points; outputs must be bit-identical."""
    H, F, E, k, qtype = cfg.H, cfg.F, cfg.E, cfg.k, cfg.qtype
    rng = np.random.default_rng(seed)
    for n, (T, xtype) in enumerate(calls):
        ws_bytes = L.moe_expert_ffn_workspace(T, H, F, qtype, xtype, E, k)
        assert ws_bytes <= L.MOE_NOALLOC_SCRATCH_MAX
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        x = _x(rng, T, H, xtype)
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        w = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
        ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
        ref = torch.full((T, k, H), float("nan"), dtype=torch.float32, device="cuda")
        got = torch.full((T, k, H), float("nan"), dtype=torch.float32, device="cuda")
        L.moe_expert_ffn(x, xtype, T, H, F, qtype, E, k, ids_d, w_d, None, E, pool, stride, None, 0, ref,
                         ws, ws_bytes)
        L.moe_expert_ffn_noalloc(x, xtype, T, H, F, qtype, E, k, ids_d, w_d, None, E, pool, stride, None, 0,
                                 got)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy(), got.cpu().numpy()
        assert np.all(np.isfinite(r)), n
        assert np.array_equal(g, r), (n, T, xtype, float(np.max(np.abs(g - r))))
    assert L.moe_device_status(clear=True) == 0


@pytest.mark.parametrize("qtype,H,F,E,k,T0", [(0, 1024, 512, 32, 8, 24), (1, 2048, 768, 16, 8, 16)])
def test_noalloc_matches_workspace_entry_point_on_calls_in_a_row(qtype, H, F, E, k, T0):
    cfg = synth.small_config(qtype, H=H, F=F, E=E, k=k, seed_cfg=990 + qtype)
    pool, stride = _pool(cfg)
    # set-up call (T = 0): resolves the array's address, computes nothing
    L.moe_expert_ffn_noalloc(None, 0, 0, H, F, qtype, E, k, None, None, None, E, None, stride, None, 0, None)
    # a batch of T0 fp32 tokens (the largest that fits the array), then 3 bf16 tokens, then 1
    # fp32 token: later calls need less scratch than the first and must not read what it left
    _compare_calls(cfg, pool, stride, [(T0, 0), (3, 1), (1, 0)], seed=qtype + 7)


def test_noalloc_prefill_path_then_decode():
    # 40 bf16 tokens on a layer with hidden 256 (a multiple of 256) and FFN 128: the tcgen05
    # grouped-GEMM path, whose scratch also fits the array; then two decode calls
    cfg = synth.small_config(1, H=256, F=128, E=8, k=2, seed_cfg=995)
    pool, stride = _pool(cfg)
    _compare_calls(cfg, pool, stride, [(40, 1), (5, 1), (2, 0)], seed=17)


def test_noalloc_rejects_requests_beyond_its_array():
    # batch 32, top-8 of a layer with hidden 4096 and FFN 14336 (q8_0): its gate/up partial
    # sums alone need far more scratch than 8 MiB
    need = L.moe_expert_ffn_workspace(32, 4096, 14336, 0, 0, 64, 8)
    assert need > L.MOE_NOALLOC_SCRATCH_MAX
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    slot = (L.moe_slot_image_bytes(0, 4096, 14336) + 255) // 256 * 256
    with pytest.raises(L.MoeError) as ei:
        L.moe_expert_ffn_noalloc(dummy, 0, 32, 4096, 14336, 0, 64, 8, dummy, dummy, None, 64, dummy, slot,
                                 None, 0, dummy)
    assert ei.value.status == L.MOE_ERR_UNSUPPORTED
