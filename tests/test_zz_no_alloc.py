"""The no-allocation expert FFN entry point (moe_expert_ffn_noalloc).

Some callers of this library cannot allocate device memory: a plugin inside a host
framework that owns all device allocations and passes it only input and output
buffers, or a latency-critical decode loop where cudaMalloc/cudaFree (which can
synchronise the whole device) is forbidden.  For them the library keeps the expert
FFN's scratch in a fixed-size device array of its own.  This file checks, through the
C-ABI, that the variant gives the same partial outputs as moe_expert_ffn with a
caller-provided workspace, on two calls in a row (the second call reuses the array
left over by the first), and that a request too large for the array is refused.
It is collected last on purpose, and passes alone or after the other tests.
"""
import numpy as np
import pytest

from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 2e-3  # the per-token normwise tolerance used by every parity test


def _pool(cfg):
    stride = (L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F) + 255) // 256 * 256
    host = torch.empty(cfg.E * stride, dtype=torch.uint8, pin_memory=True)
    for e in range(cfg.E):
        g, u, d = synth.expert_weights(cfg, 0, e, random_scales=True)
        L.moe_pack_expert(cfg.qtype, cfg.H, cfg.F, g.ctypes.data, u.ctypes.data, d.ctypes.data,
                          host.data_ptr() + e * stride)
    return host.cuda(), stride


def _rel(a, b):
    num = np.max(np.abs(a - b), axis=-1)
    den = np.max(np.abs(b), axis=-1)
    return float(np.max(num / np.where(den > 0, den, 1.0)))


@pytest.mark.parametrize("qtype,H,F,E,k,T", [(0, 1024, 512, 32, 8, 8), (1, 2048, 768, 16, 8, 3)])
def test_noalloc_matches_workspace_entry_point_twice(qtype, H, F, E, k, T):
    cfg = synth.small_config(qtype, H=H, F=F, E=E, k=k, seed_cfg=990 + qtype)
    pool, stride = _pool(cfg)
    ws_bytes = L.moe_expert_ffn_workspace(T, H, F, qtype, 0, E, k)
    assert ws_bytes <= L.MOE_NOALLOC_SCRATCH_MAX
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    rng = np.random.default_rng(qtype + 7)
    for call in range(2):
        x = torch.from_numpy(rng.standard_normal((T, H), dtype=np.float32)).cuda()
        ids = np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
        w = rng.uniform(0.1, 1.0, size=(T, k)).astype(np.float32)
        ids_d, w_d = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
        ref = torch.empty((T, k, H), dtype=torch.float32, device="cuda")
        got = torch.full((T, k, H), float("nan"), dtype=torch.float32, device="cuda")
        L.moe_expert_ffn(x, 0, T, H, F, qtype, E, k, ids_d, w_d, None, E, pool, stride, None, 0, ref,
                         ws, ws_bytes)
        L.moe_expert_ffn_noalloc(x, 0, T, H, F, qtype, E, k, ids_d, w_d, None, E, pool, stride, None, 0,
                                 got)
        torch.cuda.synchronize()
        r, g = ref.cpu().numpy().reshape(T * k, H), got.cpu().numpy().reshape(T * k, H)
        assert np.all(np.isfinite(g)), call
        assert _rel(g, r) <= TOL, call
    assert L.moe_device_status(clear=True) == 0


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
