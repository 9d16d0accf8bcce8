"""Full-size parity of the three large configurations, in the launch configuration the
bench uses (the decode-step runtime over real-size slot pools), on sampled outputs:

* Qwen3-30B-A3B-shaped stack (48 layers, 128 experts, top-8, 4-bit, two 24-layer groups of
  1,834 slots): batch 1, every layer of several decode steps, teacher-forced;
* DeepSeek-MoE-16B-shaped stack (28 layers, 64 routed + 2 shared, top-2, q8_0, 224 slots):
  batch 1 and 32;
* the Qwen-shaped prefill layer (bf16 x, all 128 experts resident): 512 tokens, sampled rows.

Routing ids and slot assignments are compared bit-exact; outputs within 2e-3.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_helpers import TOL, ids_match, rel_err
from tests.test_gpu_stack import run_steps
from routed_expert_ffn_gemv_gb300 import _lib as L, synth

torch = pytest.importorskip("torch")
pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _stack(*a, **kw):
    from routed_expert_ffn_gemv_gb300.workload import Stack
    return Stack(*a, **kw)


def test_qwen_stack_full_size_batch1():
    cfg = synth.config(2)
    st = _stack(cfg, max_T=1)
    ck = run_steps(st, cfg, 1, 4, step0=0)
    print(f"config2: worst rel err {ck.worst:.3e} over {ck.compared} token-layers, excluded {ck.excluded}")
    s0, s1 = st.cache_stats()
    assert s0["ensure_calls"] == 4 * 24 and s1["ensure_calls"] == 4 * 24
    st.close()


@pytest.fixture(scope="module")
def deepseek_stack():
    cfg = synth.config(3)
    st = _stack(cfg, max_T=32)
    yield cfg, st
    st.close()


@pytest.mark.parametrize("T", [1, 32])
def test_deepseek_stack_full_size(deepseek_stack, T):
    cfg, st = deepseek_stack
    ck = run_steps(st, cfg, T, 2, step0=50 + T)
    print(f"config3 T={T}: worst rel err {ck.worst:.3e}, excluded {ck.excluded}")


def test_qwen_prefill_layer_512_tokens_sampled():
    cfg = synth.config(4)
    T, H, F, E, k = 512, cfg.H, cfg.F, cfg.E, cfg.k
    from routed_expert_ffn_gemv_gb300.workload import PinnedImages, slot_stride
    imgs = PinnedImages(cfg, [0], range(E))
    stride = slot_stride(cfg)
    pool = imgs.buf.cuda()
    xb = synth.tokens_x(cfg, 0, T)                       # bf16 bits
    x_d = torch.from_numpy(xb.view(np.int16)).cuda()
    wr, b = synth.router_weights(cfg, 0), synth.router_bias(cfg, 0)
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    L.moe_router_topk(x_d, 1, T, H, torch.from_numpy(wr.view(np.int16)).cuda(), torch.from_numpy(b).cuda(),
                      E, k, ids, w)
    ws_bytes = L.moe_expert_ffn_workspace(T, H, F, cfg.qtype, 1, E, k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    partial = torch.empty((T, k, H), dtype=torch.float32, device="cuda")
    L.moe_expert_ffn(x_d, 1, T, H, F, cfg.qtype, E, k, ids, w, None, E, pool, stride, None, 0, partial, ws,
                     ws_bytes)
    y = torch.empty((T, H), dtype=torch.float32, device="cuda")
    L.moe_combine(partial, T, k, H, None, y)
    torch.cuda.synchronize()
    assert L.moe_device_status(clear=True) == 0
    rng = np.random.default_rng(4)
    sample = np.sort(rng.choice(T, size=24, replace=False))
    x64 = oracle.x_to_double(xb[sample], 1)
    res = oracle.moe_layer(cfg.qtype, H, F, k, x64, wr, b, lambda e: synth.expert_weights(cfg, 0, e))
    ids_h = ids.cpu().numpy()[sample]
    m = ids_match(ids_h, res.logits, res.ids, k)
    assert all(v is not False for v in m)
    ref = res.y.copy()
    near = [i for i, v in enumerate(m) if v is None]
    if near:
        sel = np.take_along_axis(res.logits[near], ids_h[near].astype(np.int64), axis=1)
        ww = np.exp(sel - sel.max(axis=1, keepdims=True))
        ww /= ww.sum(axis=1, keepdims=True)
        r2 = oracle.moe_layer(cfg.qtype, H, F, k, x64[near], wr, b, lambda e: synth.expert_weights(cfg, 0, e),
                              route_override=(ids_h[near], ww))
        ref[near] = r2.y
    err = rel_err(y.cpu().numpy()[sample].astype(np.float64), ref)
    assert err.max() <= TOL, err
