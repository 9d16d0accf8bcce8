"""Pins of the CPU oracle against things other than itself (no GPU).

Each check uses an independent route to the expected value: numpy's own fp16
decoder and matmul, hand-worked fixtures under tests/golden/, closed forms,
brute-force properties on small inputs, and the numbers printed on the pages.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.lru_sim import CapacityError, LRUSim, slots_for_budget
from routed_expert_ffn_gemv_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------------------------ decoders

def test_fp16_decoder_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoder_matches_float32_upper_half():
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 65536, size=4000).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # drop inf/nan patterns
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(got, ref)


def _np_decode_q8_0(blocks):
    """Independent numpy decoder of canonical q8_0 blocks (structured dtype)."""
    dt = np.dtype([("d", "<f2"), ("q", "i1", 32)])
    b = np.frombuffer(np.ascontiguousarray(blocks).tobytes(), dtype=dt)
    return (b["d"].astype(np.float64)[:, None] * b["q"].astype(np.float64)).reshape(-1)


def _np_decode_q4(blocks):
    dt = np.dtype([("d", "<f2"), ("m", "<f2"), ("qs", "u1", 16)])
    b = np.frombuffer(np.ascontiguousarray(blocks).tobytes(), dtype=dt)
    q = np.empty((b.size, 32), dtype=np.float64)
    q[:, 0::2] = b["qs"] & 0x0F
    q[:, 1::2] = b["qs"] >> 4
    return (b["d"].astype(np.float64)[:, None] * q + b["m"].astype(np.float64)[:, None]).reshape(-1)


def test_q8_0_dequant_all_256_codes_random_scales():
    rng = np.random.default_rng(1)
    codes = np.arange(-128, 128, dtype=np.int16).astype(np.int8)  # 8 blocks of 32
    blocks = np.zeros((8, 34), dtype=np.uint8)
    d = rng.uniform(-2, 2, size=8).astype(np.float16)
    blocks[:, 0:2] = d.view(np.uint8).reshape(8, 2)
    blocks[:, 2:] = codes.view(np.uint8).reshape(8, 32)
    got = oracle.dequant(0, blocks.reshape(-1))
    expect = (d.astype(np.float64)[:, None] * codes.reshape(8, 32).astype(np.float64)).reshape(-1)
    assert np.array_equal(got, expect)


def test_q4_dequant_every_code_in_both_nibbles():
    rng = np.random.default_rng(2)
    q = np.concatenate([np.arange(16), np.arange(15, -1, -1)])          # block 0: 0..15, 15..0
    q2 = np.array([(i * 7 + 3) % 16 for i in range(32)])                 # block 1: another pattern
    codes = np.stack([q, q2])
    d = rng.uniform(0.001, 0.01, size=2).astype(np.float16)
    m = rng.uniform(-0.05, 0.05, size=2).astype(np.float16)
    blocks = np.zeros((2, 20), dtype=np.uint8)
    blocks[:, 0:2] = d.view(np.uint8).reshape(2, 2)
    blocks[:, 2:4] = m.view(np.uint8).reshape(2, 2)
    blocks[:, 4:] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    got = oracle.dequant(1, blocks.reshape(-1)).reshape(2, 32)
    expect = d.astype(np.float64)[:, None] * codes + m.astype(np.float64)[:, None]
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("qtype", [0, 1])
def test_qmatvec_matches_numpy_decode_and_matmul_with_per_block_scales(qtype):
    rng = np.random.default_rng(3 + qtype)
    rows, cols = 40, 96
    if qtype == 0:
        mat = synth.q8_0_blocks(rng, rows, cols, 0.02 / 40, random_scales=True)
        W = _np_decode_q8_0(mat).reshape(rows, cols)
    else:
        mat = synth.q4_sm_blocks(rng, rows, cols, 0.004, -0.03, random_scales=True)
        W = _np_decode_q4(mat).reshape(rows, cols)
    x = rng.standard_normal(cols)
    y = oracle.qmatvec(qtype, mat, rows, cols, x)
    np.testing.assert_allclose(y, W @ x, rtol=1e-13, atol=1e-13)
    # a transposed or block-shifted read would differ
    assert not np.allclose(y, W[:, ::-1] @ x)


# ------------------------------------------------------------------------------------ router

def test_router_logits_match_numpy_matmul():
    rng = np.random.default_rng(4)
    T, H, E = 5, 64, 12
    x = rng.standard_normal((T, H))
    w = (rng.standard_normal((H, E)) * 0.2).astype(np.float16)
    b = rng.standard_normal(E)
    got = oracle.router_logits(x, w.view(np.uint16), b)
    np.testing.assert_allclose(got, x @ w.astype(np.float64) + b, rtol=1e-13, atol=1e-12)
    got0 = oracle.router_logits(x, w.view(np.uint16), None)
    np.testing.assert_allclose(got0, x @ w.astype(np.float64), rtol=1e-13, atol=1e-12)


def test_topk_golden_cases():
    for case in _golden("topk_cases.json")["cases"]:
        l = np.array([case["logits"]])
        ids, w, gap = oracle.topk_softmax(l, case["k"])
        assert ids[0].tolist() == case["ids"], case
        if case["gap"] is None:
            assert math.isinf(gap[0])
        else:
            assert gap[0] == case["gap"]
        assert abs(w.sum() - 1.0) < 1e-12


def test_topk_brute_force_properties():
    rng = np.random.default_rng(6)
    for trial in range(300):
        E = int(rng.integers(1, 9))
        k = int(rng.integers(1, E + 1))
        l = rng.integers(-3, 4, size=E).astype(np.float64)  # many exact ties
        ids, w, gap = oracle.topk_softmax(l[None, :], k)
        sel = ids[0].tolist()
        rest = [e for e in range(E) if e not in sel]
        assert len(set(sel)) == k
        for a in sel:
            for b in rest:
                assert l[a] > l[b] or (l[a] == l[b] and a < b)
        for j in range(k - 1):
            a, b = sel[j], sel[j + 1]
            assert l[a] > l[b] or (l[a] == l[b] and a < b)
        if rest:
            assert gap[0] == l[sel[-1]] - max(l[b] for b in rest)


def test_softmax_closed_forms():
    # k = 1 gives weight 1
    _, w, _ = oracle.topk_softmax(np.array([[0.3, -1.0, 2.0]]), 1)
    assert w[0, 0] == 1.0
    # uniform logits with k = E gives 1/E
    _, w, _ = oracle.topk_softmax(np.zeros((1, 7)), 7)
    np.testing.assert_allclose(w, np.full((1, 7), 1 / 7), rtol=0, atol=1e-15)
    # two selected: the logistic function of the difference
    l = np.array([[1.25, -0.5, 0.75, -4.0]])
    ids, w, _ = oracle.topk_softmax(l, 2)
    assert ids[0].tolist() == [0, 2]
    np.testing.assert_allclose(w[0, 0], 1.0 / (1.0 + math.exp(-(1.25 - 0.75))), rtol=1e-15)
    # invariant to a constant shift of all logits (a uniform bias)
    rng = np.random.default_rng(8)
    l = rng.standard_normal((4, 16)) * 3
    i1, w1, _ = oracle.topk_softmax(l, 5)
    i2, w2, _ = oracle.topk_softmax(l + 11.0, 5)
    assert np.array_equal(i1, i2)
    np.testing.assert_allclose(w1, w2, rtol=1e-13)
    # softmax over the selected k equals full softmax renormalised over the selected k
    full = np.exp(l - l.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    sel = np.take_along_axis(full, i1.astype(np.int64), axis=1)
    np.testing.assert_allclose(w1, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13)


# ------------------------------------------------------------------------------------ FFN

def test_silu_textbook_values():
    assert oracle.silu(0.0) == 0.0
    # logistic(1) = 0.7310585786300049, logistic(-1) = 0.2689414213699951
    assert abs(oracle.silu(1.0) - 0.7310585786300049) < 1e-15
    assert abs(oracle.silu(-1.0) + 0.2689414213699951) < 1e-15
    for z in (0.3, 2.0, 7.5):
        assert abs(oracle.silu(z) - oracle.silu(-z) - z) < 1e-14


def _const_q8_0(rows, cols, q, d):
    blk = np.zeros(34, dtype=np.uint8)
    blk[0:2] = np.array([d], dtype=np.float16).view(np.uint8)
    blk[2:] = np.int8(q).view(np.uint8)
    return np.tile(blk, rows * cols // 32)


def test_expert_ffn_closed_form_all_equal_weights():
    # H = F = 32, every weight 2^-5: g = u = s = sum(x)/32, h = silu(s)*s, y_i = 32 * 2^-5 * h = h
    H = F = 32
    W = _const_q8_0(32, 32, 1, 2.0 ** -5)
    rng = np.random.default_rng(9)
    x = rng.standard_normal(H)
    s = x.sum() / 32.0
    h = s / (1.0 + math.exp(-s)) * s
    y = oracle.expert_ffn(0, H, F, W, W, W, x)
    np.testing.assert_allclose(y, np.full(H, h), rtol=1e-14)


@pytest.mark.parametrize("qtype", [0, 1])
def test_expert_ffn_matches_numpy_dense(qtype):
    cfg = synth.small_config(qtype, H=64, F=96, E=2, k=1)
    g, u, d = synth.expert_weights(cfg, 0, 1, random_scales=True)
    dec = _np_decode_q8_0 if qtype == 0 else _np_decode_q4
    Wg, Wu, Wd = dec(g).reshape(96, 64), dec(u).reshape(96, 64), dec(d).reshape(64, 96)
    x = np.random.default_rng(10).standard_normal(64)
    gv, uv = Wg @ x, Wu @ x
    ref = Wd @ (gv / (1 + np.exp(-gv)) * uv)
    y = oracle.expert_ffn(qtype, 64, 96, g, u, d, x)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    # gate and up are not interchangeable (silu is applied to the gate only)
    y_swapped = oracle.expert_ffn(qtype, 64, 96, u, g, d, x)
    assert not np.allclose(y, y_swapped)


def _dense_layer_numpy(cfg, layer, x, wr, b, shared_ids=()):
    dec = _np_decode_q8_0 if cfg.qtype == 0 else _np_decode_q4
    H, F, E = cfg.H, cfg.F, cfg.E
    ys = []
    for e in list(range(E)) + list(shared_ids):
        g, u, d = synth.expert_weights(cfg, layer, e)
        Wg, Wu, Wd = dec(g).reshape(F, H), dec(u).reshape(F, H), dec(d).reshape(H, F)
        gv, uv = x @ Wg.T, x @ Wu.T
        ys.append((gv / (1 + np.exp(-gv)) * uv) @ Wd.T)
    return np.stack(ys, axis=1)  # [T][E(+S)][H]


@pytest.mark.parametrize("qtype", [0, 1])
def test_dense_all_experts_then_mask_equals_routed(qtype):
    cfg = synth.small_config(qtype, H=64, F=64, E=6, k=2, bias_a=1.0, n_shared=1)
    x = np.random.default_rng(11).standard_normal((3, 64))
    wr, b = synth.router_weights(cfg, 0), synth.router_bias(cfg, 0)
    res = oracle.moe_layer(qtype, 64, 64, 2, x, wr, b, lambda e: synth.expert_weights(cfg, 0, e),
                           shared=[synth.expert_weights(cfg, 0, 6)])
    ydense = _dense_layer_numpy(cfg, 0, x, wr, b, shared_ids=(6,))
    logits = x @ wr.view(np.float16).astype(np.float64) + b
    mask = np.zeros((3, 6))
    for t in range(3):
        for j in range(2):
            mask[t, res.ids[t, j]] = res.weights[t, j]
    yref = np.einsum("te,teh->th", mask, ydense[:, :6]) + ydense[:, 6]
    np.testing.assert_allclose(res.y, yref, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(res.logits, logits, rtol=1e-12, atol=1e-12)


def test_k_equals_E_uniform_weights_is_mean_of_all_experts():
    cfg = synth.small_config(0, H=32, F=64, E=4, k=4)
    x = np.random.default_rng(12).standard_normal((2, 32))
    wr = np.zeros((32, 4), dtype=np.uint16)  # all-zero router: equal logits
    res = oracle.moe_layer(0, 32, 64, 4, x, wr, None, lambda e: synth.expert_weights(cfg, 0, e))
    np.testing.assert_allclose(res.weights, 0.25, rtol=0, atol=1e-15)
    assert res.ids.tolist() == [[0, 1, 2, 3]] * 2
    ydense = _dense_layer_numpy(cfg, 0, x, wr, None)
    np.testing.assert_allclose(res.y, ydense.mean(axis=1), rtol=1e-11, atol=1e-11)


# ------------------------------------------------------------------------------------ LRU

def test_lru_golden_traces():
    for tr in _golden("lru_traces.json")["traces"]:
        sim = LRUSim(tr["n_slots"])
        for (layer, ids), slots, h, m in zip(tr["requests"], tr["slots"], tr["hits"], tr["misses"]):
            res, hit_ids, miss_ids = sim.ensure(layer, ids)
            assert {str(e): s for e, s in res.items()} == slots, tr["name"]
            assert (len(hit_ids), len(miss_ids)) == (h, m), tr["name"]
        assert sim.evictions == tr["evictions"], tr["name"]


def test_lru_capacity_error_leaves_state_unchanged():
    sim = LRUSim(2)
    sim.ensure(0, [0])
    with pytest.raises(CapacityError):
        sim.ensure(0, [1, 2, 3])
    assert sim.clock == 1 and sim.hits == 0 and sim.misses == 1
    res, hit, miss = sim.ensure(0, [0])
    assert res == {0: 0} and hit == [0]


def test_lru_request_never_evicts_its_own_members():
    rng = np.random.default_rng(13)
    sim = LRUSim(6)
    for step in range(400):
        ids = rng.integers(0, 12, size=int(rng.integers(1, 7)))
        layer = int(rng.integers(0, 3))
        res, _, _ = sim.ensure(layer, ids)
        assert len(set(res.values())) == len(res)       # distinct slots
        for e, s in res.items():
            assert sim.owner[s] == (layer, e)             # every member still resident


# ------------------------------------------------------------------------------------ page numbers

def test_slot_budget_reproduces_page_numbers():
    p = _golden("page_numbers.json")["slot_budget"]
    MiB = 1 << 20
    per = p["per_expert_bytes"]
    # the two per-expert sizes reproduce the page's 16.35 GiB of experts
    total = p["layers_per_group"] * p["experts"] * sum(per)
    assert round(total / (1 << 30), 2) == p["total_expert_gib"]
    slots = slots_for_budget(p["budget_mib"] * MiB, per, p["k"])
    assert len(slots) == 2 and abs(slots[0] - p["slots_per_group"]) <= 1
    n_exp = p["layers_per_group"] * p["experts"]
    assert round(100.0 * p["slots_per_group"] / n_exp, 1) == p["fraction_pct"]
    assert slots_for_budget(p["floor_ok_mib"] * MiB, per, p["k"]) != []
    assert slots_for_budget(p["floor_fail_mib"] * MiB, per, p["k"]) == []


def test_fp16_scale_constants():
    for v, expect in _golden("page_numbers.json")["fp16_scales"]["values"]:
        bits = synth._fp16_bits(v)
        assert oracle.fp16_to_double(bits) == expect


def test_block_sizes():
    p = _golden("page_numbers.json")["block_bytes"]
    cfg0 = synth.config(0)
    assert cfg0.block_bytes == p["q8_0_block"]
    # page 2's size example counts 4 bits per weight and no scales
    h, f, e = p["page2_shape"]
    assert h * f * e * 4 // 8 == p["page2_codes_only_bytes"]
    # our 4-bit block adds 4 bytes of scale+min per 32 weights: 20/16 of that
    assert h * f * e // 32 * synth.Q4_SM_BLOCK_BYTES == p["page2_codes_only_bytes"] * 20 // 16
    assert cfg0.expert_bytes == 417792
    assert synth.config(1).expert_bytes == 1671168
    assert synth.config(2).expert_bytes == 2949120
    assert synth.config(3).expert_bytes == 9191424


def test_rmsnorm_closed_forms():
    # [3, 4, 0]: mean of squares 25/3
    got = oracle.rmsnorm(np.array([[3.0, 4.0, 0.0]]), eps=0.0)
    np.testing.assert_allclose(got, [[3 / np.sqrt(25 / 3), 4 / np.sqrt(25 / 3), 0.0]], rtol=1e-15)
    rng = np.random.default_rng(14)
    h = rng.standard_normal((4, 64)) * 7.0
    xn = oracle.rmsnorm(h, eps=0.0)
    np.testing.assert_allclose(np.mean(xn * xn, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle.rmsnorm(h * 1e3, eps=0.0), xn, rtol=1e-13)   # scale invariant
    # eps: a constant vector c gives c / sqrt(c^2 + eps)
    c = 0.01
    np.testing.assert_allclose(oracle.rmsnorm(np.full((1, 8), c), eps=1e-6), c / np.sqrt(c * c + 1e-6), rtol=1e-14)


# ------------------------------------------------------------------------------------ comparison and inputs

def test_relative_error_hand_worked_rows():
    # row 0: |[1,-3] - [2,-4]| = [1, 1], max |ref| = 4 -> 1/4
    # row 1: reference all zero -> the raw max difference (denominator 1)
    # row 2: the largest difference sits on the smallest reference entry: 0.5 / 10
    y = np.array([[1.0, -3.0], [0.5, -0.25], [10.0, 0.6]])
    ref = np.array([[2.0, -4.0], [0.0, 0.0], [10.0, 0.1]])
    got = oracle.relative_error(y, ref)
    assert got.shape == (3,)
    assert got.tolist() == [0.25, 0.5, 0.05]
    # normwise per token: a row is not divided by its own element-wise magnitudes
    assert oracle.relative_error(np.array([[1.0, 1e-9 + 1e-6]]), np.array([[1.0, 1e-9]]))[0] == pytest.approx(1e-6)
    # the reduction runs over the hidden axis of [T][H], and y may come flattened
    y3 = np.array([1.0, 2.0, 3.0, 4.0, 5.0, 6.0])
    r3 = np.array([[1.0, 2.0, 4.0], [4.0, 5.0, 8.0]])
    assert oracle.relative_error(y3, r3).tolist() == [1.0 / 4.0, 2.0 / 8.0]


def test_x_to_double_bf16_and_fp32():
    rng = np.random.default_rng(31)
    bits = rng.integers(0, 65536, size=3000).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # drop inf / nan patterns
    got = oracle.x_to_double(bits.reshape(-1, 1), 1).reshape(-1)
    # against the oracle's own scalar decoder (pinned above against float32) ...
    scalar = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(got, scalar)
    # ... and against numpy: a bf16 pattern is the upper half of a float32
    via_np = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.array_equal(got, via_np)
    # hand values: 0x3F80 = 1.0, 0xC000 = -2.0, 0x3E80 = 0.25, 0x0001 = 2^-133
    hand = oracle.x_to_double(np.array([[0x3F80, 0xC000, 0x3E80, 0x0001]], dtype=np.uint16), 1)
    assert hand.tolist() == [[1.0, -2.0, 0.25, 2.0 ** -133]]
    # fp32 input: values unchanged, shape kept
    xf = rng.standard_normal((4, 5)).astype(np.float32)
    out = oracle.x_to_double(xf, 0)
    assert out.dtype == np.float64 and out.shape == (4, 5)
    assert np.array_equal(out, xf.astype(np.float64))


def test_route_override_uses_the_given_ids_and_weights():
    """moe_layer(route_override=(ids, w)) must weight the given experts by the given weights,
    not by the oracle's own routing or softmax (near-tie tokens are checked this way)."""
    cfg = synth.small_config(1, H=64, F=64, E=6, k=2, bias_a=1.0, n_shared=1)
    x = np.random.default_rng(41).standard_normal((3, 64))
    wr, b = synth.router_weights(cfg, 0), synth.router_bias(cfg, 0)
    own = oracle.moe_layer(1, 64, 64, 2, x, wr, b, lambda e: synth.expert_weights(cfg, 0, e),
                           shared=[synth.expert_weights(cfg, 0, 6)])
    # a route the router did not take, in the reverse order, with weights unrelated to the logits
    ids = np.array([[5, 0], [1, 4], [3, 2]], dtype=np.int32)
    for t in range(3):
        assert set(ids[t]) != set(own.ids[t]) or list(ids[t]) != list(own.ids[t])
    w = np.array([[0.9, 0.1], [0.3, 0.7], [0.55, 0.45]])
    res = oracle.moe_layer(1, 64, 64, 2, x, wr, b, lambda e: synth.expert_weights(cfg, 0, e),
                           shared=[synth.expert_weights(cfg, 0, 6)], route_override=(ids, w))
    ydense = _dense_layer_numpy(cfg, 0, x, wr, b, shared_ids=(6,))  # numpy, every expert
    yref = np.stack([w[t, 0] * ydense[t, ids[t, 0]] + w[t, 1] * ydense[t, ids[t, 1]] + ydense[t, 6]
                     for t in range(3)])
    np.testing.assert_allclose(res.y, yref, rtol=1e-11, atol=1e-11)
    assert res.ids.tolist() == ids.tolist()
    assert np.array_equal(res.weights, w)
    # the logits stay the router's own (the caller derives near-tie weights from them)
    np.testing.assert_allclose(res.logits, own.logits, rtol=0, atol=0)
    # the per-expert outputs follow the override's order
    for t in range(3):
        for j in range(2):
            np.testing.assert_allclose(res.y_experts[t, j], ydense[t, ids[t, j]], rtol=1e-11, atol=1e-11)


def test_lru_policy_golden_traces():
    """Frequency admission and the LRU window against hand-derived traces."""
    for tr in _golden("lru_traces.json")["policy_traces"]:
        sim = LRUSim(tr["n_slots"], admit_after=tr["admit_after"], window=tr["window"],
                     first_layer=tr["first_layer"])
        for (layer, ids, nt), slots, h, m in zip(tr["requests"], tr["slots"], tr["hits"], tr["misses"]):
            res, hit_ids, miss_ids = sim.ensure(layer, ids, n_tokens=nt)
            assert {str(e): s for e, s in res.items()} == slots, tr["name"]
            assert (len(hit_ids), len(miss_ids)) == (h, m), tr["name"]
        assert sim.evictions == tr["evictions"], tr["name"]
        assert sim.bypassed == tr["bypassed"], tr["name"]
        assert sim.window_evictions == tr["window_evictions"], tr["name"]


def test_lru_policies_reduce_to_plain_lru_and_keep_invariants():
    rng = np.random.default_rng(17)
    plain, same = LRUSim(6), LRUSim(6, admit_after=1, window=0)
    adm, win = LRUSim(6, admit_after=3), LRUSim(6, window=4, first_layer=0)
    for step in range(500):
        layer = int(rng.integers(0, 3))
        ids = rng.integers(0, 10, size=int(rng.integers(1, 5)))
        r0 = plain.ensure(layer, ids, n_tokens=2)
        assert same.ensure(layer, ids, n_tokens=2) == r0     # the defaults are plain LRU
        for sim in (adm, win):
            res, hit, miss = sim.ensure(layer, ids, n_tokens=2)
            slots = [s for s in res.values() if s >= 0]
            assert len(set(slots)) == len(slots)              # distinct slots
            for e, s in res.items():
                if s >= 0:
                    assert sim.owner[s] == (layer, e)
            assert set(hit) | set(miss) == set(int(e) for e in ids)
    # admission: an expert is never resident before its third access
    assert all(adm.count[key] >= 3 for key in adm.where)
    # window: nothing resident is more than 4 tokens stale after the last request
    assert all(win.tok - win.last_tok[s] <= 4 + 2 for s in range(6) if win.owner[s] is not None)
    assert adm.bypassed > 0 and win.window_evictions > 0


def test_load_threshold_drops_light_routes_without_renormalising():
    """moe_layer(load_threshold=th) against a numpy dense computation that keeps only the
    selected routes whose softmax weight is at least th (page 1, section 4.3)."""
    cfg = synth.small_config(0, H=64, F=64, E=8, k=4, bias_a=1.0)
    x = np.random.default_rng(23).standard_normal((5, 64)) * 3.0   # spread out the weights
    wr, b = synth.router_weights(cfg, 0), synth.router_bias(cfg, 0)
    ex = lambda e: synth.expert_weights(cfg, 0, e)
    full = oracle.moe_layer(0, 64, 64, 4, x, wr, b, ex)
    th = float(np.median(full.weights))         # some routes on each side
    res = oracle.moe_layer(0, 64, 64, 4, x, wr, b, ex, load_threshold=th)
    ydense = _dense_layer_numpy(cfg, 0, x, wr, b)
    expect = np.zeros((5, 64))
    n_drop = 0
    for t in range(5):
        for j in range(4):
            if full.weights[t, j] >= th:
                expect[t] += full.weights[t, j] * ydense[t, full.ids[t, j]]
                assert res.ids[t, j] == full.ids[t, j] and res.weights[t, j] == full.weights[t, j]
            else:
                n_drop += 1
                assert res.ids[t, j] == -1 and res.weights[t, j] == 0.0
    assert 0 < n_drop < 20
    np.testing.assert_allclose(res.y, expect, rtol=1e-11, atol=1e-11)
    # threshold 0 changes nothing; above every weight only shared experts would remain
    np.testing.assert_allclose(oracle.moe_layer(0, 64, 64, 4, x, wr, b, ex, load_threshold=0.0).y, full.y, rtol=0, atol=0)
    assert np.all(oracle.moe_layer(0, 64, 64, 4, x, wr, b, ex, load_threshold=1.01).y == 0.0)


def test_lru_prefetch_hand_trace():
    """Speculative requests (page 3, section 2.3, cross-layer prefetch): the same LRU rules,
    their own statistics, abandoned when a victim would be a slot of the last real request.
    Derived by hand (stamps in brackets):
      1 real (0,[0])      -> 0:s0 [1]                        last real {s0}
      2 pf   (1,[5])      -> 5:s1 [2] (free slot)
      3 real (0,[1])      -> 1:s2 [3]                        last real {s2}
      4 pf   (1,[5,6])    -> 5 hit s1 [4]; 6 evicts s0 (oldest, not s2) [5]
      5 real (1,[6])      -> hit s0 [6]                      last real {s0}
      6 pf   (2,[7])      -> evicts s2 [3] -> 7:s2 [7]
      7 real (0,[0,1])    -> 0 evicts s1 [4] -> s1 [8]; 1 evicts s0 [6] -> s0 [9]; last real {s1, s0}
      8 pf   (1,[5,6])    -> would evict s2 then s1: s1 is the last real request's -> abandoned"""
    sim = LRUSim(3)
    assert sim.ensure(0, [0])[0] == {0: 0}
    assert sim.prefetch(1, [5]) == {5: 1}
    assert sim.ensure(0, [1])[0] == {1: 2}
    assert sim.prefetch(1, [5, 6]) == {5: 1, 6: 0}
    res, hit, miss = sim.ensure(1, [6])
    assert res == {6: 0} and hit == [6]
    assert sim.prefetch(2, [7]) == {7: 2}
    assert sim.ensure(0, [0, 1])[0] == {0: 1, 1: 0}
    before = (list(sim.owner), list(sim.stamp), sim.clock)
    assert sim.prefetch(1, [5, 6]) == {}
    assert (list(sim.owner), list(sim.stamp), sim.clock) == before
    assert (sim.pf_queries, sim.pf_hits, sim.pf_fills, sim.pf_aborts) == (4, 1, 3, 1)
    assert (sim.hits, sim.misses, sim.evictions) == (1, 4, 4)
    # admission: a prediction admits what the real access would (count + 1 >= theta) but
    # stores no access
    adm = LRUSim(4, admit_after=2)
    assert adm.ensure(0, [3])[0] == {3: -1}              # count 1: bypassed
    assert adm.prefetch(0, [3]) == {3: 0} and adm.count[(0, 3)] == 1 and adm.pf_fills == 1
    res, hit, _ = adm.ensure(0, [3])                     # count 2, prefetched: a hit
    assert res == {3: 0} and hit == [3]
    assert adm.prefetch(0, [7]) == {7: -1} and adm.pf_fills == 1   # never seen: 0 + 1 < 2
