"""Host-side tests of libmoe (no GPU): build, exported symbols, slot-image packing,
slot budget, argument validation before any device work."""
import ctypes
import os
import re

import numpy as np
import pytest

from routed_expert_ffn_gemv_gb300 import _build, _lib as L, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return L.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(names) == sorted(L.EXPORTED)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert L.status_string(code) not in ("", "unknown status")
    assert L.status_string(7) == "unknown status"


@pytest.mark.parametrize("qtype", [0, 1])
def test_pack_unpack_round_trip_and_layout(lib, qtype):
    cfg = synth.small_config(qtype, H=64, F=96, E=1, k=1)
    g, u, d = synth.expert_weights(cfg, 0, 0, random_scales=True)
    n = L.moe_slot_image_bytes(qtype, 64, 96)
    assert n == g.size + u.size + d.size  # the image is as large as the canonical tensors
    img = np.zeros(n + 16, dtype=np.uint8)
    off = (-img.ctypes.data) % 16
    view = img[off:off + n]
    assert L.moe_pack_expert(qtype, 64, 96, g.ctypes.data, u.ctypes.data, d.ctypes.data, view.ctypes.data) == n
    # the same blocks regrouped; 8-bit codes in offset binary (q + 128), scales unchanged
    BB = 34 if qtype == 0 else 20
    canon = np.concatenate([g, u, d])
    if qtype == 0:
        canon = canon.reshape(-1, BB).copy()
        canon[:, 2:] ^= 0x80
        canon = canon.reshape(-1)
    assert np.array_equal(np.sort(view), np.sort(canon))
    g2, u2, d2 = np.zeros_like(g), np.zeros_like(u), np.zeros_like(d)
    L.moe_unpack_expert(qtype, 64, 96, view.ctypes.data, g2.ctypes.data, u2.ctypes.data, d2.ctypes.data)
    assert np.array_equal(g, g2) and np.array_equal(u, u2) and np.array_equal(d, d2)
    # documented layout: gate row r, block b -> tile g = r // 32, lane = r % 32, tile block
    # (g, b) at (g * nb + b) * TBB: codes (piece p of lane l at 512 p + 16 ((l + 4 p) % 32)), then the scale
    # entries with lane l at position 4 (l % 8) + l // 8
    nb = 2
    r, b = 37, 1
    blk = g[(r * nb + b) * BB:(r * nb + b + 1) * BB]
    tile, lane = r // 32, r % 32
    pos = 4 * (lane % 8) + lane // 8
    if qtype == 0:
        tb = (tile * nb + b) * 1088
        q_off = tb + 512 + ((lane + 4) % 32) * 16  # second piece of the block: codes 16..31
        assert np.array_equal(view[q_off:q_off + 16], blk[2 + 16:2 + 32] ^ 0x80)
        s_off = tb + 1024 + pos * 2
        assert np.array_equal(view[s_off:s_off + 2], blk[0:2])
    else:
        tb = (tile * nb + b) * 640
        q_off = tb + lane * 16
        assert np.array_equal(view[q_off:q_off + 16], blk[4:20])
        s_off = tb + 512 + pos * 4
        assert np.array_equal(view[s_off:s_off + 4], blk[0:4])


def test_slot_budget_matches_page_numbers(lib):
    MiB = 1 << 20
    per = [3059712, 2654208]
    rc, slots = L.moe_slots_for_budget(10000 * MiB, per, 8)
    assert rc == 0 and abs(slots[0] - 1834) <= 1 and slots[0] == slots[1]
    rc, _ = L.moe_slots_for_budget(50 * MiB, per, 8)
    assert rc == 0
    rc, slots = L.moe_slots_for_budget(49 * MiB, per, 8)
    assert rc == L.MOE_ERR_BUDGET and slots == [0, 0]


def test_argument_validation_happens_before_device_work(lib):
    ids = (ctypes.c_int32 * 16)()
    w = (ctypes.c_float * 16)()
    x = (ctypes.c_float * 256)()
    wr = (ctypes.c_uint16 * 2048)()
    # k > E, k > MOE_MAX_K, H not a multiple of 32, bad xtype
    assert lib.moe_router_topk(x, 0, 1, 256, wr, None, 4, 5, ids, w, None, None) == L.MOE_ERR_INVALID
    assert lib.moe_router_topk(x, 0, 1, 256, wr, None, 16, 9, ids, w, None, None) == L.MOE_ERR_INVALID
    assert lib.moe_router_topk(x, 0, 1, 250, wr, None, 8, 2, ids, w, None, None) == L.MOE_ERR_INVALID
    assert lib.moe_router_topk(x, 3, 1, 256, wr, None, 8, 2, ids, w, None, None) == L.MOE_ERR_INVALID
    # T == 0 is a no-op
    assert lib.moe_router_topk(None, 0, 0, 256, None, None, 8, 2, None, None, None, None) == 0
    # expert FFN: null pool, unaligned slot stride, bad qtype
    assert lib.moe_expert_ffn(x, 0, 1, 256, 512, 0, 8, 2, ids, w, None, 8, None, 417792, None, 0,
                              x, x, 1 << 20, None) == L.MOE_ERR_INVALID
    assert lib.moe_expert_ffn(x, 0, 1, 256, 512, 5, 8, 2, ids, w, None, 8, x, 417792, None, 0,
                              x, x, 1 << 20, None) == L.MOE_ERR_INVALID
    # combine: H not a multiple of 4
    assert lib.moe_combine(x, 1, 2, 6, None, x, None) == L.MOE_ERR_INVALID
    # cache: null descriptor pieces
    desc = L.CacheDesc(qtype=0, H=256, F=512, n_layers=1, n_experts=8, first_layer=0, n_slots=0,
                       slot_bytes=417792, device_pool=None, host_images=None, copy_stream=None)
    out = ctypes.c_void_p()
    assert lib.moe_cache_create(ctypes.byref(desc), ctypes.byref(out)) == L.MOE_ERR_INVALID
    # fault injection hook validates its arguments and never touches the GPU
    assert lib.moe_debug_inject_fault(7, 0) == L.MOE_ERR_INVALID
    assert lib.moe_debug_inject_fault(0, 0) == 0


def test_workspace_sizes(lib):
    # the decode workspace holds the route lists and the K-split gate/up partial sums
    n1 = L.moe_expert_ffn_workspace(1, 2048, 768, 1, 0, 128, 8)
    n8 = L.moe_expert_ffn_workspace(8, 2048, 768, 1, 0, 128, 8)
    # above the decode limit: bf16 activations take the grouped-GEMM path (its own sizing)
    assert L.moe_expert_ffn_workspace(512, 2048, 768, 1, 1, 128, 8) != \
        L.moe_expert_ffn_workspace(512, 2048, 768, 1, 0, 128, 8)
    assert n8 > n1 > 0 and n8 % 256 == 0
    assert L.moe_stack_workspace(1024, 512, 0, 32, 8, 8, 0) > n8 // 100


def test_ctypes_structs_match_the_c_header(tmp_path):
    """Every struct the binding mirrors has the C header's size and field offsets (compiled
    with the host C compiler from include/moe.h)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    pairs = [(L.CacheDesc, "moe_cache_desc"), (L.CacheStats, "moe_cache_stats"),
             (L.StackDesc, "moe_stack_desc"), (L.StackProfile, "moe_stack_profile"),
             (L.GemvTiming, "moe_gemv_timing")]
    lines = ["#include <stdio.h>", "#include <stddef.h>", '#include "moe.h"', "int main(void) {"]
    for cls, cname in pairs:
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for f in cls._fields_:
            lines.append(f'printf("{cname} {f[0]} %zu\\n", offsetof({cname}, {f[0]}));')
    lines += ["return 0;", "}"]
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    c = {" ".join(l.split()[:2]): int(l.split()[2]) for l in out if l.strip()}
    for cls, cname in pairs:
        assert c[f"{cname} size"] == ctypes.sizeof(cls), cname
        for f in cls._fields_:
            assert c[f"{cname} {f[0]}"] == getattr(cls, f[0]).offset, (cname, f[0])


def test_decode_gemv_mode_switch(lib):
    """The process-wide choice between the fused GEMV launch and the separate kernels."""
    before = L.moe_get_decode_fused()
    try:
        L.moe_set_decode_fused(True)
        assert L.moe_get_decode_fused() is True
        L.moe_set_decode_fused(False)
        assert L.moe_get_decode_fused() is False
    finally:
        L.moe_set_decode_fused(before)


def test_stack_workspace_covers_every_batch_up_to_max_T():
    """The decode FFN workspace is not monotonic in the token count (the K split of the gate/up
    GEMV is chosen per count): a stack sized for max_T must hold the FFN workspace of every
    smaller batch (the Qwen-shaped layer needs more at 27 tokens than at 32)."""
    for (q, H, F, E, k, ns) in [(1, 2048, 768, 128, 8, 0), (0, 1024, 512, 32, 8, 0), (0, 2048, 1408, 64, 2, 2)]:
        for max_T in (1, 8, 32):
            stack = L.moe_stack_workspace(H, F, q, E, k, max_T, ns)
            need = max(L.moe_expert_ffn_workspace(t, H, F, q, 0, E, k) for t in range(1, max_T + 1))
            assert stack > need, (q, H, F, E, k, max_T)
