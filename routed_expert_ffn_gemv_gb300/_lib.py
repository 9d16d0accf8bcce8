"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  Device buffers are
torch tensors (their ``data_ptr()`` is passed), streams are ``torch.cuda.Stream``
objects (or None for the current stream).  A non-zero status raises ``MoeError``.
The library must be built (``routed_expert_ffn_gemv_gb300._build``); there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from . import _build

MOE_OK = 0
MOE_ERR_INVALID = -1
MOE_ERR_CUDA = -2
MOE_ERR_CAPACITY = -3
MOE_ERR_BUDGET = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_UNSUPPORTED = -6
MOE_Q8_0 = 0
MOE_Q4_SM = 1
MOE_F32 = 0
MOE_BF16 = 1
MOE_MAX_K = 8
MOE_MAX_E = 256
MOE_DECODE_MAX_T = 32

EXPORTED = [
    "moe_status_string", "moe_router_topk", "moe_slot_image_bytes", "moe_pack_expert",
    "moe_unpack_expert", "moe_cache_create", "moe_cache_ensure", "moe_cache_wait_uploads",
    "moe_cache_release", "moe_cache_stats_get", "moe_cache_reset", "moe_cache_destroy",
    "moe_cache_lookup", "moe_slots_for_budget", "moe_expert_ffn", "moe_expert_ffn_workspace",
    "moe_combine", "moe_device_status", "moe_stack_workspace", "moe_stack_create",
    "moe_stack_decode", "moe_stack_layer", "moe_stack_profile_get", "moe_stack_profile_reset",
    "moe_stack_destroy", "moe_debug_inject_fault", "moe_stack_set_profile", "moe_stack_gemv_timing",
    "moe_set_decode_fused", "moe_get_decode_fused",
    "moe_expert_ffn_noalloc", "moe_combine_rmsnorm", "moe_cache_state_bytes", "moe_cache_plan",
    "moe_expert_ffn_fill", "moe_last_cuda_error", "moe_router_topk_threshold",
    "moe_cache_prefetch_plan", "moe_cache_prefetch_fill",
]
MOE_NOALLOC_SCRATCH_MAX = 8 << 20


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = f", {load().moe_last_cuda_error().decode()}" if status == MOE_ERR_CUDA else ""
        super().__init__(f"{fn} failed: {status} ({status_string(status)}{detail})")


_vp = ctypes.c_void_p
_sz = ctypes.c_size_t
_i = ctypes.c_int


class CacheDesc(ctypes.Structure):
    _fields_ = [("qtype", _i), ("H", _i), ("F", _i), ("n_layers", _i), ("n_experts", _i),
                ("first_layer", _i), ("n_slots", _i), ("slot_bytes", _sz), ("device_pool", _vp),
                ("host_images", ctypes.POINTER(_vp)), ("copy_stream", _vp), ("device_managed", _i),
                ("device_state", _vp), ("device_state_bytes", _sz), ("admit_after", _i),
                ("lru_window", _i)]


class CacheStats(ctypes.Structure):
    _fields_ = [("queries", ctypes.c_uint64 * 2), ("hits", ctypes.c_uint64 * 2),
                ("misses", ctypes.c_uint64 * 2), ("evictions", ctypes.c_uint64),
                ("h2d_bytes", ctypes.c_uint64), ("route_queries", ctypes.c_uint64),
                ("route_hits", ctypes.c_uint64), ("ensure_calls", ctypes.c_uint64),
                ("bypassed", ctypes.c_uint64), ("window_evictions", ctypes.c_uint64),
                ("prefetch_queries", ctypes.c_uint64), ("prefetch_hits", ctypes.c_uint64),
                ("prefetch_fills", ctypes.c_uint64), ("prefetch_aborts", ctypes.c_uint64)]

    def as_dict(self):
        return {"queries": list(self.queries), "hits": list(self.hits), "misses": list(self.misses),
                "evictions": self.evictions, "h2d_bytes": self.h2d_bytes,
                "route_queries": self.route_queries, "route_hits": self.route_hits,
                "ensure_calls": self.ensure_calls, "bypassed": self.bypassed,
                "window_evictions": self.window_evictions, "prefetch_queries": self.prefetch_queries,
                "prefetch_hits": self.prefetch_hits, "prefetch_fills": self.prefetch_fills,
                "prefetch_aborts": self.prefetch_aborts}


class StackDesc(ctypes.Structure):
    _fields_ = [("qtype", _i), ("H", _i), ("F", _i), ("E", _i), ("k", _i), ("n_layers", _i),
                ("n_shared", _i), ("w_router", ctypes.POINTER(_vp)), ("bias", ctypes.POINTER(_vp)),
                ("n_groups", _i), ("caches", ctypes.POINTER(_vp)), ("resident_pool", _vp),
                ("shared_pool", _vp), ("slot_bytes", _sz), ("max_T", _i), ("workspace", _vp),
                ("ws_bytes", _sz), ("overlap", _i), ("profile", _i), ("device_managed", _i),
                ("use_graph", _i), ("load_threshold", ctypes.c_float), ("prefetch_depth", _i)]


class StackProfile(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_uint64), ("layers", ctypes.c_uint64),
                ("router_ms", ctypes.c_double), ("permute_ms", ctypes.c_double),
                ("gateup_ms", ctypes.c_double), ("down_ms", ctypes.c_double),
                ("combine_ms", ctypes.c_double), ("gateup_launches", ctypes.c_uint64),
                ("down_launches", ctypes.c_uint64), ("gateup_bytes", ctypes.c_double),
                ("down_bytes", ctypes.c_double), ("host_wait_ms", ctypes.c_double),
                ("kernel_launches", ctypes.c_uint64), ("h2d_copies", ctypes.c_uint64)]

    def as_dict(self):
        return {f[0]: getattr(self, f[0]) for f in self._fields_}


class GemvTiming(ctypes.Structure):
    _fields_ = [("gateup_us", ctypes.c_double), ("down_us", ctypes.c_double),
                ("gateup_bytes", ctypes.c_double), ("down_bytes", ctypes.c_double), ("launches", _i),
                ("reduce_us", ctypes.c_double), ("gemv_us", ctypes.c_double), ("fused", _i)]

    def as_dict(self):
        return {f[0]: getattr(self, f[0]) for f in self._fields_}


_lib: Optional[ctypes.CDLL] = None


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load the in-tree libmoe.so (building it first if needed)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing and not _build.up_to_date():
        path = _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libmoe.so is not built ({path}); run routed_expert_ffn_gemv_gb300._build")
    L = ctypes.CDLL(path)
    P = ctypes.POINTER
    sig = {
        "moe_status_string": ([_i], ctypes.c_char_p),
        "moe_last_cuda_error": ([], ctypes.c_char_p),
        "moe_router_topk": ([_vp, _i, _i, _i, _vp, _vp, _i, _i, _vp, _vp, _vp, _vp], _i),
        "moe_router_topk_threshold": ([_vp, _i, _i, _i, _vp, _vp, _i, _i, ctypes.c_float, _vp, _vp, _vp, _vp], _i),
        "moe_slot_image_bytes": ([_i, _i, _i, P(_sz)], _i),
        "moe_pack_expert": ([_i, _i, _i, _vp, _vp, _vp, _vp, P(_sz)], _i),
        "moe_unpack_expert": ([_i, _i, _i, _vp, _vp, _vp, _vp], _i),
        "moe_cache_create": ([P(CacheDesc), P(_vp)], _i),
        "moe_cache_ensure": ([_vp, _i, _vp, _i, _i, _vp, P(_i), _vp, _vp, _vp], _i),
        "moe_cache_wait_uploads": ([_vp, _vp], _i),
        "moe_cache_release": ([_vp, _vp], _i),
        "moe_cache_stats_get": ([_vp, P(CacheStats)], _i),
        "moe_cache_reset": ([_vp], _i),
        "moe_cache_destroy": ([_vp], None),
        "moe_cache_lookup": ([_vp, _i, _i], _i),
        "moe_slots_for_budget": ([_sz, P(_sz), _i, _i, P(_i)], _i),
        "moe_expert_ffn": ([_vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _sz, _vp, _i,
                            _vp, _vp, _sz, _vp], _i),
        "moe_expert_ffn_workspace": ([_i, _i, _i, _i, _i, _i, _i, P(_sz)], _i),
        "moe_expert_ffn_noalloc": ([_vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _sz, _vp,
                                    _i, _vp, _vp], _i),
        "moe_combine": ([_vp, _i, _i, _i, _vp, _vp, _vp], _i),
        "moe_combine_rmsnorm": ([_vp, _i, _i, _i, _vp, _vp, _vp, ctypes.c_float, _vp], _i),
        "moe_cache_state_bytes": ([_i, _i, _i, P(_sz)], _i),
        "moe_cache_plan": ([_vp, _i, _vp, _i, _i, _vp, _vp, _vp], _i),
        "moe_cache_prefetch_plan": ([_vp, _i, _vp, _i, _i, _vp, _vp, _vp], _i),
        "moe_cache_prefetch_fill": ([_vp, _vp, _vp, _vp], _i),
        "moe_expert_ffn_fill": ([_vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _i, _vp, _sz, _vp, _vp, _vp,
                                 _sz, _vp], _i),
        "moe_device_status": ([P(_i), _i], _i),
        "moe_stack_workspace": ([_i, _i, _i, _i, _i, _i, _i, P(_sz)], _i),
        "moe_stack_create": ([P(StackDesc), P(_vp)], _i),
        "moe_stack_decode": ([_vp, _vp, _vp, _i, _vp, _vp, _vp], _i),
        "moe_stack_layer": ([_vp, _i, _vp, _vp, _i, _vp, _vp, _vp], _i),
        "moe_stack_profile_get": ([_vp, P(StackProfile)], _i),
        "moe_stack_profile_reset": ([_vp], _i),
        "moe_stack_destroy": ([_vp], None),
        "moe_stack_set_profile": ([_vp, _i], _i),
        "moe_stack_gemv_timing": ([_vp, _vp, _i, _i, P(GemvTiming), _vp], _i),
        "moe_set_decode_fused": ([_i], _i),
        "moe_get_decode_fused": ([], _i),
        "moe_debug_inject_fault": ([_i, _i], _i),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def status_string(status: int) -> str:
    return load().moe_status_string(int(status)).decode()


def _ck(fn: str, rc: int) -> int:
    if rc != MOE_OK:
        raise MoeError(fn, rc)
    return rc


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ------------------------------------------------------------------------------ entry points

def moe_router_topk(x, xtype: int, T: int, H: int, w_router, bias, E: int, k: int, ids, weights,
                    logits=None, stream=None) -> None:
    _ck("moe_router_topk", load().moe_router_topk(_ptr(x), xtype, T, H, _ptr(w_router), _ptr(bias), E, k,
                                                  _ptr(ids), _ptr(weights), _ptr(logits), _stream(stream)))


def moe_router_topk_threshold(x, xtype: int, T: int, H: int, w_router, bias, E: int, k: int, min_weight: float,
                              ids, weights, logits=None, stream=None) -> None:
    _ck("moe_router_topk_threshold",
        load().moe_router_topk_threshold(_ptr(x), xtype, T, H, _ptr(w_router), _ptr(bias), E, k, float(min_weight),
                                         _ptr(ids), _ptr(weights), _ptr(logits), _stream(stream)))


def moe_slot_image_bytes(qtype: int, H: int, F: int) -> int:
    out = _sz()
    _ck("moe_slot_image_bytes", load().moe_slot_image_bytes(qtype, H, F, ctypes.byref(out)))
    return out.value


def moe_pack_expert(qtype: int, H: int, F: int, gate_ptr: int, up_ptr: int, down_ptr: int,
                    dst_ptr: int) -> int:
    out = _sz()
    _ck("moe_pack_expert", load().moe_pack_expert(qtype, H, F, gate_ptr, up_ptr, down_ptr, dst_ptr,
                                                  ctypes.byref(out)))
    return out.value


def moe_unpack_expert(qtype: int, H: int, F: int, src_ptr: int, gate_ptr: int, up_ptr: int,
                      down_ptr: int) -> None:
    _ck("moe_unpack_expert", load().moe_unpack_expert(qtype, H, F, src_ptr, gate_ptr, up_ptr, down_ptr))


def moe_cache_create(desc: CacheDesc) -> int:
    out = _vp()
    _ck("moe_cache_create", load().moe_cache_create(ctypes.byref(desc), ctypes.byref(out)))
    return out.value


def moe_cache_ensure(cache: int, layer: int, ids_host_ptr: int, n_tokens: int, k: int,
                     slots_host_ptr: int, miss_mask_ptr: Optional[int], d_slot_table, stream=None) -> int:
    n_miss = _i()
    _ck("moe_cache_ensure", load().moe_cache_ensure(cache, layer, ids_host_ptr, n_tokens, k,
                                                    slots_host_ptr, ctypes.byref(n_miss), miss_mask_ptr,
                                                    _ptr(d_slot_table), _stream(stream)))
    return n_miss.value


def moe_cache_ensure_status(cache: int, layer: int, ids_host_ptr: int, n_tokens: int, k: int,
                            slots_host_ptr: int, d_slot_table=None, stream=None) -> int:
    """Like moe_cache_ensure but returns the raw status (for error-path tests)."""
    n_miss = _i()
    return load().moe_cache_ensure(cache, layer, ids_host_ptr, n_tokens, k, slots_host_ptr,
                                   ctypes.byref(n_miss), None, _ptr(d_slot_table), _stream(stream))


def moe_cache_state_bytes(n_layers: int, n_experts: int, n_slots: int) -> int:
    out = _sz()
    _ck("moe_cache_state_bytes", load().moe_cache_state_bytes(n_layers, n_experts, n_slots, ctypes.byref(out)))
    return out.value


def moe_cache_plan(cache: int, layer: int, d_ids, n_tokens: int, k: int, d_table, d_fill_src,
                   stream=None) -> None:
    _ck("moe_cache_plan", load().moe_cache_plan(cache, layer, _ptr(d_ids), n_tokens, k, _ptr(d_table),
                                                _ptr(d_fill_src), _stream(stream)))


def moe_cache_prefetch_plan(cache: int, layer: int, d_ids, n_tokens: int, k: int, d_table, d_fill_src,
                            stream=None) -> None:
    _ck("moe_cache_prefetch_plan", load().moe_cache_prefetch_plan(cache, layer, _ptr(d_ids), n_tokens, k,
                                                                  _ptr(d_table), _ptr(d_fill_src), _stream(stream)))


def moe_cache_prefetch_fill(cache: int, d_table, d_fill_src, stream=None) -> None:
    _ck("moe_cache_prefetch_fill", load().moe_cache_prefetch_fill(cache, _ptr(d_table), _ptr(d_fill_src),
                                                                  _stream(stream)))


def moe_expert_ffn_fill(x, xtype: int, T: int, H: int, F: int, qtype: int, E: int, k: int, ids, weights,
                        d_slot_table, n_slots: int, pool, slot_bytes: int, d_fill_src, partial, workspace,
                        ws_bytes: int, stream=None) -> None:
    _ck("moe_expert_ffn_fill",
        load().moe_expert_ffn_fill(_ptr(x), xtype, T, H, F, qtype, E, k, _ptr(ids), _ptr(weights),
                                   _ptr(d_slot_table), n_slots, _ptr(pool), slot_bytes, _ptr(d_fill_src),
                                   _ptr(partial), _ptr(workspace), ws_bytes, _stream(stream)))


def moe_cache_wait_uploads(cache: int, stream=None) -> None:
    _ck("moe_cache_wait_uploads", load().moe_cache_wait_uploads(cache, _stream(stream)))


def moe_cache_release(cache: int, stream=None) -> None:
    _ck("moe_cache_release", load().moe_cache_release(cache, _stream(stream)))


def moe_cache_stats_get(cache: int) -> dict:
    st = CacheStats()
    _ck("moe_cache_stats_get", load().moe_cache_stats_get(cache, ctypes.byref(st)))
    return st.as_dict()


def moe_cache_reset(cache: int) -> None:
    _ck("moe_cache_reset", load().moe_cache_reset(cache))


def moe_cache_destroy(cache: int) -> None:
    load().moe_cache_destroy(cache)


def moe_cache_lookup(cache: int, layer: int, expert: int) -> int:
    return int(load().moe_cache_lookup(cache, layer, expert))


def moe_slots_for_budget(budget_bytes: int, per_expert_bytes: Sequence[int], k: int):
    n = len(per_expert_bytes)
    arr = (_sz * n)(*per_expert_bytes)
    out = (_i * n)()
    rc = load().moe_slots_for_budget(budget_bytes, arr, n, k, out)
    return rc, list(out)


def moe_expert_ffn(x, xtype: int, T: int, H: int, F: int, qtype: int, E: int, k: int, ids, weights,
                   d_slot_table, n_slots: int, pool, slot_bytes: int, expert_subset, n_subset: int,
                   partial, workspace, ws_bytes: int, stream=None) -> None:
    _ck("moe_expert_ffn", load().moe_expert_ffn(_ptr(x), xtype, T, H, F, qtype, E, k, _ptr(ids),
                                                _ptr(weights), _ptr(d_slot_table), n_slots, _ptr(pool),
                                                slot_bytes, _ptr(expert_subset), n_subset, _ptr(partial),
                                                _ptr(workspace), ws_bytes, _stream(stream)))


def moe_expert_ffn_workspace(T: int, H: int, F: int, qtype: int, xtype: int, E: int, k: int) -> int:
    out = _sz()
    _ck("moe_expert_ffn_workspace", load().moe_expert_ffn_workspace(T, H, F, qtype, xtype, E, k,
                                                                    ctypes.byref(out)))
    return out.value


def moe_expert_ffn_noalloc(x, xtype: int, T: int, H: int, F: int, qtype: int, E: int, k: int, ids,
                           weights, d_slot_table, n_slots: int, pool, slot_bytes: int, expert_subset,
                           n_subset: int, partial, stream=None) -> None:
    _ck("moe_expert_ffn_noalloc",
        load().moe_expert_ffn_noalloc(_ptr(x), xtype, T, H, F, qtype, E, k, _ptr(ids), _ptr(weights),
                                      _ptr(d_slot_table), n_slots, _ptr(pool), slot_bytes,
                                      _ptr(expert_subset), n_subset, _ptr(partial), _stream(stream)))


def moe_combine(partial, T: int, k: int, H: int, extra, y, stream=None) -> None:
    _ck("moe_combine", load().moe_combine(_ptr(partial), T, k, H, _ptr(extra), _ptr(y), _stream(stream)))


def moe_combine_rmsnorm(partial, T: int, k: int, H: int, extra, y, xn, eps: float = 1e-6,
                        stream=None) -> None:
    _ck("moe_combine_rmsnorm", load().moe_combine_rmsnorm(_ptr(partial), T, k, H, _ptr(extra), _ptr(y), _ptr(xn),
                                                          eps, _stream(stream)))


def moe_device_status(clear: bool = True) -> int:
    out = _i()
    _ck("moe_device_status", load().moe_device_status(ctypes.byref(out), int(clear)))
    return out.value


def moe_stack_workspace(H: int, F: int, qtype: int, E: int, k: int, max_T: int, n_shared: int) -> int:
    out = _sz()
    _ck("moe_stack_workspace", load().moe_stack_workspace(H, F, qtype, E, k, max_T, n_shared, ctypes.byref(out)))
    return out.value


def moe_stack_create(desc: StackDesc) -> int:
    out = _vp()
    _ck("moe_stack_create", load().moe_stack_create(ctypes.byref(desc), ctypes.byref(out)))
    return out.value


def moe_stack_decode(stack: int, x, y, T: int, ids_host_ptr=None, weights_host_ptr=None, stream=None) -> None:
    _ck("moe_stack_decode", load().moe_stack_decode(stack, _ptr(x), _ptr(y), T, ids_host_ptr,
                                                    weights_host_ptr, _stream(stream)))


def moe_stack_layer(stack: int, layer: int, x, y, T: int, ids_host_ptr=None, weights_host_ptr=None,
                    stream=None) -> None:
    _ck("moe_stack_layer", load().moe_stack_layer(stack, layer, _ptr(x), _ptr(y), T, ids_host_ptr,
                                                  weights_host_ptr, _stream(stream)))


def moe_stack_profile_get(stack: int) -> dict:
    p = StackProfile()
    _ck("moe_stack_profile_get", load().moe_stack_profile_get(stack, ctypes.byref(p)))
    return p.as_dict()


def moe_stack_profile_reset(stack: int) -> None:
    _ck("moe_stack_profile_reset", load().moe_stack_profile_reset(stack))


def moe_stack_set_profile(stack: int, level: int) -> None:
    _ck("moe_stack_set_profile", load().moe_stack_set_profile(stack, level))


def moe_stack_gemv_timing(stack: int, x, T: int, reps: int, stream=None) -> dict:
    t = GemvTiming()
    _ck("moe_stack_gemv_timing", load().moe_stack_gemv_timing(stack, _ptr(x), T, reps, ctypes.byref(t),
                                                              _stream(stream)))
    return t.as_dict()


def moe_set_decode_fused(on: bool) -> None:
    _ck("moe_set_decode_fused", load().moe_set_decode_fused(1 if on else 0))


def moe_get_decode_fused() -> bool:
    return bool(load().moe_get_decode_fused())


def moe_stack_destroy(stack: int) -> None:
    load().moe_stack_destroy(stack)


def moe_debug_inject_fault(kind: int, countdown: int = 0) -> None:
    _ck("moe_debug_inject_fault", load().moe_debug_inject_fault(kind, countdown))
