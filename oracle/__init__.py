"""CPU oracle for the routed-expert MoE FFN layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product library never does, and
this package never imports the product package (inputs come in as arrays).

Parts:
  * ``moe_oracle.c`` (fp64 C, built by ``oracle/build.py``): exact dequantisation,
    router logits, top-k + softmax, per-expert SwiGLU FFN.
  * this module: ctypes wrappers and the layer / stack composition in the order
    the method states (router -> top-k -> softmax over the selected -> expert
    FFNs -> weighted sum (+ shared experts) -> residual for stacks).
  * ``lru_sim.py``: the slot-pool LRU replayed in pure Python.

Parity status: every function here is pinned by a ``-m "not gpu"`` test against
something other than itself (numpy decoders and matmuls, closed forms,
hand-built traces, the pages' printed numbers).
"""
from __future__ import annotations

import ctypes
import os
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np

from . import build as _build

_lib: Optional[ctypes.CDLL] = None

_D = ctypes.POINTER(ctypes.c_double)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_U16 = ctypes.POINTER(ctypes.c_uint16)
_I32 = ctypes.POINTER(ctypes.c_int32)


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_fp16_to_double.restype = ctypes.c_double
        L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_double.restype = ctypes.c_double
        L.oracle_dequant_q8_0.argtypes = [_U8, ctypes.c_int64, _D]
        L.oracle_dequant_q4.argtypes = [_U8, ctypes.c_int64, _D]
        L.oracle_qmatvec.argtypes = [ctypes.c_int, _U8, ctypes.c_int, ctypes.c_int, _D, _D]
        L.oracle_router_logits.argtypes = [_D, ctypes.c_int, ctypes.c_int, _U16, _D, ctypes.c_int, _D]
        L.oracle_topk_softmax.argtypes = [_D, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I32, _D, _D]
        L.oracle_silu.argtypes = [ctypes.c_double]
        L.oracle_silu.restype = ctypes.c_double
        L.oracle_expert_ffn.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, _U8, _U8, _U8,
                                        _D, _D, _D]
        L.oracle_num_threads.restype = ctypes.c_int
        L.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = L
    return _lib


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_num_threads(n: int) -> None:
    lib().oracle_set_num_threads(int(n))


# ------------------------------------------------------------------------------ scalars / blocks

def fp16_to_double(bits: int) -> float:
    return float(lib().oracle_fp16_to_double(int(bits)))


def bf16_to_double(bits: int) -> float:
    return float(lib().oracle_bf16_to_double(int(bits)))


def dequant(qtype: int, blocks: np.ndarray) -> np.ndarray:
    """Exact fp64 dequantisation of a run of canonical blocks (q8_0: 34 B, 4-bit: 20 B)."""
    b = np.ascontiguousarray(blocks, dtype=np.uint8)
    bsz = 34 if qtype == 0 else 20
    nb = b.size // bsz
    out = np.empty(nb * 32, dtype=np.float64)
    fn = lib().oracle_dequant_q8_0 if qtype == 0 else lib().oracle_dequant_q4
    fn(_p(b, _U8), nb, _p(out, _D))
    return out


def qmatvec(qtype: int, mat: np.ndarray, rows: int, cols: int, x: np.ndarray) -> np.ndarray:
    m = np.ascontiguousarray(mat, dtype=np.uint8)
    xv = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(rows, dtype=np.float64)
    lib().oracle_qmatvec(qtype, _p(m, _U8), rows, cols, _p(xv, _D), _p(y, _D))
    return y


def silu(z: float) -> float:
    return float(lib().oracle_silu(float(z)))


# ------------------------------------------------------------------------------ router

def x_to_double(x: np.ndarray, xtype: int) -> np.ndarray:
    """Input activations as exact fp64 (fp32 values, or bf16 bit patterns when xtype == 1)."""
    if xtype == 1:
        u = np.asarray(x, dtype=np.uint16).astype(np.uint32) << 16
        return u.view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float32).astype(np.float64)


def router_logits(x: np.ndarray, w_router_bits: np.ndarray, bias: Optional[np.ndarray]) -> np.ndarray:
    xd = np.ascontiguousarray(x, dtype=np.float64)
    T, H = xd.shape
    w = np.ascontiguousarray(w_router_bits, dtype=np.uint16)
    E = w.shape[1]
    assert w.shape[0] == H
    out = np.empty((T, E), dtype=np.float64)
    bd = None if bias is None else np.ascontiguousarray(bias, dtype=np.float64)
    lib().oracle_router_logits(_p(xd, _D), T, H, _p(w, _U16),
                               None if bd is None else _p(bd, _D), E, _p(out, _D))
    return out


def topk_softmax(logits: np.ndarray, k: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(ids [T][k] int32, weights [T][k] fp64, gap [T] fp64) from fp64 logits."""
    l = np.ascontiguousarray(logits, dtype=np.float64)
    T, E = l.shape
    assert 1 <= k <= E <= 4096
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    gap = np.empty(T, dtype=np.float64)
    lib().oracle_topk_softmax(_p(l, _D), T, E, k, _p(ids, _I32), _p(w, _D), _p(gap, _D))
    return ids, w, gap


# ------------------------------------------------------------------------------ experts

def expert_ffn(qtype: int, H: int, F: int, gate: np.ndarray, up: np.ndarray, down: np.ndarray,
               x: np.ndarray) -> np.ndarray:
    """y = W_down (silu(W_gate x) * (W_up x)) for one token, fp64."""
    g = np.ascontiguousarray(gate, dtype=np.uint8)
    u = np.ascontiguousarray(up, dtype=np.uint8)
    d = np.ascontiguousarray(down, dtype=np.uint8)
    xv = np.ascontiguousarray(x, dtype=np.float64)
    assert xv.shape == (H,)
    y = np.empty(H, dtype=np.float64)
    scratch = np.empty(3 * F, dtype=np.float64)
    lib().oracle_expert_ffn(qtype, H, F, _p(g, _U8), _p(u, _U8), _p(d, _U8), _p(xv, _D),
                            _p(y, _D), _p(scratch, _D))
    return y


ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


class LayerResult:
    """Oracle result for one MoE layer on T tokens."""

    def __init__(self, logits, ids, weights, gap, y_experts, y):
        self.logits = logits      # [T][E] fp64
        self.ids = ids            # [T][k] int32
        self.weights = weights    # [T][k] fp64
        self.gap = gap            # [T] fp64 margin between k-th and (k+1)-th logit
        self.y_experts = y_experts  # [T][k][H] fp64 unweighted expert outputs
        self.y = y                # [T][H] fp64: sum_j w_j y_j + sum_s y_s


def moe_layer(qtype: int, H: int, F: int, k: int, x: np.ndarray, w_router_bits: np.ndarray,
              bias: Optional[np.ndarray], experts: ExpertFn,
              shared: Sequence[Tuple[np.ndarray, np.ndarray, np.ndarray]] = (),
              route_override: Optional[Tuple[np.ndarray, np.ndarray]] = None,
              load_threshold: float = 0.0) -> LayerResult:
    """One MoE FFN layer, in the method's order.

    x: [T][H] fp64 (exact input values).  ``experts(e)`` returns expert e's canonical
    (gate, up, down) blocks.  ``route_override`` = (ids, weights) replaces the oracle's
    own routing (used to check outputs on near-tie tokens with a given route); an id of -1
    there is a dropped route.  ``load_threshold`` (page 1, "MoE 模型卸载" blog, section 4.3:
    experts whose gate score is below the threshold are not loaded): a selected route whose
    softmax weight is below it is dropped — not computed, its term left out of the sum,
    the other weights unchanged; its id becomes -1 and its weight 0 in the result.
    """
    xd = np.ascontiguousarray(x, dtype=np.float64)
    T = xd.shape[0]
    logits = router_logits(xd, w_router_bits, bias)
    ids, w, gap = topk_softmax(logits, k)
    if load_threshold > 0.0:
        drop = w < load_threshold
        ids = np.where(drop, -1, ids).astype(np.int32)
        w = np.where(drop, 0.0, w)
    if route_override is not None:
        ids = np.asarray(route_override[0], dtype=np.int32)
        w = np.asarray(route_override[1], dtype=np.float64)
    cache = {}
    y_exp = np.zeros((T, k, H), dtype=np.float64)
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue  # a dropped route
            if e not in cache:
                cache[e] = experts(e)
            gt, ut, dt = cache[e]
            y_exp[t, j] = expert_ffn(qtype, H, F, gt, ut, dt, xd[t])
        for j in range(k):
            if ids[t, j] >= 0:
                y[t] += w[t, j] * y_exp[t, j]
        for (gs, us, ds) in shared:
            y[t] += expert_ffn(qtype, H, F, gs, us, ds, xd[t])
    return LayerResult(logits, ids, w, gap, y_exp, y)


STACK_EPS = 1e-6


def rmsnorm(h: np.ndarray, eps: float = STACK_EPS) -> np.ndarray:
    """Per-row RMS normalisation with unit weight: h / sqrt(mean(h^2) + eps), fp64.

    The stacks feed each layer's MoE FFN the normalised residual stream (pre-norm), so
    that every layer sees inputs of unit scale; the pages fix no normalisation.
    """
    h = np.asarray(h, dtype=np.float64)
    return h / np.sqrt(np.mean(h * h, axis=-1, keepdims=True) + eps)


def relative_error(y: np.ndarray, y_ref: np.ndarray) -> np.ndarray:
    """Per-token normwise error max_i |y_i - ref_i| / max_i |ref_i| (rows of [T][H])."""
    y = np.asarray(y, dtype=np.float64).reshape(y_ref.shape)
    num = np.max(np.abs(y - y_ref), axis=-1)
    den = np.max(np.abs(y_ref), axis=-1)
    return num / np.where(den > 0, den, 1.0)
