"""Materialise a synthetic MoE stack for the C-ABI: pinned slot images, slot pools,
router weights, and a moe_stack.

Device memory and streams come from PyTorch; every computation runs in libmoe.
"""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import os
from typing import Dict, List, Optional, Sequence

import numpy as np
import torch

from . import _lib as L
from . import synth


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def slot_stride(cfg: synth.MoEConfig) -> int:
    return _round_up(L.moe_slot_image_bytes(cfg.qtype, cfg.H, cfg.F), 256)


def pack_into(cfg: synth.MoEConfig, layer: int, expert: int, dst_ptr: int,
              random_scales: bool = False) -> None:
    g, u, d = synth.expert_weights(cfg, layer, expert, random_scales)
    L.moe_pack_expert(cfg.qtype, cfg.H, cfg.F, g.ctypes.data, u.ctypes.data, d.ctypes.data, dst_ptr)


class PinnedImages:
    """All routed (and shared) expert slot images of a config in one pinned host buffer."""

    def __init__(self, cfg: synth.MoEConfig, layers: Sequence[int], experts: Sequence[int],
                 random_scales: bool = False, threads: Optional[int] = None):
        self.cfg = cfg
        self.stride = slot_stride(cfg)
        self.layers = list(layers)
        self.experts = list(experts)
        n = len(self.layers) * len(self.experts)
        self.buf = torch.empty(n * self.stride, dtype=torch.uint8, pin_memory=True)
        base = self.buf.data_ptr()
        jobs = [(li, ei) for li in range(len(self.layers)) for ei in range(len(self.experts))]

        def work(job):
            li, ei = job
            pack_into(cfg, self.layers[li], self.experts[ei],
                      base + (li * len(self.experts) + ei) * self.stride, random_scales)

        nthreads = threads or min(32, os.cpu_count() or 4)
        with cf.ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(work, jobs))

    def ptr(self, li: int, ei: int) -> int:
        return self.buf.data_ptr() + (li * len(self.experts) + ei) * self.stride


class Stack:
    """A full decode stack of one configuration on the current CUDA device.

    pool_slots: override the per-group slot counts (None: the configuration's); a config
    with no groups keeps every expert resident in one device pool.  admit_after / lru_window:
    the pools' policy variants (0: plain LRU; see moe_cache_desc).
    """

    def __init__(self, cfg: synth.MoEConfig, max_T: Optional[int] = None, overlap: bool = True,
                 profile: int = 0, pool_slots: Optional[Sequence[int]] = None,
                 n_layers: Optional[int] = None, random_scales: bool = False,
                 resident: bool = False, device_managed: bool = False, use_graph: bool = False,
                 images: Optional[PinnedImages] = None, admit_after: int = 0, lru_window: int = 0,
                 load_threshold: float = 0.0, prefetch_depth: int = 0):
        self.cfg = cfg
        self.L = n_layers or cfg.L
        self.max_T = max_T or max(cfg.tokens)
        assert self.max_T <= L.MOE_DECODE_MAX_T
        self.dev = torch.device("cuda", torch.cuda.current_device())
        self.stride = slot_stride(cfg)
        H, F, E, k = cfg.H, cfg.F, cfg.E, cfg.k
        # router weights / bias per layer
        self.w_router = [torch.from_numpy(synth.router_weights(cfg, l).view(np.int16)).to(self.dev)
                         for l in range(self.L)]
        self.bias = []
        for l in range(self.L):
            b = synth.router_bias(cfg, l)
            self.bias.append(None if b is None else torch.from_numpy(b).to(self.dev))
        # routed expert images (an existing set of the same config may be shared)
        if images is not None:
            assert images.cfg == cfg and images.layers[: self.L] == list(range(self.L))
            assert images.experts == list(range(E)) and not random_scales
            self.images = images
        else:
            self.images = PinnedImages(cfg, range(self.L), range(E), random_scales)
        self.caches: List[int] = []
        self.pools: List[torch.Tensor] = []
        self.states: List[torch.Tensor] = []
        self.device_managed = device_managed
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        groups = [] if resident else list(cfg.groups)
        self.resident_pool = None
        if not groups:
            self.resident_pool = torch.empty(self.L * E * self.stride, dtype=torch.uint8, device=self.dev)
            self.resident_pool.copy_(self.images.buf[: self.L * E * self.stride])
            torch.cuda.synchronize()
        else:
            for gi, grp in enumerate(groups):
                n_layers_g = min(grp.n_layers, self.L - grp.first_layer)
                if n_layers_g <= 0:
                    continue
                n_slots = pool_slots[gi] if pool_slots is not None else grp.n_slots
                pool = torch.empty(n_slots * self.stride, dtype=torch.uint8, device=self.dev)
                imgs = (ctypes.c_void_p * (n_layers_g * E))(
                    *[self.images.ptr(grp.first_layer + li, e) for li in range(n_layers_g) for e in range(E)])
                state, state_bytes = None, 0
                if device_managed:
                    state_bytes = L.moe_cache_state_bytes(n_layers_g, E, n_slots)
                    state = torch.empty(state_bytes, dtype=torch.uint8, device=self.dev)
                    self.states.append(state)
                desc = L.CacheDesc(qtype=cfg.qtype, H=H, F=F, n_layers=n_layers_g, n_experts=E,
                                   first_layer=grp.first_layer, n_slots=n_slots, slot_bytes=self.stride,
                                   device_pool=pool.data_ptr(),
                                   host_images=ctypes.cast(imgs, ctypes.POINTER(ctypes.c_void_p)),
                                   copy_stream=self.copy_stream.cuda_stream,
                                   device_managed=int(device_managed),
                                   device_state=None if state is None else state.data_ptr(),
                                   device_state_bytes=state_bytes, admit_after=admit_after,
                                   lru_window=lru_window)
                self.caches.append(L.moe_cache_create(desc))
                self.pools.append(pool)
        # shared experts (always resident)
        self.shared_pool = None
        if cfg.n_shared > 0:
            simg = PinnedImages(cfg, range(self.L), range(E, E + cfg.n_shared), random_scales)
            self.shared_pool = torch.empty(self.L * cfg.n_shared * self.stride, dtype=torch.uint8,
                                           device=self.dev)
            self.shared_pool.copy_(simg.buf)
        ws = L.moe_stack_workspace(H, F, cfg.qtype, E, k, self.max_T, cfg.n_shared)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=self.dev)
        self._wr = (ctypes.c_void_p * self.L)(*[w.data_ptr() for w in self.w_router])
        self._bias = (ctypes.c_void_p * self.L)(*[0 if b is None else b.data_ptr() for b in self.bias])
        self._caches = (ctypes.c_void_p * max(1, len(self.caches)))(*self.caches)
        desc = L.StackDesc(qtype=cfg.qtype, H=H, F=F, E=E, k=k, n_layers=self.L, n_shared=cfg.n_shared,
                           w_router=ctypes.cast(self._wr, ctypes.POINTER(ctypes.c_void_p)),
                           bias=ctypes.cast(self._bias, ctypes.POINTER(ctypes.c_void_p)),
                           n_groups=len(self.caches),
                           caches=ctypes.cast(self._caches, ctypes.POINTER(ctypes.c_void_p)),
                           resident_pool=None if self.resident_pool is None else self.resident_pool.data_ptr(),
                           shared_pool=None if self.shared_pool is None else self.shared_pool.data_ptr(),
                           slot_bytes=self.stride, max_T=self.max_T, workspace=self.workspace.data_ptr(),
                           ws_bytes=ws, overlap=int(overlap), profile=int(profile),
                           device_managed=int(device_managed and bool(self.caches)),
                           use_graph=int(use_graph), load_threshold=float(load_threshold),
                           prefetch_depth=int(prefetch_depth))
        torch.cuda.synchronize()
        self.handle = L.moe_stack_create(desc)

    # -------------------------------------------------------------------------------- API
    def decode(self, x: torch.Tensor, y: torch.Tensor, ids_out: Optional[np.ndarray] = None,
               w_out: Optional[np.ndarray] = None, stream=None) -> None:
        T = x.shape[0]
        L.moe_stack_decode(self.handle, x, y, T,
                           None if ids_out is None else ids_out.ctypes.data,
                           None if w_out is None else w_out.ctypes.data, stream)

    def layer(self, layer: int, x: torch.Tensor, y: torch.Tensor, ids_out: Optional[np.ndarray] = None,
              w_out: Optional[np.ndarray] = None, stream=None) -> None:
        L.moe_stack_layer(self.handle, layer, x, y, x.shape[0],
                          None if ids_out is None else ids_out.ctypes.data,
                          None if w_out is None else w_out.ctypes.data, stream)

    def cache_stats(self) -> List[dict]:
        return [L.moe_cache_stats_get(c) for c in self.caches]

    def profile(self) -> dict:
        return L.moe_stack_profile_get(self.handle)

    def set_profile(self, level: int) -> None:
        L.moe_stack_set_profile(self.handle, level)

    def profile_reset(self) -> None:
        L.moe_stack_profile_reset(self.handle)

    def gemv_timing(self, x: torch.Tensor, reps: int, stream=None) -> dict:
        """The decode GEMV kernels timed alone (resident stacks): every layer's router and
        permute for x, then reps rounds of back-to-back gate/up launches over all layers,
        then of down launches; average microseconds and bytes per launch."""
        return L.moe_stack_gemv_timing(self.handle, x, x.shape[0], reps, stream)

    def reset_caches(self) -> None:
        for c in self.caches:
            L.moe_cache_reset(c)

    def close(self) -> None:
        if getattr(self, "handle", None):
            L.moe_stack_destroy(self.handle)
            self.handle = None
        for c in self.caches:
            L.moe_cache_destroy(c)
        self.caches = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
