"""Seeded synthetic inputs for the MoE decode / prefill FFN layer.

This module is shared by the CUDA path (tests, ``bench.py``) and by the
CPU oracle's callers.  It holds NO arithmetic of the method itself: no
dequantisation, routing, softmax, FFN or combine.  It only draws random
numbers and lays them out in the canonical input formats:

* q8_0 block (34 bytes): little-endian fp16 scale ``d`` then 32 int8 codes.
  The block format is the one named on page 5 ("GPU 卸载研究笔记",
  section 1.2, quantised blocks such as q8_0's 34-byte block kept as-is).
* 4-bit scale+min block (20 bytes): fp16 ``d``, fp16 ``m``, then 16 bytes of
  codes, byte ``i`` holding code ``2i`` in its low nibble and ``2i+1`` in its
  high nibble.

Expert tensors follow page 2's ``ffn_{gate,up,down}_exps`` layout
("llama.cpp MoE GGUF 张量加载" notes, expert tensor shapes): expert-major,
each matrix stored row by row (one row per output feature), each row a run
of blocks along the reduction dimension.  gate and up are [F rows][H cols],
down is [H rows][F cols].

Workload shapes follow the five configurations of the decode / prefill
study (tiny layer, Granite-, Qwen3-30B-A3B- and DeepSeek-MoE-16B-shaped
stacks, and the Qwen-shaped prefill layer).  Seeds are
``1000*cfg + {0: weights, 1: router, 2: bias permutation, 3+step: x}``;
per (layer, expert) streams are independent so any expert can be
regenerated on demand without materialising a whole stack.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence, Tuple

import numpy as np

Q8_0 = 0
Q4_SM = 1
X_F32 = 0
X_BF16 = 1

Q8_0_BLOCK_BYTES = 34
Q4_SM_BLOCK_BYTES = 20
QK = 32  # weights per block


@dataclasses.dataclass(frozen=True)
class PoolGroup:
    """One type/shape group of layers sharing an LRU slot pool."""
    first_layer: int
    n_layers: int
    n_slots: int


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    index: int
    name: str
    H: int
    F: int
    E: int
    k: int
    L: int
    qtype: int
    n_shared: int
    bias_a: float           # 0.0: no router bias
    router_var: float       # variance of the fp16 router weights
    xtype: int
    tokens: Tuple[int, ...]
    steps: int
    groups: Tuple[PoolGroup, ...]   # empty: every expert resident
    weight_seed_cfg: int            # whose weight/router/bias seeds to use
    d_value: float = 0.02 / 40.0
    m_value: float = 0.0

    @property
    def block_bytes(self) -> int:
        return Q8_0_BLOCK_BYTES if self.qtype == Q8_0 else Q4_SM_BLOCK_BYTES

    def matrix_bytes(self, rows: int, cols: int) -> int:
        return rows * (cols // QK) * self.block_bytes

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert (gate + up + down) in the canonical format."""
        return 2 * self.matrix_bytes(self.F, self.H) + self.matrix_bytes(self.H, self.F)

    @property
    def seed_base(self) -> int:
        return 1000 * self.weight_seed_cfg


def _cfgs() -> Tuple[MoEConfig, ...]:
    v2048 = 1.0 / math.sqrt(2048.0)
    return (
        MoEConfig(0, "tiny-moe-layer", H=256, F=512, E=8, k=2, L=1, qtype=Q8_0, n_shared=0,
                  bias_a=0.0, router_var=1.0 / 16.0, xtype=X_F32, tokens=(1,), steps=1,
                  groups=(), weight_seed_cfg=0),
        MoEConfig(1, "granite-moe-24L-h1024-e32-top8-q8_0", H=1024, F=512, E=32, k=8, L=24,
                  qtype=Q8_0, n_shared=0, bias_a=1.0, router_var=1.0 / 32.0, xtype=X_F32,
                  tokens=(1, 4, 8), steps=256, groups=(PoolGroup(0, 24, 384),), weight_seed_cfg=1),
        MoEConfig(2, "qwen3-30b-a3b-48L-h2048-e128-top8-q4", H=2048, F=768, E=128, k=8, L=48,
                  qtype=Q4_SM, n_shared=0, bias_a=1.1, router_var=v2048, xtype=X_F32,
                  tokens=(1,), steps=256,
                  groups=(PoolGroup(0, 24, 1834), PoolGroup(24, 24, 1834)), weight_seed_cfg=2,
                  d_value=0.004, m_value=-0.03),
        MoEConfig(3, "deepseek-moe-16b-28L-h2048-e64+2-top2-q8_0", H=2048, F=1408, E=64, k=2, L=28,
                  qtype=Q8_0, n_shared=2, bias_a=1.2, router_var=v2048, xtype=X_F32,
                  tokens=(1, 32), steps=256, groups=(PoolGroup(0, 28, 224),), weight_seed_cfg=3),
        MoEConfig(4, "qwen3-30b-a3b-layer-prefill-q4", H=2048, F=768, E=128, k=8, L=1,
                  qtype=Q4_SM, n_shared=0, bias_a=1.1, router_var=v2048, xtype=X_BF16,
                  tokens=(512, 4096), steps=1, groups=(), weight_seed_cfg=2,
                  d_value=0.004, m_value=-0.03),
    )


CONFIGS: Tuple[MoEConfig, ...] = _cfgs()


def config(i: int) -> MoEConfig:
    return CONFIGS[i]


def small_config(qtype: int, H: int, F: int, E: int, k: int, L: int = 1, n_shared: int = 0,
                 bias_a: float = 0.0, xtype: int = X_F32, seed_cfg: int = 900,
                 groups: Tuple[PoolGroup, ...] = ()) -> MoEConfig:
    """A reduced-size configuration with the same generators (for fast tests)."""
    d, m = (0.02 / 40.0, 0.0) if qtype == Q8_0 else (0.004, -0.03)
    return MoEConfig(seed_cfg, f"small-q{qtype}-h{H}-f{F}-e{E}-k{k}", H=H, F=F, E=E, k=k, L=L,
                     qtype=qtype, n_shared=n_shared, bias_a=bias_a,
                     router_var=1.0 / math.sqrt(H), xtype=xtype, tokens=(1,), steps=1,
                     groups=groups, weight_seed_cfg=seed_cfg, d_value=d, m_value=m)


# ----------------------------------------------------------------------------------------------
# random streams

def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(k) for k in key])))


def _fp16_bits(value: float) -> int:
    return int(np.array([value], dtype=np.float16).view(np.uint16)[0])


def _round_half_away(v: np.ndarray) -> np.ndarray:
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


def q8_0_blocks(rng: np.random.Generator, rows: int, cols: int, d_value: float,
                random_scales: bool = False) -> np.ndarray:
    """Canonical q8_0 matrix: [rows][cols/32] blocks of (fp16 d, int8 q[32]) as raw bytes.

    Codes are round(N(0,1)*40) clipped to [-127, 127] (round half away from zero).
    """
    nb = cols // QK
    z = rng.standard_normal((rows, nb, QK), dtype=np.float32)
    z *= np.float32(40.0)
    z += np.copysign(np.float32(0.5), z)   # round half away from zero: trunc(z + sign(z)/2)
    np.trunc(z, out=z)
    np.clip(z, -127, 127, out=z)
    q = z.astype(np.int8)
    out = np.empty((rows, nb, Q8_0_BLOCK_BYTES), dtype=np.uint8)
    if random_scales:
        d = (rng.uniform(0.25, 4.0, size=(rows, nb)) * d_value).astype(np.float16)
        out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
    else:
        bits = _fp16_bits(d_value)
        out[:, :, 0] = bits & 0xFF
        out[:, :, 1] = bits >> 8
    out[:, :, 2:] = q.view(np.uint8)
    return out.reshape(-1)


def q4_sm_blocks(rng: np.random.Generator, rows: int, cols: int, d_value: float, m_value: float,
                 random_scales: bool = False) -> np.ndarray:
    """Canonical 4-bit scale+min matrix: [rows][cols/32] blocks of (fp16 d, fp16 m, 16 bytes).

    Codes are uniform on 0..15; two codes per byte (even index in the low nibble), so a
    uniform random byte carries two independent uniform codes.
    """
    nb = cols // QK
    out = np.empty((rows, nb, Q4_SM_BLOCK_BYTES), dtype=np.uint8)
    out[:, :, 4:] = rng.integers(0, 256, size=(rows, nb, 16), dtype=np.uint8)
    if random_scales:
        d = (rng.uniform(0.25, 4.0, size=(rows, nb)) * d_value).astype(np.float16)
        m = (rng.uniform(-2.0, 2.0, size=(rows, nb)) * abs(m_value if m_value else 0.03)).astype(np.float16)
        out[:, :, 0:2] = d.view(np.uint8).reshape(rows, nb, 2)
        out[:, :, 2:4] = m.view(np.uint8).reshape(rows, nb, 2)
    else:
        db, mb = _fp16_bits(d_value), _fp16_bits(m_value)
        out[:, :, 0], out[:, :, 1] = db & 0xFF, db >> 8
        out[:, :, 2], out[:, :, 3] = mb & 0xFF, mb >> 8
    return out.reshape(-1)


def expert_weights(cfg: MoEConfig, layer: int, expert: int, random_scales: bool = False
                   ) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """(gate, up, down) canonical block bytes of one expert.

    Routed experts are 0..E-1; shared experts are E..E+n_shared-1 in the same stream.
    """
    rng = _rng(cfg.seed_base + 0, layer, expert, int(random_scales))
    H, F = cfg.H, cfg.F
    if cfg.qtype == Q8_0:
        g = q8_0_blocks(rng, F, H, cfg.d_value, random_scales)
        u = q8_0_blocks(rng, F, H, cfg.d_value, random_scales)
        d = q8_0_blocks(rng, H, F, cfg.d_value, random_scales)
    else:
        g = q4_sm_blocks(rng, F, H, cfg.d_value, cfg.m_value, random_scales)
        u = q4_sm_blocks(rng, F, H, cfg.d_value, cfg.m_value, random_scales)
        d = q4_sm_blocks(rng, H, F, cfg.d_value, cfg.m_value, random_scales)
    return g, u, d


def router_weights(cfg: MoEConfig, layer: int) -> np.ndarray:
    """fp16 router matrix W_r [H][E] (row-major) ~ N(0, router_var), returned as uint16 bits."""
    rng = _rng(cfg.seed_base + 1, layer)
    w = rng.standard_normal((cfg.H, cfg.E)) * math.sqrt(cfg.router_var)
    return w.astype(np.float16).view(np.uint16)


def router_bias(cfg: MoEConfig, layer: int) -> Optional[np.ndarray]:
    """Per-layer expert bias -a*ln(rank) over a seeded permutation (fp32), or None.

    Rank r = 1..E is given to expert perm[r-1]; rank 1 gets bias 0.
    """
    if cfg.bias_a == 0.0:
        return None
    rng = _rng(cfg.seed_base + 2, layer)
    perm = rng.permutation(cfg.E)
    b = np.empty(cfg.E, dtype=np.float32)
    ranks = np.arange(1, cfg.E + 1, dtype=np.float64)
    b[perm] = (-cfg.bias_a * np.log(ranks)).astype(np.float32)
    return b


def tokens_x(cfg: MoEConfig, step: int, T: int) -> np.ndarray:
    """Decode/prefill input x ~ N(0,1), [T][H]; fp32, or bf16 bits (uint16) for bf16 configs."""
    rng = _rng(1000 * cfg.index + 3 + step, T)
    x = rng.standard_normal((T, cfg.H), dtype=np.float32)
    if cfg.xtype == X_BF16:
        return f32_to_bf16_bits(x)
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def routed_slot_bytes(cfg: MoEConfig) -> int:
    """Bytes per expert in the canonical format (the slot payload before alignment)."""
    return cfg.expert_bytes


def all_expert_ids(cfg: MoEConfig) -> Sequence[int]:
    return range(cfg.E)
