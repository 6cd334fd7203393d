"""Seeded synthetic workloads: shapes, value distributions and input generators.

This module is shared by the parity tests, the benchmark and the smoke check. It
holds no arithmetic of the quantization methods: it only draws inputs (keys,
values, queries, fp16 tails, codebooks are NOT here) and rounds them to the
configured storage dtype.

Every tile of input is addressable on its own: the generator for tile
(b, h, block, kind) is seeded with ``SeedSequence([seed, cfg_id, b, h, block,
kind])``, so any block of a million-token context can be regenerated on the CPU
without drawing the blocks before it.

Workloads (the pages' model shapes stand in for their models; no weights or
datasets exist here, values are drawn from the stated distributions):

1. single-head decode, RTN 4-bit, L = 2048, fp16, K channels {6,30,64,98} x12
2. LLaMA-7B-shaped MHA layer (32 heads), nuq3 + 1% CSR outliers, pre-RoPE keys,
   theta = 10000, L = 32768, fp16
3. Llama-3.1-8B-shaped GQA (32 q / 8 KV heads), batch 8, L = 16384, KVarN 2-bit,
   K ~ Student-t(3) with channels {3,17,40,81,122} x10, V ~ N(0,1)
4. TurboQuant-style int4 absmax, GQA 32/8, batch 32, L = 32768, bf16 inputs
5. LLaMA-7B-shaped MHA, batch 1, L = 1,048,576, RTN 2-bit, K channels x12
"""
from __future__ import annotations

import dataclasses
import numpy as np

T = 128   # tokens per block
D = 128   # head dim


@dataclasses.dataclass(frozen=True)
class Workload:
    cfg_id: int
    name: str
    method: str          # "rtn" | "nuq" | "varn" | "int4"
    bits: int
    batch: int
    n_kv_heads: int
    n_q_heads: int
    ctx: int             # context length in tokens (a multiple of 128)
    dtype: str           # "f16" | "bf16"
    k_dist: str          # "normal" | "student_t3"
    k_outlier_channels: tuple = ()
    k_outlier_gain: float = 1.0
    pre_rope: bool = False
    rope_theta: float = 10000.0
    outlier_frac: float = 0.01
    varn_iters: int = 8
    scale_group: int = 128   # int4 / int8 absmax: channels per scale (128 or 64)

    @property
    def n_blocks(self) -> int:
        return self.ctx // T

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def scaled(self, **kw) -> "Workload":
        """Same workload with some fields replaced (smaller contexts/batches for tests)."""
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    1: Workload(1, "single-head RTN4, L=2048", "rtn", 4, 1, 1, 1, 2048, "f16",
                "normal", (6, 30, 64, 98), 12.0),
    2: Workload(2, "LLaMA-7B MHA 32x128, nuq3 + 1% CSR, pre-RoPE, L=32768", "nuq", 3,
                1, 32, 32, 32768, "f16", "normal", pre_rope=True, rope_theta=10000.0,
                outlier_frac=0.01),
    3: Workload(3, "Llama-3.1-8B GQA 32/8, KVarN 2-bit, B=8, L=16384", "varn", 2,
                8, 8, 32, 16384, "f16", "student_t3", (3, 17, 40, 81, 122), 10.0,
                varn_iters=8),
    4: Workload(4, "TurboQuant int4 GQA 32/8, B=32, L=32768, bf16", "int4", 4,
                32, 8, 32, 32768, "bf16", "normal"),
    5: Workload(5, "LLaMA-7B MHA 32x128, RTN2, B=1, L=1048576, streaming", "rtn", 2,
                1, 32, 32, 1048576, "f16", "normal", (6, 30, 64, 98), 12.0),
}


# ---------------------------------------------------------------- dtype rounding

def round_f16(x: np.ndarray) -> np.ndarray:
    """fp32 values rounded to the nearest fp16 (ties to even), returned as float32."""
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even. Finite inputs."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    bias = 0x7FFF + ((u >> 16) & 1)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def round_bf16(x: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(f32_to_bf16_bits(x))


def round_dtype(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_f16(x) if dtype == "f16" else round_bf16(x)


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Values (already representable) -> the uint16 bit patterns a device buffer holds."""
    if dtype == "f16":
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)
    return f32_to_bf16_bits(x)


# ---------------------------------------------------------------- generators

KIND_K, KIND_V = 0, 1


def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed)] + [int(k) for k in key]))


def tile(w: Workload, b: int, h: int, blk: int, kind: int, seed: int = 0) -> np.ndarray:
    """One 128-token x 128-channel tile of K (kind 0) or V (kind 1), float32 values
    exactly representable in the workload dtype."""
    g = _rng(seed, w.cfg_id, b, h, blk, kind)
    if kind == KIND_K and w.k_dist == "student_t3":
        x = g.standard_t(3, size=(T, D)).astype(np.float32)
    else:
        x = g.standard_normal((T, D), dtype=np.float32)
    if kind == KIND_K and w.k_outlier_channels:
        x[:, list(w.k_outlier_channels)] *= np.float32(w.k_outlier_gain)
    return round_dtype(x, w.dtype)


def block(w: Workload, blk: int, seed: int = 0):
    """K and V for one block of all (batch, KV head): two float32 [B][H_kv][128][128]."""
    K = np.empty((w.batch, w.n_kv_heads, T, D), np.float32)
    V = np.empty_like(K)
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            K[b, h] = tile(w, b, h, blk, KIND_K, seed)
            V[b, h] = tile(w, b, h, blk, KIND_V, seed)
    return K, V


def blocks(w: Workload, first: int, n: int, seed: int = 0):
    """K and V for blocks [first, first+n): float32 [B][H_kv][n*128][128]."""
    K = np.empty((w.batch, w.n_kv_heads, n * T, D), np.float32)
    V = np.empty_like(K)
    for i in range(n):
        k, v = block(w, first + i, seed)
        K[:, :, i * T:(i + 1) * T] = k
        V[:, :, i * T:(i + 1) * T] = v
    return K, V


def query(w: Workload, step: int = 0, seed: int = 0) -> np.ndarray:
    """Decode query [B][H_q][128] ~ N(0,1), rounded to the workload dtype. For pre-RoPE
    workloads the query is taken as already position-encoded."""
    g = _rng(seed, w.cfg_id, 1_000_003, step)
    return round_dtype(g.standard_normal((w.batch, w.n_q_heads, D), dtype=np.float32), w.dtype)


def tail(w: Workload, n_tail: int, step: int = 0, seed: int = 0):
    """fp residual tail (< 128 newest tokens not yet in a full block): K, V float32
    [B][H_kv][n_tail][128], same distributions as the cached blocks."""
    g = _rng(seed, w.cfg_id, 2_000_003, step)
    shape = (w.batch, w.n_kv_heads, n_tail, D)
    if w.k_dist == "student_t3":
        k = g.standard_t(3, size=shape).astype(np.float32)
    else:
        k = g.standard_normal(shape, dtype=np.float32)
    if w.k_outlier_channels:
        k[..., list(w.k_outlier_channels)] *= np.float32(w.k_outlier_gain)
    v = g.standard_normal(shape, dtype=np.float32)
    return round_dtype(k, w.dtype), round_dtype(v, w.dtype)
