"""Seeded synthetic workloads for the LongFlow decode step.

This module only draws inputs. It holds none of the decode step's arithmetic,
so both the CUDA path and the fp64 oracle can be fed from it without sharing
any of the method's code.

The shapes follow the workloads that "LongFlow: Efficient KV Cache Compression
for Reasoning Models" measures or describes:

* Fig. 1: Qwen3-8B attention layer (32 query heads, 8 KV heads, head dim 128),
  batch 128, sequence 3200, one eviction per attention call.
* Table 1: a KV budget of 2400 slots (DeepSeek-R1-Distill-Llama-8B, same GQA
  shape).
* Abstract: long-output reasoning decodes, which is where the 16384-slot
  ragged stress workload comes from.

The paper prints no input data, so every value here is synthetic:
N(0, 1) fp32 drawn from numpy's PCG64, rounded to bf16 (round to nearest even).

Determinism across machines and thread counts comes from giving every
sequence ``b`` (and every decode step) its own ``SeedSequence`` child. Any
subset of sequences can be regenerated bit for bit without drawing the rest,
which is how the oracle gets the units it checks at full size.

Draw order inside a sequence's generator:

1. the live length L_b (ragged workloads only);
2. K [Hkv, S, d], then V [Hkv, S, d];
3. the per-slot lognormal K factors [Hkv, S] (only when ``k_lognormal_sigma`` > 0);
4. for each KV head, the heavy-hitter picks among its live slots (only when
   ``heavy_frac`` > 0).

Draw order inside a step's generator: q [B, Hq, d], new_k [B, Hkv, d],
new_v [B, Hkv, d], then the lognormal factors of new_k [B, Hkv] (only when
``k_lognormal_sigma`` > 0).

Mask encoding, as the library reads it: one int32 per (b, kvh, slot). -1 marks an
empty or masked slot. A value >= 0 is the slot's age in decode steps. Live slots
fill a prefix: slot j < L_b holds token j, whose age is L_b - 1 - j.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "WORKLOADS",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "sequence_state",
    "initial_state",
    "step_inputs",
    "live_lengths",
    "algorithmic_bytes",
]

_STATE_KEY = 0
_STEP_KEY = 1


@dataclass(frozen=True)
class Workload:
    """One decode-step workload: shapes, value recipe and step count."""

    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    S: int
    W: int
    steps: int
    seed: int
    # Live slots per sequence: an int (same for every sequence), or an
    # inclusive (lo, hi) range drawn uniformly per sequence.
    live: int | tuple[int, int]
    k_lognormal_sigma: float = 0.0
    heavy_frac: float = 0.0
    heavy_scale: float = 4.0
    description: str = ""
    scale: float = field(default=float("nan"))

    def __post_init__(self):
        if math.isnan(self.scale):
            object.__setattr__(self, "scale", float(np.float32(1.0 / math.sqrt(self.d))))

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def units(self) -> int:
        return self.B * self.Hkv

    def shapes(self) -> dict:
        return {
            "q": (self.B, self.Hq, self.d),
            "k_cache": (self.B, self.Hkv, self.S, self.d),
            "v_cache": (self.B, self.Hkv, self.S, self.d),
            "mask": (self.B, self.Hkv, self.S),
            "new_k": (self.B, self.Hkv, self.d),
            "new_v": (self.B, self.Hkv, self.d),
            "write_slot": (self.B, self.Hkv),
            "out": (self.B, self.Hq, self.d),
            "next_slot": (self.B, self.Hkv),
        }

    def with_batch(self, B: int) -> "Workload":
        """The same per-sequence recipe with a different batch (used for shards)."""
        return Workload(
            name=self.name, B=B, Hq=self.Hq, Hkv=self.Hkv, d=self.d, S=self.S, W=self.W,
            steps=self.steps, seed=self.seed, live=self.live,
            k_lognormal_sigma=self.k_lognormal_sigma, heavy_frac=self.heavy_frac,
            heavy_scale=self.heavy_scale, description=self.description, scale=self.scale)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload(
            name="tiny_b2_s256", B=2, Hq=4, Hkv=2, d=64, S=256, W=8, steps=16, seed=0,
            live=240,
            description="B=2 Hq=4 Hkv=2 d=64, S=256 (slots 240..255 masked), W=8, N(0,1)"),
        Workload(
            name="qwen3_8b_b1_s2400", B=1, Hq=32, Hkv=8, d=128, S=2400, W=32, steps=256,
            seed=1, live=2400, k_lognormal_sigma=0.5,
            description="Qwen3-8B layer, one sequence, budget 2400 slots all live, W=32, "
                        "K rows x lognormal(0,0.5)"),
        Workload(
            name="qwen3_8b_b128_s3200", B=128, Hq=32, Hkv=8, d=128, S=3200, W=32, steps=64,
            seed=2, live=3200, k_lognormal_sigma=0.5,
            description="Qwen3-8B Fig. 1 shape: batch 128, 3200 slots all live, W=32, "
                        "K rows x lognormal(0,0.5)"),
        Workload(
            name="llama8b_b256_s2400_ragged", B=256, Hq=32, Hkv=8, d=128, S=2400, W=64,
            steps=128, seed=3, live=(600, 2400),
            description="Llama-8B-class GQA batch 256, budget 2400, live length "
                        "U{600..2400} per sequence, W=64"),
        Workload(
            name="long_b32_s16384_ragged", B=32, Hq=32, Hkv=8, d=128, S=16384, W=128,
            steps=64, seed=4, live=(4096, 16384), heavy_frac=0.01, heavy_scale=4.0,
            description="long-output stress: batch 32, 16384 slots, live length "
                        "U{4096..16384}, W=128, 1% heavy-hitter keys x4"),
    ]
}


# ---------------------------------------------------------------------------
# bf16 bit conversions (round to nearest even; inputs are finite)
# ---------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return the raw bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bits to fp32 exactly."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ---------------------------------------------------------------------------
# Generators
# ---------------------------------------------------------------------------

def _rng(seed: int, key: int, idx: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(key, idx))))


def _live_len(wl: Workload, rng: np.random.Generator) -> int:
    if isinstance(wl.live, tuple):
        lo, hi = wl.live
        return int(rng.integers(lo, hi + 1))
    return int(wl.live)


def sequence_state(wl: Workload, b: int):
    """Initial cache and mask of sequence ``b``.

    Returns (k [Hkv,S,d] u16, v [Hkv,S,d] u16, mask [Hkv,S] i32, L_b).
    """
    rng = _rng(wl.seed, _STATE_KEY, b)
    L = _live_len(wl, rng)
    shape = (wl.Hkv, wl.S, wl.d)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    if wl.k_lognormal_sigma > 0:
        z = rng.standard_normal((wl.Hkv, wl.S), dtype=np.float32)
        k *= np.exp(np.float32(wl.k_lognormal_sigma) * z)[:, :, None]
    if wl.heavy_frac > 0 and L > 0:
        n_heavy = max(1, int(round(wl.heavy_frac * L)))
        for h in range(wl.Hkv):
            picks = rng.choice(L, size=n_heavy, replace=False)
            k[h, picks, :] *= np.float32(wl.heavy_scale)
    mask = np.full((wl.Hkv, wl.S), -1, dtype=np.int32)
    mask[:, :L] = (L - 1 - np.arange(L, dtype=np.int32))[None, :]
    return f32_to_bf16_bits(k), f32_to_bf16_bits(v), mask, L


def live_lengths(wl: Workload) -> np.ndarray:
    """L_b for every sequence, drawn exactly as ``sequence_state`` draws it."""
    return np.array([_live_len(wl, _rng(wl.seed, _STATE_KEY, b)) for b in range(wl.B)],
                    dtype=np.int64)


def initial_state(wl: Workload, threads: int | None = None, batch_offset: int = 0):
    """Whole-batch initial state as numpy arrays (bf16 as uint16 bits).

    ``batch_offset`` selects sequences [batch_offset, batch_offset + wl.B) of the
    recipe, so a shard of a larger batch regenerates the same bits.
    """
    k = np.empty((wl.B, wl.Hkv, wl.S, wl.d), dtype=np.uint16)
    v = np.empty_like(k)
    mask = np.empty((wl.B, wl.Hkv, wl.S), dtype=np.int32)
    lengths = np.empty(wl.B, dtype=np.int64)

    def fill(b):
        kb, vb, mb, L = sequence_state(wl, batch_offset + b)
        k[b], v[b], mask[b], lengths[b] = kb, vb, mb, L

    threads = threads or min(16, os.cpu_count() or 1)
    if threads > 1 and wl.B > 1:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, range(wl.B)))
    else:
        for b in range(wl.B):
            fill(b)
    return {"k_cache": k, "v_cache": v, "mask": mask, "lengths": lengths}


def step_inputs(wl: Workload, step: int, batch_offset: int = 0, full_batch: int | None = None):
    """q, new_k, new_v for decode step ``step`` (bf16 bits).

    The step draw covers the full batch of the recipe (``full_batch``, default
    ``wl.B``) and returns rows [batch_offset, batch_offset + wl.B), so shards agree
    with the unsharded run.
    """
    nb = full_batch or wl.B
    rng = _rng(wl.seed, _STEP_KEY, step)
    q = rng.standard_normal((nb, wl.Hq, wl.d), dtype=np.float32)
    nk = rng.standard_normal((nb, wl.Hkv, wl.d), dtype=np.float32)
    nv = rng.standard_normal((nb, wl.Hkv, wl.d), dtype=np.float32)
    if wl.k_lognormal_sigma > 0:
        z = rng.standard_normal((nb, wl.Hkv), dtype=np.float32)
        nk *= np.exp(np.float32(wl.k_lognormal_sigma) * z)[:, :, None]
    sl = slice(batch_offset, batch_offset + wl.B)
    return {
        "q": f32_to_bf16_bits(q[sl]),
        "new_k": f32_to_bf16_bits(nk[sl]),
        "new_v": f32_to_bf16_bits(nv[sl]),
    }


def algorithmic_bytes(wl: Workload, lengths: np.ndarray | None = None) -> int:
    """Useful HBM bytes of one decode step.

    Live K and V rows read once, q read, out written, the new K/V row written.
    Mask traffic and any scratch are overhead and are not counted.
    """
    if lengths is None:
        lengths = live_lengths(wl)
    kv = int(np.sum(lengths)) * wl.Hkv * 4 * wl.d
    return kv + wl.B * wl.Hq * wl.d * 2 * 2 + wl.B * wl.Hkv * wl.d * 2 * 2
