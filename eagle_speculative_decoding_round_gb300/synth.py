"""Seeded synthetic inputs for one EAGLE-3 round.

This module holds no arithmetic of the method itself: only random numbers,
shapes and layouts.  Both the CUDA path's tests/bench and the CPU oracle's
tests draw their inputs from here.

* Normal tensors: numpy PCG64 streams (CPU) keyed by (seed, name).
* Uniforms for accept/reject: SplitMix64 (Steele, Lea & Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014) chained over
  (seed, purpose, request, node); the high 32 bits are the uint32 uniform.
* Paged KV: pages of ``page_size`` tokens, shuffled in the pool.
* A tiny synthetic target (token/position-keyed Q/K/V tables, rotary positions,
  random LM head) used by the greedy-equals-sequential-decoding check.
"""
from __future__ import annotations

import hashlib

import numpy as np

MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)
PURPOSE_ACCEPT = 1
PURPOSE_BONUS = 2


def _seed_of(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little")


def rng(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(_seed_of(seed, name)))


def normal(seed: int, name: str, shape, std: float = 0.02) -> np.ndarray:
    """N(0, std^2) fp32 array."""
    return (rng(seed, name).standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def splitmix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser applied to x + golden gamma (uint64, wrapping)."""
    with np.errstate(over="ignore"):
        z = (np.asarray(x, np.uint64) + np.uint64(0x9E3779B97F4A7C15)) & MASK64
        z = ((z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)) & MASK64
        z = ((z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)) & MASK64
        return z ^ (z >> np.uint64(31))


def uniforms(seed: int, purpose: int, n_req: int, n_node: int, req0: int = 0) -> np.ndarray:
    """uint32 uniforms [n_req, n_node] keyed by (seed, purpose, request, node)."""
    r = np.arange(req0, req0 + n_req, dtype=np.uint64)[:, None]
    j = np.arange(n_node, dtype=np.uint64)[None, :]
    h = splitmix64(np.full((1, 1), seed, np.uint64))
    h = splitmix64(h ^ np.uint64(purpose))
    h = splitmix64(h ^ r)
    h = splitmix64(h ^ j)
    return (h >> np.uint64(32)).astype(np.uint32)


def to_bf16_f32(a: np.ndarray) -> np.ndarray:
    """Round fp32 -> bf16 (nearest even) and return the rounded values as fp32."""
    a = np.ascontiguousarray(a, np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    nan = np.isnan(a)
    out = (r & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    out = np.where(nan, a, out)
    return out.astype(np.float32)


def bf16_bits(a32: np.ndarray) -> np.ndarray:
    """fp32 values already on the bf16 grid -> uint16 bit patterns."""
    return (np.ascontiguousarray(a32, np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def page_table(seed: int, lens, page_size: int, extra_pages: int = 0):
    """Random page assignment.  Returns (page_table [B, max_pages] int32, n_pages).

    Request b owns ceil(lens[b] / page_size) pages drawn without replacement from
    a shuffled pool; unused table entries point at page 0.
    """
    lens = [int(x) for x in lens]
    need = [(n + page_size - 1) // page_size for n in lens]
    total = sum(need) + extra_pages
    perm = rng(seed, "pages").permutation(total).astype(np.int32)
    maxp = max(need) if need else 1
    pt = np.zeros((len(lens), max(maxp, 1)), np.int32)
    o = 0
    for b, n in enumerate(need):
        pt[b, :n] = perm[o:o + n]
        o += n
    return pt, total


# ---------------------------------------------------------------------------
# tiny synthetic target (token/position-keyed), for sequential-decoding checks
# ---------------------------------------------------------------------------

def rope(x: np.ndarray, pos: int, base: float = 10000.0) -> np.ndarray:
    """Rotate pairs (2i, 2i+1) of the last axis by pos * base^(-2i/hd) (fp64)."""
    x = np.asarray(x, np.float64)
    hd = x.shape[-1]
    i = np.arange(hd // 2, dtype=np.float64)
    th = pos * base ** (-2.0 * i / hd)
    c, s = np.cos(th), np.sin(th)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 0::2] * s + x[..., 1::2] * c
    return out


class TinyTarget:
    """One-layer synthetic target: q/k/v of token x at position p are rows of
    random tables with rotary position applied to q and k; the final hidden is
    the attention output reshaped to [H*hd]; logits = W_lm @ hidden."""

    def __init__(self, seed: int, V: int, H: int, KVH: int, hd: int, std: float = 0.02,
                 lm_std: float = 1.0):
        self.V, self.H, self.KVH, self.hd = V, H, KVH, hd
        self.Qtab = normal(seed, "tt.q", (V, H, hd), 1.0)
        self.Ktab = normal(seed, "tt.k", (V, KVH, hd), 1.0)
        self.Vtab = normal(seed, "tt.v", (V, KVH, hd), std)
        self.W_lm = normal(seed, "tt.lm", (V, H * hd), lm_std)

    def q(self, tok: int, pos: int) -> np.ndarray:
        return rope(self.Qtab[tok], pos).astype(np.float32)

    def k(self, tok: int, pos: int) -> np.ndarray:
        return rope(self.Ktab[tok], pos).astype(np.float32)

    def v(self, tok: int, pos: int) -> np.ndarray:
        return self.Vtab[tok].astype(np.float32)
