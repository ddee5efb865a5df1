"""Seeded synthetic inputs for the HERALD hot path.

This module draws random numbers and rounds them to bf16; it holds none of
the method's arithmetic (no score, softmax, selection or attention).  Both
the CUDA path and the fp64 oracle consume what it produces: the CUDA side the
bf16 bit patterns, the oracle their exact fp64 widening.

Recipe per (workload, layer, sequence n), numpy PCG64 seeded with
1000*index + 100*layer + n:
  * one topic vector mu_g ~ N(0, I_d) per KV group g;
  * every query of the group (all heads, block positions and steps) is
    sqrt(rho)*mu_g + sqrt(1-rho)*eps with rho = 0.5, eps ~ N(0, I) -- marginally
    N(0, 1), but correlated inside a group the way one block's queries are;
  * cache keys and values ~ N(0, 1);
  * planted heavy hitters: key = 3 * (population mean query of the group,
    i.e. sqrt(rho)*mu_g) + N(0, I), either at distinct uniform positions or as
    64-aligned spans of 64 contiguous tokens, always inside [S, L-W);
  * optional "sink" boost: the first n_boost keys scaled by sink_boost;
  * block keys/values of every denoising step ~ N(0, 1).
q_merge is the previous block's first-step queries, q_steps[t] the current
block's step-t queries (q_steps[0] is what stage 2 scores with).
"""
from __future__ import annotations

import numpy as np

from .workloads import Workload

RHO = 0.5


def bf16_bits(x) -> np.ndarray:
    """Round to the nearest bf16, ties to even; returns the uint16 patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + r) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 patterns to float64."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _normal(rng, shape):
    return rng.standard_normal(shape, dtype=np.float32)


def planted_positions(w: Workload, rng) -> np.ndarray:
    lo, hi = w.S, w.L - w.W
    if hi <= lo or w.n_planted <= 0:
        return np.zeros(0, dtype=np.int64)
    if w.planted == "spans":
        first = (lo + w.span - 1) // w.span
        last = (hi - w.span) // w.span
        slots = np.arange(first, last + 1)
        pick = rng.choice(slots, size=min(w.n_planted, len(slots)), replace=False)
        pos = (np.sort(pick)[:, None] * w.span + np.arange(w.span)[None, :]).ravel()
        return pos.astype(np.int64)
    n = min(w.n_planted, hi - lo)
    return np.sort(rng.choice(np.arange(lo, hi), size=n, replace=False)).astype(np.int64)


def make_layer(w: Workload, layer: int = 0, steps: int | None = None) -> dict:
    """All bf16 inputs of one layer for one block, as uint16 arrays.

    Returns q_merge [N,B,Hq,d], q_steps [T,N,B,Hq,d], k_cache / v_cache
    [N,Hkv,L_max,d] (rows >= ctx are zero), block_k / block_v [T,N,B,Hkv,d],
    ctx [N] int32 and planted positions per sequence.
    """
    T = w.T if steps is None else steps
    N, B, Hq, Hkv, d, G = w.N, w.B, w.Hq, w.Hkv, w.d, w.G
    q_merge = np.empty((N, B, Hq, d), np.uint16)
    q_steps = np.empty((T, N, B, Hq, d), np.uint16)
    k_cache = np.zeros((N, Hkv, w.L_max, d), np.uint16)
    v_cache = np.zeros((N, Hkv, w.L_max, d), np.uint16)
    block_k = np.empty((T, N, B, Hkv, d), np.uint16)
    block_v = np.empty((T, N, B, Hkv, d), np.uint16)
    planted = []
    a, c = np.float32(np.sqrt(RHO)), np.float32(np.sqrt(1.0 - RHO))
    for n in range(N):
        rng = np.random.Generator(np.random.PCG64(1000 * w.index + 100 * layer + n))
        mu = _normal(rng, (Hkv, d))
        mu_h = np.repeat(mu, G, axis=0)                      # [Hq, d]
        q_merge[n] = bf16_bits(a * mu_h[None] + c * _normal(rng, (B, Hq, d)))
        for t in range(T):
            q_steps[t, n] = bf16_bits(a * mu_h[None] + c * _normal(rng, (B, Hq, d)))
        kk = _normal(rng, (Hkv, w.L, d))
        vv = _normal(rng, (Hkv, w.L, d))
        pos = planted_positions(w, rng)
        if len(pos):
            kk[:, pos, :] = 3.0 * a * mu[:, None, :] + _normal(rng, (Hkv, len(pos), d))
        if w.n_boost:
            kk[:, : w.n_boost, :] *= np.float32(w.sink_boost)
        k_cache[n, :, : w.L] = bf16_bits(kk)
        v_cache[n, :, : w.L] = bf16_bits(vv)
        for t in range(T):
            block_k[t, n] = bf16_bits(_normal(rng, (B, Hkv, d)))
            block_v[t, n] = bf16_bits(_normal(rng, (B, Hkv, d)))
        planted.append(pos)
    return dict(q_merge=q_merge, q_steps=q_steps, k_cache=k_cache,
                v_cache=v_cache, block_k=block_k, block_v=block_v,
                ctx=np.full(N, w.L, np.int32), planted=planted)


def random_bf16(rng, shape, scale: float = 1.0) -> np.ndarray:
    """Plain N(0, scale^2) bf16 patterns, for edge-case tests."""
    return bf16_bits(np.float32(scale) * _normal(rng, shape))
