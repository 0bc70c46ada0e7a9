"""Seeded synthetic inputs for exact attention.

This module draws random numbers and rounds them to the storage dtype. It holds
none of the attention arithmetic, so both the CUDA path (through the tests and
the benchmark) and the fp64 oracle can consume its arrays without sharing any
of the method's code.

Recipe (the pages' workloads, synthetic by construction):
  * ``numpy.random.default_rng(seed)`` (PCG64), ``standard_normal(dtype=float32)``
    draws Q, K, V and then dO, in that order, each of the full tensor shape;
  * the float32 draws are rounded to the storage dtype with round-to-nearest-even
    (fp16 through numpy's float16, bf16 by the integer RNE rule below);
  * the decode KV cache is drawn one (batch, head) at a time from
    ``default_rng([seed, b, h])`` so any single head can be regenerated on the host
    without materialising the whole cache.

Arrays are returned in their storage form:
  f32  -> numpy float32
  f16  -> numpy float16
  bf16 -> numpy uint16 holding the bf16 bit pattern
and :func:`to_f64` gives the exact real values of any of them.
"""
from __future__ import annotations

import numpy as np

DTYPES = ("f32", "f16", "bf16")


def round_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 draws to the storage dtype (round to nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        bits = x.view(np.uint32)
        lsb = (bits >> np.uint32(16)) & np.uint32(1)
        return ((bits + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    raise ValueError(f"unknown dtype {dtype!r}")


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of an array in storage form."""
    if dtype == "bf16":
        return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def normal(rng: np.random.Generator, shape, dtype: str, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return round_f32(x, dtype)


def attention_inputs(B: int, H: int, M: int, N: int, D: int, dtype: str, seed: int = 0,
                     std: float = 1.0, with_dout: bool = False):
    """Q [B,H,M,D], K/V [B,H,N,D] (and dO [B,H,M,D]) iid N(0, std^2), rounded to dtype."""
    rng = np.random.default_rng(seed)
    q = normal(rng, (B, H, M, D), dtype, std)
    k = normal(rng, (B, H, N, D), dtype, std)
    v = normal(rng, (B, H, N, D), dtype, std)
    if not with_dout:
        return q, k, v
    do = normal(rng, (B, H, M, D), dtype, 1.0)
    return q, k, v, do


def decode_query(B: int, H: int, D: int, dtype: str, seed: int = 0) -> np.ndarray:
    """One query row per (batch, head): q [B,H,1,D]."""
    rng = np.random.default_rng([seed, 0x7175])  # distinct stream from the caches
    return normal(rng, (B, H, 1, D), dtype)


def decode_head_kv(b: int, h: int, N: int, D: int, dtype: str, seed: int = 0):
    """K and V of one (batch, head) of the decode cache: two [N, D] arrays."""
    rng = np.random.default_rng([seed, b, h])
    k = normal(rng, (N, D), dtype)
    v = normal(rng, (N, D), dtype)
    return k, v


def iter_decode_heads(B: int, H: int, N: int, D: int, dtype: str, seed: int = 0, workers: int = 0):
    """Yields (b, h, K_bh, V_bh) for every head, drawn on a thread pool (each head
    has its own generator, so the values do not depend on the number of workers)."""
    import concurrent.futures as cf
    import os
    heads = [(b, h) for b in range(B) for h in range(H)]
    workers = workers or min(16, os.cpu_count() or 1)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        futs = [ex.submit(decode_head_kv, b, h, N, D, dtype, seed) for b, h in heads]
        for (b, h), f in zip(heads, futs):
            k, v = f.result()
            yield b, h, k, v


def decode_inputs(B: int, H: int, N: int, D: int, dtype: str, seed: int = 0):
    """q [B,H,1,D] and the caches K/V [B,H,N,D], head by head from decode_head_kv."""
    q = decode_query(B, H, D, dtype, seed)
    st = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[dtype]
    k = np.empty((B, H, N, D), dtype=st)
    v = np.empty((B, H, N, D), dtype=st)
    for b, h, kh, vh in iter_decode_heads(B, H, N, D, dtype, seed, workers=1 if B * H * N < (1 << 20) else 0):
        k[b, h], v[b, h] = kh, vh
    return q, k, v


def hadamard_signs(d: int, seed: int = 0) -> np.ndarray:
    """d random signs (+1 / -1 as int8) for the FP8 path's incoherent processing."""
    rng = np.random.default_rng([seed, 0x5167])
    return np.where(rng.integers(0, 2, size=d) == 1, 1, -1).astype(np.int8)
