"""Seeded synthetic inputs for exact attention.

This module only draws random numbers and rounds them to bf16.  It holds
none of the attention arithmetic, so both the CPU oracle (through the tests)
and the CUDA path can consume its output without sharing any code of the
method itself.

Recipe
------
* ``numpy.random.default_rng(seed)`` draws float32 standard normals, which
  are multiplied by the requested standard deviation and rounded to bf16
  with round-to-nearest-even.  The same uint16 bit patterns go to the GPU
  (viewed as ``torch.bfloat16``) and, upcast exactly, to the fp64 oracle.
* Tensors are [B, H, N, d], row-major, in the order Q, K, V, dO.
* Seeds are ``1000 * workload_id + case_index``.
* Sampled query rows for large problems: per head,
  ``default_rng(seed + 7).choice(N, min(N, 1024), replace=False)``.

Degenerate inputs (the online-softmax invariants of the paper's forward
algorithm, "FlashAttention V2 in depth", section 6):
* ``identical_keys``: every key of a head equals that head's key row 0.
* ``dominant_key``: one key row j* (drawn from [0, N/4)) is multiplied by 50
  after bf16 rounding and rounded to bf16 again.
* ``rising_keys``: 1 is added to every query component and j / (4 sqrt(d))
  to every component of key row j before the bf16 rounding, so a query's
  logits grow by about a quarter per key (some 46 in log2 units per 128
  keys): each new key tile raises every row's running maximum by far more
  than any correction threshold, and the running output must be rescaled
  at every tile.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

SAMPLE_ROWS = 1024


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even).

    Returns the uint16 bit patterns.  Inputs here are finite normals, so the
    NaN path of the format is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact upcast of bf16 bit patterns to float64."""
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u = bits.astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def normal_bits(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x = x * np.float32(std)
    return bf16_bits(x)


@dataclasses.dataclass
class Case:
    """One seeded attention problem, held as bf16 bit patterns."""

    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: Optional[np.ndarray] = None
    dominant_key: Optional[int] = None

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    def f64(self, name: str) -> np.ndarray:
        return bits_to_f64(getattr(self, name))


def make_case(
    B: int,
    H: int,
    N: int,
    d: int,
    causal: bool,
    seed: int,
    q_std: float = 1.0,
    k_std: float = 1.0,
    v_std: float = 1.0,
    with_do: bool = False,
    degenerate: Optional[str] = None,
) -> Case:
    rng = np.random.default_rng(seed)
    shape = (B, H, N, d)
    if degenerate == "rising_keys":
        q = bf16_bits(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(q_std) + np.float32(1.0))
        ramp = (np.arange(N, dtype=np.float32) / np.float32(4.0 * np.sqrt(d)))[:, None]
        k = bf16_bits(rng.standard_normal(size=shape, dtype=np.float32) * np.float32(k_std) + ramp)
    else:
        q = normal_bits(rng, shape, q_std)
        k = normal_bits(rng, shape, k_std)
    v = normal_bits(rng, shape, v_std)
    do = normal_bits(rng, shape, 1.0) if with_do else None
    jstar = None
    if degenerate == "identical_keys":
        k = np.ascontiguousarray(np.broadcast_to(k[:, :, :1, :], shape))
    elif degenerate == "dominant_key":
        jstar = int(rng.integers(0, max(1, N // 4)))
        row = bits_to_f32(k[:, :, jstar, :]) * np.float32(50.0)
        k = k.copy()
        k[:, :, jstar, :] = bf16_bits(row)
    elif degenerate is not None and degenerate != "rising_keys":
        raise ValueError(f"unknown degenerate case {degenerate!r}")
    return Case(B, H, N, d, causal, seed, q, k, v, do, jstar)


def sample_rows(seed: int, N: int, n: int = SAMPLE_ROWS) -> np.ndarray:
    """Seeded query rows checked when N is large (sorted)."""
    if N <= n:
        return np.arange(N)
    rng = np.random.default_rng(seed + 7)
    return np.sort(rng.choice(N, n, replace=False))


def sample_rows_per_head(seed: int, B: int, H: int, N: int, n: int = SAMPLE_ROWS) -> np.ndarray:
    """[B, H, min(N, n)] sorted query rows, drawn head after head from one
    ``default_rng(seed + 7)`` stream (all rows when N <= n)."""
    if N <= n:
        return np.broadcast_to(np.arange(N), (B, H, N)).copy()
    rng = np.random.default_rng(seed + 7)
    out = np.empty((B, H, n), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            out[b, h] = np.sort(rng.choice(N, n, replace=False))
    return out


# Workloads: the five problem families exact attention is measured on.
# Each entry: (workload_id, name, list of case dicts).

def workload_cases():
    """All seeded cases, grouped by workload id (1..5)."""
    out = {}
    out[1] = [
        dict(B=1, H=1, N=128, d=64, causal=False, seed=1000),
        dict(B=1, H=1, N=128, d=64, causal=True, seed=1001),
    ]
    out[2] = [
        dict(B=4, H=16, N=1024, d=64, causal=False, seed=2000),
        dict(B=4, H=16, N=1024, d=64, causal=True, seed=2001),
        dict(B=4, H=16, N=1024, d=64, causal=False, seed=2002, degenerate="identical_keys"),
        dict(B=4, H=16, N=1024, d=64, causal=True, seed=2003, degenerate="identical_keys"),
        dict(B=4, H=16, N=1024, d=64, causal=False, seed=2004, degenerate="dominant_key"),
        dict(B=4, H=16, N=1024, d=64, causal=True, seed=2005, degenerate="dominant_key"),
    ]
    sweep = []
    idx = 0
    for d in (64, 128):
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            for causal in (False, True):
                sweep.append(dict(B=16384 // N, H=2048 // d, N=N, d=d, causal=causal, seed=3000 + idx))
                idx += 1
    out[3] = sweep
    out[4] = [
        dict(B=8, H=32, N=4096, d=128, causal=True, seed=4000, q_std=3.0, k_std=3.0),
        dict(B=1, H=1, N=65536, d=128, causal=True, seed=4001),
        dict(B=1, H=1, N=65536, d=128, causal=False, seed=4002),
    ]
    out[5] = [
        dict(B=2, H=16, N=4096, d=128, causal=True, seed=5000, with_do=True),
    ]
    return out


def fwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Forward FLOPs as counted for throughput: 4*B*H*N^2*d, halved if causal."""
    f = 4.0 * B * H * N * N * d
    return f / 2 if causal else f


def bwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    """Backward FLOPs as counted for throughput: 2.5x the forward count."""
    return 2.5 * fwd_flops(B, H, N, d, causal)
