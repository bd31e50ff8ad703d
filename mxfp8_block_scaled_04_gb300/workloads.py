"""Seeded synthetic BF16 inputs for the quantize workloads.

This module only draws random numbers and rounds them to BF16; it holds none
of the quantization arithmetic, so both the CUDA path's tests and the CPU
oracle's tests can take their inputs from here.  Every array is returned as
the BF16 bit pattern (numpy uint16, row-major).

The five workloads (names are what they are, with their sizes):

``small_128x256``
    128x256, N(0,1), seed 0; E4M3 rowwise + colwise.
``act_4096x4096``
    4096x4096 activations: N(0,1) scaled per row by lognormal(0,2); 0.1% of
    entries replaced by +-U(100,1000) outliers; 1% of the 1x32 row blocks
    zeroed.  E4M3.
``fc1_8192x28672``
    8192x28672 MLP FC1 activation, N(0,0.5) with 1e-3 of entries replaced by
    +-U(1e3,1e4).  E4M3.  The throughput shape.
``grad_16384x8192``
    16384x8192 gradient, N(0,1e-3); 5% of entries replaced by BF16-subnormal
    values N(0,1)*1e-39; 1% by +-2^k with k uniform in [-20, 0]; rows 0..31,
    columns 0..31 all subnormal and columns 32..63 all exact powers of two.
    E5M2 with fused dbias.
``moe_64x65536x7168``
    64 experts, ragged row counts (multiples of 32, Zipf s=1.1 over a seeded
    permutation, 4 experts forced empty) summing to 65536 rows, hidden 7168,
    N(0,1) scaled per expert by lognormal(0,1).  E4M3, grouped.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3 = 0
E5M2 = 1


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32/float64 values to BF16 (nearest-even, via torch) and return the uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def normal_bf16(M: int, N: int, seed: int, std: float = 1.0) -> np.ndarray:
    """N(0, std^2) BF16 matrix [M,N]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N), dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return to_bf16_bits(a)


def banded_bf16(M: int, N: int, seed: int, band: int = 256) -> np.ndarray:
    """A large BF16 matrix [M,N] made cheaply: one N(0,1) block of `band` rows, repeated down the
    matrix with each band scaled by its own power of two 2^k, k in [-8, 8] (seeded), applied to the
    exponent field (exact: the block's zeros and values below 2^-118 are replaced by +-1 first, so
    every shifted value stays in the normal range)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    block = normal_bf16(band, N, seed)
    tiny = (block & 0x7F80) <= (8 << 7)
    block[tiny] = (block[tiny] & 0x8000) | 0x3F80
    assert np.all((block & 0x7F80) > 8 << 7) and np.all((block & 0x7F80) < 0x7F80 - (8 << 7))
    k = rng.integers(-8, 9, size=(M + band - 1) // band)
    out = np.empty((M, N), np.uint16)
    for b in range(k.size):
        r0 = b * band
        rows = min(band, M - r0)
        out[r0:r0 + rows] = (block[:rows].astype(np.int32) + (int(k[b]) << 7)).astype(np.uint16)
    return out


def _scatter(rng, a_flat, frac, values_fn):
    count = int(round(frac * a_flat.size))
    if count:
        idx = rng.integers(0, a_flat.size, size=count)
        a_flat[idx] = values_fn(count)


def act_bf16(M: int, N: int, seed: int) -> np.ndarray:
    """Activation-like matrix: per-row lognormal(0,2) scale, 0.1% outliers, 1% zero row blocks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N), dtype=np.float32)
    a *= rng.lognormal(0.0, 2.0, size=(M, 1)).astype(np.float32)
    flat = a.reshape(-1)
    _scatter(rng, flat, 1e-3,
             lambda n: (rng.choice([-1.0, 1.0], n) * rng.uniform(100.0, 1000.0, n)).astype(np.float32))
    blocks = a.reshape(M, N // 32, 32)
    nblk = M * (N // 32)
    zb = rng.integers(0, nblk, size=int(round(0.01 * nblk)))
    blocks.reshape(nblk, 32)[zb] = 0.0
    return to_bf16_bits(a)


def fc1_bf16(M: int, N: int, seed: int) -> np.ndarray:
    """N(0,0.5) with 1e-3 of entries replaced by +-U(1e3,1e4)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N), dtype=np.float32)
    a *= np.float32(0.5)
    _scatter(rng, a.reshape(-1), 1e-3,
             lambda n: (rng.choice([-1.0, 1.0], n) * rng.uniform(1e3, 1e4, n)).astype(np.float32))
    return to_bf16_bits(a)


def grad_bf16(M: int, N: int, seed: int) -> np.ndarray:
    """Gradient-like matrix with subnormal-range entries and exact powers of two."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N), dtype=np.float32)
    a *= np.float32(1e-3)
    flat = a.reshape(-1)
    _scatter(rng, flat, 0.05, lambda n: (rng.standard_normal(n) * 1e-39).astype(np.float32))
    _scatter(rng, flat, 0.01,
             lambda n: (rng.choice([-1.0, 1.0], n) * np.exp2(rng.integers(-20, 1, n))).astype(np.float32))
    rows = min(32, M)
    if N >= 32:
        a[:rows, 0:32] = (rng.standard_normal((rows, 32)) * 1e-39).astype(np.float32)
    if N >= 64:
        a[:rows, 32:64] = (rng.choice([-1.0, 1.0], (rows, 32)) *
                           np.exp2(rng.integers(-30, 10, (rows, 32)))).astype(np.float32)
    return to_bf16_bits(a)


def moe_group_sizes(num_groups: int, total_rows: int, seed: int, zipf_s: float = 1.1,
                    forced_empty: int = 4, unit: int = 32) -> np.ndarray:
    """Ragged expert row counts: multiples of ``unit`` summing to ``total_rows``.

    ``total_rows/unit`` units are split by Zipf(s) weights over a seeded random
    permutation of ranks; ``forced_empty`` experts get no rows; the split is
    rounded down and the remaining units go to the largest fractional parts,
    so the sum is exact.
    """
    assert total_rows % unit == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    units = total_rows // unit
    empty = rng.choice(num_groups, size=min(forced_empty, num_groups), replace=False)
    live = np.setdiff1d(np.arange(num_groups), empty)
    ranks = rng.permutation(live.size) + 1
    w = 1.0 / ranks.astype(np.float64) ** zipf_s
    share = units * w / w.sum()
    base = np.floor(share).astype(np.int64)
    rest = units - int(base.sum())
    order = np.argsort(-(share - base), kind="stable")
    base[order[:rest]] += 1
    sizes = np.zeros(num_groups, np.int64)
    sizes[live] = base * unit
    assert int(sizes.sum()) == total_rows
    return sizes


def offsets_from_sizes(sizes: np.ndarray) -> np.ndarray:
    """Prefix sums [G+1] (int64) starting at 0."""
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


def moe_bf16(sizes: np.ndarray, N: int, seed: int) -> np.ndarray:
    """Concatenated expert inputs: N(0,1) scaled per expert by lognormal(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    total = int(sizes.sum())
    a = rng.standard_normal((total, N), dtype=np.float32)
    scale = rng.lognormal(0.0, 1.0, size=sizes.size).astype(np.float32)
    a *= np.repeat(scale, sizes)[:, None]
    return to_bf16_bits(a)


WORKLOADS = {
    # name: (M, N, fmt, with_dbias, grouped, seed)
    "small_128x256": (128, 256, E4M3, False, False, 0),
    "act_4096x4096": (4096, 4096, E4M3, False, False, 1),
    "fc1_8192x28672": (8192, 28672, E4M3, False, False, 2),
    "grad_16384x8192": (16384, 8192, E5M2, True, False, 3),
    "moe_64x65536x7168": (65536, 7168, E4M3, False, True, 4),
}


def make(name: str, seed: int | None = None, shape: tuple[int, int] | None = None):
    """Return ``dict(x=uint16 bits [M,N], fmt, with_dbias, offsets or None)`` for a named workload.

    ``shape`` draws the same value recipe at another (M, N) (total rows for the grouped one).
    """
    M, N, fmt, dbias, grouped, s0 = WORKLOADS[name]
    if shape is not None:
        M, N = shape
    seed = s0 if seed is None else seed
    offsets = None
    if name == "small_128x256":
        x = normal_bf16(M, N, seed)
    elif name == "act_4096x4096":
        x = act_bf16(M, N, seed)
    elif name == "fc1_8192x28672":
        x = fc1_bf16(M, N, seed)
    elif name == "grad_16384x8192":
        x = grad_bf16(M, N, seed)
    else:
        sizes = moe_group_sizes(64, M, seed)
        offsets = offsets_from_sizes(sizes)
        x = moe_bf16(sizes, N, seed)
    return dict(x=x, fmt=fmt, with_dbias=dbias, offsets=offsets, M=M, N=N)
