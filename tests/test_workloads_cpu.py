"""Seeded input generators (CPU): the large banded matrix is its block times one power of two per band."""
import numpy as np
import torch

from mxfp8_block_scaled_04_gb300 import workloads as wl


def as_float(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def test_banded_bands_are_exact_power_of_two_multiples():
    M, N, band = 1000, 96, 256
    x = as_float(wl.banded_bf16(M, N, seed=5, band=band))
    block = as_float(wl.normal_bf16(band, N, seed=5))
    block = np.where(np.abs(block) <= 2.0 ** -118, np.copysign(1.0, block), block)
    for b in range((M + band - 1) // band):
        rows = x[b * band:(b + 1) * band]
        ratio = rows / block[:rows.shape[0]]
        k = np.log2(np.abs(ratio[0, 0]))
        assert k == round(k) and -8 <= k <= 8
        assert np.all(ratio == ratio[0, 0])
    assert np.all(np.abs(x) >= 2.0 ** -126) and np.all(np.isfinite(x))


def test_banded_is_deterministic():
    assert np.array_equal(wl.banded_bf16(300, 32, seed=9), wl.banded_bf16(300, 32, seed=9))
