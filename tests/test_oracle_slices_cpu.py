"""The parallel column-slice driver of the oracle reassembles the whole-matrix result exactly.

The full-size GPU parity tests compare against tests/oracle_slices.py; here it is
pinned to the oracle's own single call, byte for byte (dbias bit for bit), on
shapes whose slices cut through rowwise blocks' neighbours, end on a partial
block, and cross group boundaries.
"""
import numpy as np
import pytest

import oracle_slices
from mxfp8_block_scaled_04_gb300 import workloads as wl


@pytest.mark.parametrize("shape,threads", [((96, 1008), 3), ((45, 80), 2), ((64, 4096), 5), ((33, 16), 4)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_slices_equal_whole_matrix(oracle_mod, shape, threads, fmt):
    M, N = shape
    x = wl.normal_bf16(M, N, seed=M + N + fmt, std=3.0)
    want = oracle_mod.quantize(x, fmt, with_dbias=True)
    got = oracle_slices.quantize(oracle_mod, x, fmt, with_dbias=True, threads=threads)
    for g, w in zip(got, want):
        assert np.array_equal(g, w)


@pytest.mark.parametrize("N", [224, 200, 40])
def test_slices_grouped_equal_whole_matrix(oracle_mod, N):
    sizes = np.array([64, 0, 32, 416, 0, 128, 96], np.int64)
    off = wl.offsets_from_sizes(sizes)
    x = wl.moe_bf16(sizes, N, seed=4)
    for g, w in zip(oracle_slices.quantize_grouped(oracle_mod, x, off, 0, threads=3),
                    oracle_mod.quantize_grouped(x, off, 0)):
        assert np.array_equal(g, w)
    # the grouped oracle is the flat oracle on the concatenated rows, partial last blocks included
    for g, w in zip(oracle_mod.quantize_grouped(x, off, 0), oracle_mod.quantize(x, 0)[:4]):
        assert np.array_equal(g, w)
    assert np.array_equal(oracle_slices.grouped_dbias(oracle_mod, x, off, threads=3),
                          oracle_mod.grouped_dbias(x, off))


def test_column_bounds_cover_and_align():
    for N in (16, 32, 80, 1008, 28672, 7168):
        for parts in (1, 3, 7, 64):
            b = oracle_slices.column_bounds(N, parts)
            assert b[0][0] == 0 and b[-1][1] == N
            assert all(b[i][1] == b[i + 1][0] for i in range(len(b) - 1))
            assert all(j0 % 32 == 0 and j1 > j0 for j0, j1 in b)
