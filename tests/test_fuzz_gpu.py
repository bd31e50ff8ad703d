"""Seeded random sweep against the oracle.

Each case draws a shape (M any in 1..699, N a multiple of 8 up to 1200), a format, the directions,
and the options (dbias, GEMM-ready scales, amax), plus one of the value recipes, and compares every
FP8 byte and scale byte with the oracle (dbias within 1e-5 * sum |x| per column, amax exactly).
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

CASES = 48


def draw(i):
    rng = np.random.Generator(np.random.PCG64(7000 + i))
    M = int(rng.integers(1, 700))
    N = 8 * int(rng.integers(1, 151))
    fmt = int(rng.integers(0, 2))
    dirs = int(rng.integers(1, 4))  # 1 rowwise, 2 columnwise, 3 both
    opts = dict(with_dbias=bool(rng.integers(0, 2)), swizzled=bool(rng.integers(0, 2)),
                with_amax=bool(rng.integers(0, 2)))
    recipe = int(rng.integers(0, 4 if N % 32 == 0 else 3))
    gen = [wl.normal_bf16, wl.grad_bf16, wl.fc1_bf16, wl.act_bf16][recipe]
    return M, N, fmt, dirs, opts, gen(M, N, 100 + i)


@pytest.mark.gpu
@pytest.mark.parametrize("i", range(CASES))
def test_random_case(oracle_mod, i):
    M, N, fmt, dirs, opts, x_bits = draw(i)
    row, col = bool(dirs & 1), bool(dirs & 2)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    r = mx.quantize(x, fmt, rowwise=row, colwise=col, **opts)
    torch.cuda.synchronize()
    o_row, s_row, o_col, s_col, db = oracle_mod.quantize(x_bits, fmt, rowwise=row, colwise=col,
                                                         with_dbias=opts["with_dbias"])
    swz = oracle_mod.swizzle_scales if opts["swizzled"] else (lambda s: s)
    if row:
        assert np.array_equal(r.out_row.cpu().numpy(), o_row)
        assert np.array_equal(r.scale_row.cpu().numpy(), swz(s_row))
    if col:
        assert np.array_equal(r.out_col.cpu().numpy(), o_col)
        want_col = swz(np.ascontiguousarray(s_col.T)) if opts["swizzled"] else s_col
        assert np.array_equal(r.scale_col.cpu().numpy(), want_col)
    if opts["with_dbias"]:
        xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().abs().sum(0).numpy()
        assert np.all(np.abs(r.dbias.cpu().numpy().astype(np.float64) - db) <= 1e-5 * xv)
    if opts["with_amax"]:
        assert float(r.amax.item()) == oracle_mod.amax(x_bits)


def test_draws_cover_the_options():
    seen = set()
    for i in range(CASES):
        M, N, fmt, dirs, opts, _ = draw(i)
        seen |= {("fmt", fmt), ("dirs", dirs), ("ragged_M", M % 32 != 0), ("ragged_N", N % 32 != 0),
                 ("N_8_mod_16", N % 16 == 8)}
        seen |= {(k, v) for k, v in opts.items()}
    for need in [("fmt", 0), ("fmt", 1), ("dirs", 1), ("dirs", 2), ("dirs", 3), ("ragged_M", True),
                 ("ragged_N", True), ("N_8_mod_16", True), ("with_dbias", True), ("swizzled", True),
                 ("with_amax", True)]:
        assert need in seen, need
