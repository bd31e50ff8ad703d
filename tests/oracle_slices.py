"""The CPU oracle over a whole large matrix, on every host core.

The oracle is plain scalar C and releases the GIL inside each call, so running
it on column slices in threads uses every core.  A slice starts on a multiple
of 32 columns and spans every row, so it holds whole 1x32 rowwise blocks,
whole 32x1 columnwise blocks and whole columns: the outputs of the slices,
placed side by side, are the oracle's outputs for the whole matrix byte for
byte, and each column's dbias is that column's own sum.  Nothing here computes
anything itself; it only cuts, calls and reassembles.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np


def host_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return os.cpu_count() or 1


def column_bounds(N: int, parts: int):
    """Boundaries 0 = b0 < b1 < ... = N, inner ones multiples of 32, at most `parts` slices."""
    blocks = -(-N // 32)
    parts = max(1, min(parts, blocks))
    b = sorted({min(N, 32 * (blocks * k // parts)) for k in range(parts + 1)})
    return [(b[i], b[i + 1]) for i in range(len(b) - 1) if b[i + 1] > b[i]]


def _run(fn, x_bits, threads):
    M, N = x_bits.shape
    slices = column_bounds(N, 4 * (threads or host_threads()))

    def one(jj):
        j0, j1 = jj
        return fn(np.ascontiguousarray(x_bits[:, j0:j1]))

    with ThreadPoolExecutor(max_workers=threads or host_threads()) as pool:
        return slices, list(pool.map(one, slices))


def quantize(oracle, x_bits, fmt, rowwise=True, colwise=True, with_dbias=False, threads=None):
    """oracle.quantize on the whole matrix, computed slice by slice in parallel."""
    M, N = x_bits.shape
    slices, parts = _run(lambda xs: oracle.quantize(xs, fmt, rowwise, colwise, with_dbias), x_bits, threads)
    out_row = np.empty((M, N), np.uint8) if rowwise else None
    scale_row = np.empty((M, -(-N // 32)), np.uint8) if rowwise else None
    out_col = np.empty((M, N), np.uint8) if colwise else None
    scale_col = np.empty((-(-M // 32), N), np.uint8) if colwise else None
    dbias = np.empty((N,), np.float32) if with_dbias else None
    for (j0, j1), (o_r, s_r, o_c, s_c, db) in zip(slices, parts):
        if rowwise:
            out_row[:, j0:j1] = o_r
            scale_row[:, j0 // 32:j0 // 32 + s_r.shape[1]] = s_r
        if colwise:
            out_col[:, j0:j1] = o_c
            scale_col[:, j0:j1] = s_c
        if with_dbias:
            dbias[j0:j1] = db
    return out_row, scale_row, out_col, scale_col, dbias


def quantize_grouped(oracle, x_bits, offsets, fmt, threads=None):
    """oracle.quantize_grouped on the whole matrix (groups are row ranges, so column slices keep them)."""
    M, N = x_bits.shape
    slices, parts = _run(lambda xs: oracle.quantize_grouped(xs, offsets, fmt), x_bits, threads)
    out_row = np.empty((M, N), np.uint8)
    scale_row = np.empty((M, -(-N // 32)), np.uint8)
    out_col = np.empty((M, N), np.uint8)
    scale_col = np.empty((oracle.grouped_scale_col_rows(offsets), N), np.uint8)
    for (j0, j1), (o_r, s_r, o_c, s_c) in zip(slices, parts):
        out_row[:, j0:j1] = o_r
        scale_row[:, j0 // 32:j0 // 32 + s_r.shape[1]] = s_r
        out_col[:, j0:j1] = o_c
        scale_col[:, j0:j1] = s_c
    return out_row, scale_row, out_col, scale_col


def grouped_dbias(oracle, x_bits, offsets, threads=None):
    """oracle.grouped_dbias [G, N] computed on column slices in parallel."""
    M, N = x_bits.shape
    slices, parts = _run(lambda xs: oracle.grouped_dbias(xs, offsets), x_bits, threads)
    out = np.empty((len(offsets) - 1, N), np.float32)
    for (j0, j1), d in zip(slices, parts):
        out[:, j0:j1] = d
    return out
