"""The host pipelines' chunk plans and copy ranges, on the CPU.

mxfp8_quantize_host, mxfp8_quantize_ex_host and the two- and three-input host calls cut the rows
into chunks (chunk_plan in csrc/api.cu; the grouped call's plan, which adds a per-group move, is
exported as mxfp8_grouped_host_chunks and equals the flat plan for a single group).  This file checks
the plan's invariants over many shapes and restates each pipeline's host copy arithmetic (the same
expressions as csrc/api.cu) to check that the chunks' copies cover every byte of every host buffer
exactly once and stay in bounds, plain and GEMM-ready layouts alike.  It computes nothing of the
method.
"""
import pytest

import mxfp8_block_scaled_04_gb300 as mx

BM = 128
CHUNK_BYTES = 32 << 20


def rows_chunk(M, in_bytes_per_row):
    r = max(BM, CHUNK_BYTES // in_bytes_per_row // BM * BM)
    return min(r, -(-M // BM) * BM)


def flat_plan(M, N):
    """The flat pipeline's boundaries, through the grouped export with one group."""
    return mx.mxfp8_grouped_host_chunks([0, M], M, N)


def cover(size, ranges):
    """The byte ranges (start, length) tile [0, size) exactly: sorted, each starts where the last ended."""
    pos = 0
    for a, n in sorted(ranges):
        assert n > 0 and a == pos, (a, n, pos, size)
        pos = a + n
    assert pos == size, (pos, size)


SHAPES = [(1, 8), (127, 64), (128, 64), (129, 64), (4195, 4096), (8192, 28672), (1056, 28672), (300, 1032),
          (5000, 200000), (100000, 256), (33, 131072)]


@pytest.mark.parametrize("M,N", SHAPES)
def test_flat_plan_invariants(M, N):
    b = flat_plan(M, N)
    R = rows_chunk(M, 2 * N)
    assert b[0] == 0 and b[-1] == M and all(x < y for x, y in zip(b, b[1:]))
    assert all(x % BM == 0 for x in b[:-1])                   # every chunk starts on a 128-row tile
    assert all(y - x <= R for x, y in zip(b, b[1:]))          # fits a slot


@pytest.mark.parametrize("M,N", SHAPES)
@pytest.mark.parametrize("swz", [False, True])
def test_flat_pipeline_copies_cover_the_host_buffers(M, N, swz):
    b = flat_plan(M, N)
    Cn = -(-N // 32)
    row_tiles, col_tiles = -(-M // BM), -(-N // 128)
    x, o_r, o_c, s_r, s_c = [], [], [], [], []
    for r0, r1 in zip(b, b[1:]):
        rows = r1 - r0
        x.append((r0 * N * 2, rows * N * 2))
        o_r.append((r0 * N, rows * N))
        o_c.append((r0 * N, rows * N))
        rt0, crt = r0 // BM, -(-rows // BM)
        if swz:
            s_r.append((rt0 * col_tiles * 512, crt * col_tiles * 512))
            for i in range(col_tiles):                         # the strided copy: one band per tile row
                s_c.append((i * row_tiles * 512 + rt0 * 512, crt * 512))
        else:
            s_r.append((r0 * Cn, rows * Cn))
            s_c.append((r0 // 32 * N, -(-rows // 32) * N))
    cover(M * N * 2, x)
    cover(M * N, o_r)
    cover(M * N, o_c)
    if swz:
        cover(mx.mxfp8_scale_bytes(M, Cn, mx.SCALES_SWIZZLED), s_r)
        cover(mx.mxfp8_scale_bytes(N, -(-M // 32), mx.SCALES_SWIZZLED), s_c)
    else:
        cover(M * Cn, s_r)
        cover(-(-M // 32) * N, s_c)


@pytest.mark.parametrize("M,N", [(3000, 8192), (300, 1032), (400, 28672), (8192, 28672), (129, 64)])
@pytest.mark.parametrize("which", ["dact", "gated", "dgated"])
def test_two_input_pipeline_copies_cover_the_host_buffers(M, N, which):
    b0, b1, W, SR = {"dact": (2 * N, 2 * N, N, -(-N // 32)), "gated": (4 * N, 0, N, -(-N // 32)),
                     "dgated": (2 * N, 4 * N, 2 * N, 2 * -(-N // 32))}[which]
    R = rows_chunk(M, b0 + b1)
    # the rows pipeline uses the flat plan for chunk rows R; rebuild it through the export, whose
    # chunk rows come from 2N bytes per row: pick the N' with the same R
    Np = max(8, (CHUNK_BYTES // R) // 2 // 8 * 8)
    assert rows_chunk(M, 2 * Np) == R
    b = flat_plan(M, Np)
    assert all(y - x <= R for x, y in zip(b, b[1:]))
    ins0, ins1, outs, srs, scs = [], [], [], [], []
    for r0, r1 in zip(b, b[1:]):
        rows = r1 - r0
        ins0.append((r0 * b0, rows * b0))
        if b1:
            ins1.append((r0 * b1, rows * b1))
        outs.append((r0 * W, rows * W))
        srs.append((r0 * SR, rows * SR))
        scs.append((r0 // 32 * W, -(-rows // 32) * W))
    cover(M * b0, ins0)
    if b1:
        cover(M * b1, ins1)
    cover(M * W, outs)
    cover(M * SR, srs)
    cover(-(-M // 32) * W, scs)


@pytest.mark.parametrize("off,N", [([0, 45, 45, 1500, 1533, 4001, 4700, 5000], 16384), ([0, 4097], 16384),
                                   ([0] + [10 * i for i in range(1, 300)] + [3000], 16384),
                                   ([0, 1024, 1024, 2048, 4096, 6144], 7168), ([0, 37, 5000], 200000)])
def test_grouped_pipeline_copies_cover_the_host_buffers(off, N):
    """mxfp8_quantize_grouped_host: rows and the chunk's columnwise scale rows (sum over the groups
    clipped to the chunk of ceil(rows / 32), placed after the previous chunks') tile the outputs."""
    M = off[-1]
    b = mx.mxfp8_grouped_host_chunks(off, M, N)
    Cn = -(-N // 32)
    rows_r, srow_r, scol_r, s0 = [], [], [], 0
    for r0, r1 in zip(b, b[1:]):
        rows_r.append((r0 * N, (r1 - r0) * N))
        srow_r.append((r0 * Cn, (r1 - r0) * Cn))
        sc = sum(-(-(min(max(e, r0), r1) - min(max(a, r0), r1)) // 32) for a, e in zip(off, off[1:]))
        if sc:
            scol_r.append((s0 * N, sc * N))
        s0 += sc
    cover(M * N, rows_r)
    cover(M * Cn, srow_r)
    cover(mx.grouped_scale_col_rows(off) * N, scol_r)
