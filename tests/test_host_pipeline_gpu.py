"""mxfp8_quantize_host: host buffers in and out, pipelined over row chunks.

Its results must be byte-identical to mxfp8_quantize on the same data (dbias
too: the chunks fill one workspace and the same reduce runs once), and every
FP8 and scale byte must equal the CPU oracle's, dbias within 1e-5 * sum|x| of
the oracle's fp64 column sum.  Shapes are chosen so the call cuts the rows
into several chunks with a ragged last one; pageable host memory must give
the same bytes as pinned memory.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
import oracle_slices
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def device_reference(x_bits, fmt, with_dbias, rowwise=True, colwise=True):
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    r = mx.quantize(x, fmt, rowwise=rowwise, colwise=colwise, with_dbias=with_dbias)
    torch.cuda.synchronize()
    return [t.cpu() if t is not None else None for t in r]


@pytest.mark.parametrize("shape,fmt,with_dbias,pinned", [
    ((4192, 4096), mx.E4M3, False, True),     # 1024-row chunks, last one 96 rows
    ((1056, 28672), mx.E5M2, True, True),     # 128-row chunks, last one 32 rows
    ((1056, 28672), mx.E5M2, True, False),    # pageable host memory
    ((96, 160), mx.E4M3, True, True),         # a single chunk smaller than a tile
    ((4195, 4096), mx.E5M2, True, True),      # M not a multiple of 32: last chunk 99 rows
    ((1000, 1040), mx.E4M3, False, True),     # N = 16 mod 32
    ((1033, 1032), mx.E5M2, True, True),      # N = 8 mod 16: FP8 rows 8-byte aligned
])
def test_host_pipeline_matches_device_path(shape, fmt, with_dbias, pinned):
    M, N = shape
    x_bits = wl.grad_bf16(M, N, seed=M + N)
    want = device_reference(x_bits, fmt, with_dbias)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16)
    x_host = x_host.pin_memory() if pinned else x_host.clone()
    before = mx.mxfp8_kernel_launch_count()
    got = mx.quantize_host(x_host, fmt, with_dbias=with_dbias)
    torch.cuda.synchronize()
    assert mx.mxfp8_kernel_launch_count() > before
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col", "dbias"), got, want):
        if w is None:
            assert g is None
            continue
        assert torch.equal(g, w), name


@pytest.mark.parametrize("shape,fmt", [
    ((4195, 4096), mx.E5M2),      # five chunks, the last one 99 rows
    ((1033, 1032), mx.E4M3),      # N = 8 mod 16, ragged row and column blocks
])
def test_host_pipeline_matches_oracle(oracle_mod, shape, fmt):
    M, N = shape
    x_bits = wl.grad_bf16(M, N, seed=7 * M + N)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    got = mx.quantize_host(x_host, fmt, with_dbias=True)
    torch.cuda.synchronize()
    o_row, s_row, o_col, s_col, dbias = oracle_slices.quantize(oracle_mod, x_bits, fmt, with_dbias=True)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"),
                          (got.out_row, got.scale_row, got.out_col, got.scale_col),
                          (o_row, s_row, o_col, s_col)):
        assert np.array_equal(g.numpy(), w), name
    tol = 1e-5 * np.abs(torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().numpy()).sum(0)
    assert bool((np.abs(got.dbias.double().numpy() - dbias) <= tol).all())


def test_host_pipeline_single_direction_and_staging_reuse():
    M, N = 2080, 4096
    x_bits = wl.fc1_bf16(M, N, seed=3)
    want = device_reference(x_bits, mx.E4M3, False, rowwise=False, colwise=True)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    staging = torch.empty(mx.mxfp8_quantize_host_staging_bytes(M, N, False), dtype=torch.uint8, device="cuda")
    for _ in range(2):
        got = mx.quantize_host(x_host, mx.E4M3, rowwise=False, colwise=True, staging=staging)
        torch.cuda.synchronize()
        assert got.out_row is None
        assert torch.equal(got.out_col, want[2]) and torch.equal(got.scale_col, want[3])


# ---- the grouped cast with host buffers ---------------------------------------------------------

GROUPED_HOST_CASES = [
    # (rows, N, offsets): N = 16384 gives 1024-row chunks, so every case spans several chunks and
    # boundaries fall inside groups that do not start on a multiple of 32
    (5000, 16384, [0, 45, 45, 1500, 1533, 4001, 4700, 5000]),
    (4097, 16384, [0, 4097]),                                   # one group cut into every chunk
    (3000, 16384, [0] + [10 * i for i in range(1, 300)] + [3000]),  # 300 groups, most 10 rows
    (6144, 7168, [0, 1024, 1024, 2048, 4096, 6144]),            # 32-row-multiple groups, 2304-row chunks
]


def _grouped_host_input(rows, N, seed):
    return wl.grad_bf16(rows, N, seed=seed)


@pytest.mark.parametrize("case", range(len(GROUPED_HOST_CASES)))
@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_grouped_host_matches_device_path(case, act):
    rows, N, off = GROUPED_HOST_CASES[case]
    assert len(mx.mxfp8_grouped_host_chunks(off, rows, N)) > 3
    x_bits = _grouped_host_input(rows, N, seed=rows + case)
    off_t = torch.tensor(off, dtype=torch.int64)
    x_dev = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    want = mx.quantize_grouped(x_dev, off_t.cuda(), mx.E4M3, activation=act)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    before = mx.mxfp8_kernel_launch_count()
    got = mx.quantize_grouped_host(x_host, off_t, mx.E4M3, activation=act)
    torch.cuda.synchronize()
    assert mx.mxfp8_kernel_launch_count() > before
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got[:4], want[:4]):
        assert torch.equal(g, w.cpu()), name


def test_grouped_host_matches_oracle(oracle_mod):
    rows, N, off = GROUPED_HOST_CASES[0]
    x_bits = _grouped_host_input(rows, N, seed=99)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    got = mx.quantize_grouped_host(x_host, torch.tensor(off), mx.E5M2)
    torch.cuda.synchronize()
    want = oracle_mod.quantize_grouped(x_bits, np.array(off, np.int64), mx.E5M2)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got[:4], want[:4]):
        assert np.array_equal(g.numpy(), w), name


def test_grouped_host_pageable_single_direction_and_staging_reuse():
    rows, N, off = GROUPED_HOST_CASES[1]
    x_bits = _grouped_host_input(rows, N, seed=5)
    off_t = torch.tensor(off, dtype=torch.int64)
    x_dev = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    want = mx.quantize_grouped(x_dev, off_t.cuda(), mx.E4M3, rowwise=False, colwise=True)
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).clone()     # pageable
    staging = torch.empty(mx.mxfp8_quantize_grouped_host_staging_bytes(rows, N, 1), dtype=torch.uint8,
                          device="cuda")
    for _ in range(2):
        got = mx.quantize_grouped_host(x_host, off_t, mx.E4M3, rowwise=False, colwise=True, staging=staging)
        torch.cuda.synchronize()
        assert got.out_row is None and got.scale_row is None
        assert torch.equal(got.out_col, want.out_col.cpu()) and torch.equal(got.scale_col, want.scale_col.cpu())


# ---- the config call's options with host buffers ------------------------------------------------

@pytest.mark.parametrize("shape", [(4195, 16384), (1056, 28672), (300, 1032)])
@pytest.mark.parametrize("opts", [dict(swizzled=True), dict(with_amax=True), dict(activation="gelu"),
                                  dict(swizzled=True, with_amax=True, activation="relu"),
                                  dict(swizzled=True, activation="silu", colwise=False),
                                  dict(swizzled=True, with_dbias=True), dict(with_amax=True, with_dbias=True)])
def test_ex_host_matches_device_path(shape, opts):
    M, N = shape
    x_bits = wl.fc1_bf16(M, N, seed=M + 3 * N)
    kw = dict(opts)
    colwise = kw.pop("colwise", True)
    want = mx.quantize(torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda(), mx.E4M3,
                       colwise=colwise, **kw)
    torch.cuda.synchronize()
    x_host = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    before = mx.mxfp8_kernel_launch_count()
    got = mx.quantize_host(x_host, mx.E4M3, colwise=colwise, **kw)
    torch.cuda.synchronize()
    assert mx.mxfp8_kernel_launch_count() > before
    for name in ("out_row", "scale_row", "out_col", "scale_col", "dbias", "amax"):
        g, w = getattr(got, name), getattr(want, name)
        if w is None:
            assert g is None, name
            continue
        assert torch.equal(g, w.cpu()), name      # dbias too: the same partials and the same reduce


# ---- the two- and three-input calls with host buffers ------------------------------------------

@pytest.mark.parametrize("shape", [(3000, 8192), (300, 1032), (400, 28672)])
@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_two_input_host_calls_match_device_paths(shape, act):
    """Backward fusion (with dbias), gated cast and gated backward: host buffers give the device
    calls' bytes; 3000 x 8192 spans several chunks with a ragged last one, and 400 x 28672 gives the
    gated backward (6N bytes of input per row) chunks of 128 rows with no ramp."""
    M, N = shape
    g_bits = wl.grad_bf16(M, N, seed=M + N)
    x_bits = wl.normal_bf16(M, N, seed=N + 1)
    xg_bits = np.ascontiguousarray(np.concatenate([wl.normal_bf16(M, N, seed=5), wl.normal_bf16(M, N, seed=6)], 1))

    def host(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).pin_memory()

    def cuda(bits):
        return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()

    pairs = [
        (mx.quantize_dact(cuda(g_bits), cuda(x_bits), mx.E5M2, act, with_dbias=True),
         mx.quantize_dact_host(host(g_bits), host(x_bits), mx.E5M2, act, with_dbias=True)),
        (mx.quantize_gated(cuda(xg_bits), mx.E4M3, act), mx.quantize_gated_host(host(xg_bits), mx.E4M3, act)),
        (mx.quantize_dgated(cuda(g_bits), cuda(xg_bits), mx.E5M2, act),
         mx.quantize_dgated_host(host(g_bits), host(xg_bits), mx.E5M2, act)),
    ]
    torch.cuda.synchronize()
    for k, (want, got) in enumerate(pairs):
        for name in ("out_row", "scale_row", "out_col", "scale_col", "dbias"):
            w, g = getattr(want, name), getattr(got, name)
            if w is None:
                assert g is None, (k, name)
                continue
            assert torch.equal(g, w.cpu()), (k, name)
