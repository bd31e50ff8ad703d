"""The quantize calls inside a captured CUDA graph.

Each call is made once outside capture (the first call on a device sets up
kernel attributes), then captured with torch.cuda.graph; the input is
overwritten in place and the graph replayed: the outputs must match the
oracle on the new input, so the captured launches read the live buffers.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def run_graph(call, x, new_bits):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert call(s) == 0                     # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        status = call(s)
    assert status == 0
    x.copy_(bf16(new_bits).cuda())
    g.replay()
    torch.cuda.synchronize()


def test_graph_plain_and_dbias(oracle_mod):
    M, N = 1056, 1024
    x = bf16(wl.normal_bf16(M, N, seed=1)).cuda()
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = [torch.empty((M, N), **u8), torch.empty((M, N // 32), **u8), torch.empty((M, N), **u8),
         torch.empty((M // 32, N), **u8)]
    dbias = torch.empty((N,), dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.mxfp8_quantize_workspace_bytes(M, N, True), **u8)
    new = wl.grad_bf16(M, N, seed=2)
    run_graph(lambda s: mx.mxfp8_quantize(x, M, N, mx.E5M2, *o, dbias, ws, None, s), x, new)
    want = oracle_mod.quantize(new, mx.E5M2, with_dbias=True)
    for g, w in zip(o, want[:4]):
        assert np.array_equal(g.cpu().numpy(), w)
    xv = torch.from_numpy(new.view(np.int16)).view(torch.bfloat16).double().abs().sum(0).numpy()
    assert np.all(np.abs(dbias.cpu().numpy().astype(np.float64) - want[4]) <= 1e-5 * xv)


def test_graph_ex_swizzled_amax(oracle_mod):
    M, N = 544, 1056
    x = bf16(wl.normal_bf16(M, N, seed=3)).cuda()
    u8 = dict(dtype=torch.uint8, device="cuda")
    orow, ocol = torch.empty((M, N), **u8), torch.empty((M, N), **u8)
    srow = torch.empty((mx.mxfp8_scale_bytes(M, N // 32, mx.SCALES_SWIZZLED),), **u8)
    scol = torch.empty((mx.mxfp8_scale_bytes(N, M // 32, mx.SCALES_SWIZZLED),), **u8)
    amax = torch.empty((1,), dtype=torch.float32, device="cuda")
    cfg = mx.make_config(x, M, N, mx.E4M3, orow, srow, ocol, scol, scale_layout=mx.SCALES_SWIZZLED, amax=amax)
    new = wl.act_bf16(M, N, seed=4)
    run_graph(lambda s: mx.mxfp8_quantize_ex(cfg, s), x, new)
    o_row, s_row, o_col, s_col, _ = oracle_mod.quantize(new, mx.E4M3)
    assert np.array_equal(orow.cpu().numpy(), o_row) and np.array_equal(ocol.cpu().numpy(), o_col)
    assert np.array_equal(srow.cpu().numpy(), oracle_mod.swizzle_scales(s_row))
    assert np.array_equal(scol.cpu().numpy(), oracle_mod.swizzle_scales(np.ascontiguousarray(s_col.T)))
    assert float(amax.item()) == oracle_mod.amax(new)


def test_graph_grouped(oracle_mod):
    sizes = np.array([64, 0, 96, 32, 128], np.int64)
    off_np = wl.offsets_from_sizes(sizes)
    total, N = int(sizes.sum()), 192
    x = bf16(wl.moe_bf16(sizes, N, seed=5)).cuda()
    off = torch.from_numpy(off_np).cuda()
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = [torch.empty((total, N), **u8), torch.empty((total, N // 32), **u8), torch.empty((total, N), **u8),
         torch.empty((total // 32, N), **u8)]
    new = wl.moe_bf16(sizes, N, seed=6)
    run_graph(lambda s: mx.mxfp8_quantize_grouped(x, total, N, len(sizes), off, mx.E4M3, *o, None, None, None, s),
              x, new)
    for g, w in zip(o, oracle_mod.quantize_grouped(new, off_np, mx.E4M3)):
        assert np.array_equal(g.cpu().numpy(), w)


def test_graph_gated_and_its_backward(oracle_mod):
    M, N = 160, 96
    x = bf16(np.concatenate([wl.normal_bf16(M, N, seed=5), wl.normal_bf16(M, N, seed=6)], axis=1)).cuda()
    g = bf16(wl.grad_bf16(M, N, seed=7)).cuda()
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = [torch.empty((M, N), **u8), torch.empty((M, N // 32), **u8), torch.empty((M, N), **u8),
         torch.empty((M // 32, N), **u8)]
    od = [torch.empty((M, 2 * N), **u8), torch.empty((M, 2 * N // 32), **u8), torch.empty((M, 2 * N), **u8),
          torch.empty((M // 32, 2 * N), **u8)]
    new = np.concatenate([wl.normal_bf16(M, N, seed=8), wl.normal_bf16(M, N, seed=9)], axis=1)

    def both(s):   # ReGLU and its backward: exact, so bytes must match the oracle
        st = mx.mxfp8_quantize_gated(x, M, N, mx.E4M3, "relu", *o, None, s)
        return st or mx.mxfp8_quantize_dgated(g, x, M, N, mx.E5M2, "relu", *od, None, s)
    run_graph(both, x, new)
    for got, want in zip(o, oracle_mod.quantize_gated(new, mx.E4M3, 1)):
        assert np.array_equal(got.cpu().numpy(), want)
    g_bits = g.cpu().view(torch.int16).numpy().view(np.uint16)
    for got, want in zip(od, oracle_mod.quantize_dgated(g_bits, new, mx.E5M2, 1)):
        assert np.array_equal(got.cpu().numpy(), want)
