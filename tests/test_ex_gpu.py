"""mxfp8_quantize_ex on the GPU: GEMM-ready (swizzled) scale planes and the amax output.

The swizzled planes must equal the oracle's plain scales run through the
oracle's swizzle (rowwise: rows = M, scale columns = N/32; columnwise: the
transposed operand, rows = N, scale columns = M/32), padding zeroed; the FP8
bytes must equal the plain call's; amax must equal max |x| exactly.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.parametrize("shape,fmt", [((256, 256), 0), ((96, 160), 1), ((160, 96), 0), ((1056, 288), 1),
                                       ((8192, 1024), 0)])
def test_swizzled_scales_and_amax(oracle_mod, shape, fmt):
    M, N = shape
    x_bits = wl.grad_bf16(M, N, seed=M ^ N) if fmt else wl.act_bf16(M, N, seed=M ^ N)
    x = dev(x_bits)
    u8 = dict(dtype=torch.uint8, device="cuda")
    srow = torch.full((mx.mxfp8_scale_bytes(M, N // 32, mx.SCALES_SWIZZLED),), 0xFF, **u8)   # NaN bytes
    scol = torch.full((mx.mxfp8_scale_bytes(N, M // 32, mx.SCALES_SWIZZLED),), 0xFF, **u8)
    orow, ocol = torch.empty((M, N), **u8), torch.empty((M, N), **u8)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    cfg = mx.make_config(x, M, N, fmt, orow, srow, ocol, scol, scale_layout=mx.SCALES_SWIZZLED, amax=amax)
    assert mx.mxfp8_quantize_ex(cfg, None) == 0
    torch.cuda.synchronize()
    o_row, s_row, o_col, s_col, _ = oracle_mod.quantize(x_bits, fmt)
    assert np.array_equal(orow.cpu().numpy(), o_row)
    assert np.array_equal(ocol.cpu().numpy(), o_col)
    assert np.array_equal(srow.cpu().numpy(), oracle_mod.swizzle_scales(s_row))
    assert np.array_equal(scol.cpu().numpy(), oracle_mod.swizzle_scales(np.ascontiguousarray(s_col.T)))
    assert float(amax.item()) == oracle_mod.amax(x_bits)


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_amax_one_direction_plain_layout(oracle_mod, rowwise, colwise):
    x_bits = wl.act_bf16(544, 1056, seed=4)
    r = mx.quantize(dev(x_bits), mx.E4M3, rowwise=rowwise, colwise=colwise, with_amax=True)
    torch.cuda.synchronize()
    assert float(r.amax.item()) == oracle_mod.amax(x_bits)
    o = oracle_mod.quantize(x_bits, mx.E4M3, rowwise, colwise)
    for g, w in zip(r[:4], o[:4]):
        if w is not None:
            assert np.array_equal(g.cpu().numpy(), w)


def test_ex_with_dbias_swizzled_matches_plain(oracle_mod):
    x_bits = wl.grad_bf16(4096, 512, seed=8)
    x = dev(x_bits)
    plain = mx.quantize(x, mx.E5M2, with_dbias=True)
    swz = mx.quantize(x, mx.E5M2, with_dbias=True, swizzled=True, with_amax=True)
    torch.cuda.synchronize()
    assert torch.equal(plain.out_row, swz.out_row) and torch.equal(plain.out_col, swz.out_col)
    assert torch.equal(plain.dbias, swz.dbias)
    assert np.array_equal(swz.scale_row.cpu().numpy(), oracle_mod.swizzle_scales(plain.scale_row.cpu().numpy()))


def test_ex_noop_leaves_amax_and_padding_untouched():
    x = dev(wl.normal_bf16(96, 160, seed=2))
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    srow = torch.full((mx.mxfp8_scale_bytes(96, 5, 1),), 0x3C, **u8)
    orow = torch.full((96, 160), 0x3C, **u8)
    amax = torch.full((1,), 7.0, dtype=torch.float32, device="cuda")
    cfg = mx.make_config(x, 96, 160, 0, orow, srow, noop=one, scale_layout=1, amax=amax)
    assert mx.mxfp8_quantize_ex(cfg, None) == 0
    torch.cuda.synchronize()
    assert bool((srow == 0x3C).all()) and bool((orow == 0x3C).all()) and float(amax.item()) == 7.0


@pytest.mark.parametrize("shape", [(45, 80), (130, 144), (257, 4112), (96, 40), (33, 8), (129, 1032)])
def test_swizzled_ragged_shapes(oracle_mod, shape):
    M, N = shape
    x_bits = wl.act_bf16(M, N, seed=M + N) if M % 32 == 0 and N % 32 == 0 else wl.grad_bf16(M, N, seed=M + N)
    r = mx.quantize(dev(x_bits), mx.E4M3, swizzled=True, with_amax=True)
    torch.cuda.synchronize()
    o_row, s_row, o_col, s_col, _ = oracle_mod.quantize(x_bits, mx.E4M3)
    assert np.array_equal(r.out_row.cpu().numpy(), o_row) and np.array_equal(r.out_col.cpu().numpy(), o_col)
    assert np.array_equal(r.scale_row.cpu().numpy(), oracle_mod.swizzle_scales(s_row))
    assert np.array_equal(r.scale_col.cpu().numpy(), oracle_mod.swizzle_scales(np.ascontiguousarray(s_col.T)))
    assert float(r.amax.item()) == oracle_mod.amax(x_bits)
