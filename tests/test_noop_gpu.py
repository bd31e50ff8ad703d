"""The device noop flag on every entry point that the other tests do not cover.

With *noop == 1.0f every kernel of the call returns before writing: outputs, scale planes and dbias
keep their prefill.  With *noop == 0 the same call writes them (so the prefill check is not vacuous).
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

U8 = dict(dtype=torch.uint8, device="cuda")


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def outputs(M, N):
    return [torch.full((M, N), 0x3C, **U8), torch.full((M, N // 32), 0x3C, **U8),
            torch.full((M, N), 0x3C, **U8), torch.full((M // 32, N), 0x3C, **U8)]


def flags():
    return (torch.ones(1, dtype=torch.float32, device="cuda"), torch.zeros(1, dtype=torch.float32, device="cuda"))


def untouched(ts, dbias=None):
    torch.cuda.synchronize()
    return all(bool((t == 0x3C).all()) for t in ts) and (dbias is None or bool((dbias == 3.0).all()))


def refill(ts, dbias=None):
    for t in ts:
        t.fill_(0x3C)
    if dbias is not None:
        dbias.fill_(3.0)


def test_noop_backward_fusion_with_dbias():
    M, N = 256, 192
    dy, x = dev(wl.grad_bf16(M, N, seed=1)), dev(wl.normal_bf16(M, N, seed=2))
    o = outputs(M, N)
    dbias = torch.full((N,), 3.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.mxfp8_quantize_workspace_bytes(M, N, True), **U8)
    one, zero = flags()
    for act in ("relu", "gelu"):
        a = mx.binding.ACTIVATIONS[act]
        assert mx.mxfp8_quantize_dact(dy, x, M, N, 1, a, *o, dbias, ws, one, None) == 0
        assert untouched(o, dbias), act
        assert mx.mxfp8_quantize_dact(dy, x, M, N, 1, a, *o, dbias, ws, zero, None) == 0
        assert not untouched(o) and not bool((dbias == 3.0).all()), act
        refill(o, dbias)


def test_noop_grouped_dbias():
    sizes = np.array([64, 0, 128, 32], np.int64)
    total, N, G = int(sizes.sum()), 96, len(sizes)
    x = dev(wl.moe_bf16(sizes, N, seed=3))
    off = torch.from_numpy(wl.offsets_from_sizes(sizes)).cuda()
    o = outputs(total, N)
    dbias = torch.full((G, N), 3.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.mxfp8_quantize_grouped_dbias_workspace_bytes(total, N, G), **U8)
    one, zero = flags()
    assert mx.mxfp8_quantize_grouped_dbias(x, total, N, G, off, 0, *o, dbias, ws, one, None, None) == 0
    assert untouched(o, dbias)
    assert mx.mxfp8_quantize_grouped_dbias(x, total, N, G, off, 0, *o, dbias, ws, zero, None, None) == 0
    assert not untouched(o) and not bool((dbias == 3.0).all())


@pytest.mark.parametrize("act", ["relu", "silu"])
def test_noop_activation_variants(act):
    M, N = 160, 256
    x = dev(wl.act_bf16(M, N, seed=4))
    o = outputs(M, N)
    amax = torch.full((1,), 3.0, dtype=torch.float32, device="cuda")
    one, zero = flags()
    cfg = mx.make_config(x, M, N, 0, *o, noop=one, amax=amax, activation=act)
    assert mx.mxfp8_quantize_ex(cfg, None) == 0
    assert untouched(o, amax)
    cfg = mx.make_config(x, M, N, 0, *o, noop=zero, amax=amax, activation=act)
    assert mx.mxfp8_quantize_ex(cfg, None) == 0
    assert not untouched(o) and not bool((amax == 3.0).all())

