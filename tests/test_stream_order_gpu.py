"""Back-to-back calls on one stream into the same buffers.

The kernels are launched for programmatic dependent launch: each may start while the previous one
drains and must wait on the device before touching global memory.  Alternating two inputs into the
same outputs and workspace, with no synchronisation between calls, checks that no write of an
earlier call lands after a later call's (outputs), and that no quantize kernel overwrites the dbias
workspace while the previous call's reduce still reads it.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def test_alternating_inputs_same_buffers_with_dbias(oracle_mod):
    M, N, fmt = 4096, 2048, 1
    a_bits, b_bits = wl.grad_bf16(M, N, seed=11), wl.normal_bf16(M, N, seed=12)
    xa, xb = dev(a_bits), dev(b_bits)
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = [torch.empty((M, N), **u8), torch.empty((M, N // 32), **u8), torch.empty((M, N), **u8),
         torch.empty((M // 32, N), **u8)]
    dbias = torch.empty((N,), dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.mxfp8_quantize_workspace_bytes(M, N, True), **u8)
    for i in range(41):  # ends on xa
        x = xa if i % 2 == 0 else xb
        assert mx.mxfp8_quantize(x, M, N, fmt, *o, dbias, ws, None, None) == 0
    torch.cuda.synchronize()
    want = oracle_mod.quantize(a_bits, fmt, with_dbias=True)
    for g, w in zip(o, want[:4]):
        assert np.array_equal(g.cpu().numpy(), w)
    xv = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16).double().abs().sum(0).numpy()
    assert np.all(np.abs(dbias.cpu().numpy().astype(np.float64) - want[4]) <= 1e-5 * xv)


def test_alternating_grouped_dbias_same_workspace(oracle_mod):
    sizes_a = np.array([256, 0, 992, 32, 768], np.int64)
    sizes_b = np.array([32, 1024, 0, 992, 0], np.int64)
    N, fmt = 512, 0
    off_a, off_b = wl.offsets_from_sizes(sizes_a), wl.offsets_from_sizes(sizes_b)
    a_bits, b_bits = wl.moe_bf16(sizes_a, N, seed=3), wl.moe_bf16(sizes_b, N, seed=4)
    total = int(sizes_a.sum())
    assert total == int(sizes_b.sum())
    xa, xb = dev(a_bits), dev(b_bits)
    oa, ob = torch.from_numpy(off_a).cuda(), torch.from_numpy(off_b).cuda()
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = [torch.empty((total, N), **u8), torch.empty((total, N // 32), **u8), torch.empty((total, N), **u8),
         torch.empty((total // 32, N), **u8)]
    G = len(sizes_a)
    dbias = torch.empty((G, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.mxfp8_quantize_grouped_dbias_workspace_bytes(total, N, G), **u8)
    for i in range(41):  # ends on a
        x, off = (xa, oa) if i % 2 == 0 else (xb, ob)
        assert mx.mxfp8_quantize_grouped_dbias(x, total, N, G, off, fmt, *o, dbias, ws, None, None, None) == 0
    torch.cuda.synchronize()
    for g, w in zip(o, oracle_mod.quantize_grouped(a_bits, off_a, fmt)):
        assert np.array_equal(g.cpu().numpy(), w)
    want = oracle_mod.grouped_dbias(a_bits, off_a)
    xv = torch.from_numpy(a_bits.view(np.int16)).view(torch.bfloat16).double().abs().numpy()
    got = dbias.cpu().numpy().astype(np.float64)
    for g in range(G):
        assert np.all(np.abs(got[g] - want[g]) <= 1e-5 * xv[off_a[g]:off_a[g + 1]].sum(0)), g


def test_concurrent_host_threads_on_their_own_streams():
    """Several host threads enqueue calls at once, each on its own stream and buffers, the first
    call of some variants among them (the per-variant set-up runs under a lock): every thread's
    outputs equal a single-threaded call's."""
    import threading
    M, N = 2048, 4096
    inputs = [wl.normal_bf16(M, N, seed=40 + t) for t in range(4)]
    variants = [dict(), dict(swizzled=True), dict(activation="silu"), dict(with_amax=True, activation="relu")]
    ref = []
    for t, bits in enumerate(inputs):
        r = mx.quantize(dev(bits), mx.E4M3, **variants[t])
        torch.cuda.synchronize()
        ref.append([v.cpu() if v is not None else None for v in r])
    results, errors = [None] * 4, []

    def work(t):
        try:
            s = torch.cuda.Stream()
            x = dev(inputs[t])
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                for _ in range(20):
                    r = mx.quantize(x, mx.E4M3, stream=s, **variants[t])
            s.synchronize()
            results[t] = [v.cpu() if v is not None else None for v in r]
        except Exception as e:  # reported on the main thread
            errors.append((t, e))

    threads = [threading.Thread(target=work, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for t in range(4):
        for g, w in zip(results[t], ref[t]):
            assert (g is None and w is None) or torch.equal(g, w), t
