"""mxfp8_quantize_dbias_noalloc: dbias quantize for callers that cannot allocate.

Some callers have no way to allocate device memory (a plugin or callback that
is handed only its input and output tensors, or code that must not allocate
once it is running), so they cannot supply the dbias workspace.  This entry
point keeps that workspace in a static 8 MiB device array inside the library.
The test calls it through the C ABI twice in a row, on different inputs and
shapes, and checks that every output matches the regular entry point given an
explicit workspace: FP8 and scale bytes identical, dbias within
1e-5 * sum|x| per column (the same tolerance as the other dbias tests).  Two
calls in a row are also held to the CPU oracle directly.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
import oracle_slices
from mxfp8_block_scaled_04_gb300 import binding
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def outputs(M, N):
    u8 = dict(dtype=torch.uint8, device="cuda")
    return [torch.full((M, N), 0x11, **u8), torch.full((M, N // 32), 0x11, **u8),
            torch.full((M, N), 0x11, **u8), torch.full((M // 32, N), 0x11, **u8),
            torch.full((N,), 7.0, dtype=torch.float32, device="cuda")]


def _compare_one_call(fmt, M, N, seed, call):
    x_bits = wl.grad_bf16(M, N, seed=seed)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    ref = outputs(M, N)
    ws = torch.empty(mx.mxfp8_quantize_workspace_bytes(M, N, True), dtype=torch.uint8, device="cuda")
    assert mx.mxfp8_quantize(x, M, N, fmt, *ref[:4], ref[4], ws, None, None) == 0
    got = outputs(M, N)
    assert binding.mxfp8_quantize_dbias_noalloc(x, M, N, fmt, *got[:4], got[4], None, None) == 0
    torch.cuda.synchronize()
    for name, a, b in zip(("out_row", "scale_row", "out_col", "scale_col"), ref[:4], got[:4]):
        assert torch.equal(a, b), f"call {call}: {name} differs"
    tol = 1e-5 * torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().abs().sum(0)
    diff = (ref[4].double().cpu() - got[4].double().cpu()).abs()
    assert bool((diff <= tol).all()), f"call {call}: dbias differs"


@pytest.mark.parametrize("fmt", [mx.E5M2, mx.E4M3])
def test_noalloc_larger_then_smaller_call_same_columns(fmt):
    """A smaller call after a larger one with the same N: the array still holds the larger call's
    partial sums past the smaller call's row tiles, which the smaller call must neither need nor read."""
    for call, M in enumerate([4096, 1056]):
        _compare_one_call(fmt, M, 1024, seed=200 + call, call=call)


def test_noalloc_at_the_scratch_limit():
    """16384 x 16384 needs exactly 128 * 16384 * 4 bytes = 8 MiB of workspace: the largest accepted size."""
    M, N = 16384, 16384
    assert mx.mxfp8_quantize_workspace_bytes(M, N, True) == mx.binding.NOALLOC_SCRATCH_BYTES
    _compare_one_call(mx.E5M2, M, N, seed=300, call=0)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("fmt", [mx.E5M2, mx.E4M3])
def test_noalloc_matches_workspace_entry_point_two_calls(fmt):
    for call, (M, N) in enumerate([(1056, 288), (4096, 1024)]):
        x_bits = wl.grad_bf16(M, N, seed=100 + call)
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
        ref = outputs(M, N)
        ws = torch.empty(mx.mxfp8_quantize_workspace_bytes(M, N, True), dtype=torch.uint8, device="cuda")
        assert mx.mxfp8_quantize(x, M, N, fmt, *ref[:4], ref[4], ws, None, None) == 0
        got = outputs(M, N)
        assert binding.mxfp8_quantize_dbias_noalloc(x, M, N, fmt, *got[:4], got[4], None, None) == 0
        torch.cuda.synchronize()
        for name, a, b in zip(("out_row", "scale_row", "out_col", "scale_col"), ref[:4], got[:4]):
            assert torch.equal(a, b), f"call {call}: {name} differs"
        tol = 1e-5 * torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().abs().sum(0)
        diff = (ref[4].double().cpu() - got[4].double().cpu()).abs()
        assert bool((diff <= tol).all()), f"call {call}: dbias differs"


def test_noalloc_matches_oracle_two_calls(oracle_mod):
    for call, (M, N, fmt) in enumerate([(2080, 4096, mx.E5M2), (1000, 1032, mx.E4M3)]):
        x_bits = wl.grad_bf16(M, N, seed=400 + call)
        x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
        u8 = dict(dtype=torch.uint8, device="cuda")
        got = [torch.full((M, N), 0x11, **u8), torch.full((M, -(-N // 32)), 0x11, **u8),
               torch.full((M, N), 0x11, **u8), torch.full((-(-M // 32), N), 0x11, **u8),
               torch.full((N,), 7.0, dtype=torch.float32, device="cuda")]
        assert binding.mxfp8_quantize_dbias_noalloc(x, M, N, fmt, *got[:4], got[4], None, None) == 0
        torch.cuda.synchronize()
        want = oracle_slices.quantize(oracle_mod, x_bits, fmt, with_dbias=True)
        for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got[:4], want[:4]):
            assert np.array_equal(g.cpu().numpy(), w), f"call {call}: {name} differs from the oracle"
        tol = 1e-5 * np.abs(torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().numpy()).sum(0)
        assert bool((np.abs(got[4].double().cpu().numpy() - want[4]) <= tol).all()), f"call {call}: dbias"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 32768 x 16384 needs 256 * 16384 * 4 = 16 MiB of workspace > 8 MiB; rejected
    # on the host before any pointer is touched.
    A = 1 << 20
    st = binding.mxfp8_quantize_dbias_noalloc(A, 32768, 16384, mx.E4M3, A, A, A, A, A, None, None)
    assert st == 2      # MXFP8_ERR_SHAPE
    assert binding.mxfp8_quantize_dbias_noalloc(A, 64, 64, mx.E4M3, A, A, A, A, None, None, None) == 1


def test_noalloc_noop_writes_nothing():
    """*noop == 1.0f: neither kernel of the call writes (outputs and dbias keep their prefill)."""
    M, N = 128, 256
    x_bits = wl.grad_bf16(M, N, seed=5)
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda()
    o = outputs(M, N)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    zero = torch.zeros(1, dtype=torch.float32, device="cuda")
    assert mx.mxfp8_quantize_dbias_noalloc(x, M, N, mx.E5M2, *o[:4], o[4], one, None) == 0
    torch.cuda.synchronize()
    assert all(bool((t == 0x11).all()) for t in o[:4]) and bool((o[4] == 7.0).all())
    assert mx.mxfp8_quantize_dbias_noalloc(x, M, N, mx.E5M2, *o[:4], o[4], zero, None) == 0
    torch.cuda.synchronize()
    assert not all(bool((t == 0x11).all()) for t in o[:4]) and not bool((o[4] == 7.0).all())


def test_noalloc_inside_a_captured_graph(oracle_mod):
    """A first call outside capture, then the call captured and replayed on new input: the
    replayed launches use the static workspace and the live buffers."""
    M, N = 1056, 512
    x = torch.from_numpy(wl.grad_bf16(M, N, seed=600).view(np.int16)).view(torch.bfloat16).cuda()
    o = outputs(M, N)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert binding.mxfp8_quantize_dbias_noalloc(x, M, N, mx.E5M2, *o[:4], o[4], None, s) == 0
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        st = binding.mxfp8_quantize_dbias_noalloc(x, M, N, mx.E5M2, *o[:4], o[4], None, s)
    assert st == 0
    new = wl.grad_bf16(M, N, seed=601)
    x.copy_(torch.from_numpy(new.view(np.int16)).view(torch.bfloat16).cuda())
    graph.replay()
    torch.cuda.synchronize()
    want = oracle_slices.quantize(oracle_mod, new, mx.E5M2, with_dbias=True)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), o[:4], want[:4]):
        assert np.array_equal(g.cpu().numpy(), w), name
    tol = 1e-5 * np.abs(torch.from_numpy(new.view(np.int16)).view(torch.bfloat16).double().numpy()).sum(0)
    assert bool((np.abs(o[4].double().cpu().numpy() - want[4]) <= tol).all())
