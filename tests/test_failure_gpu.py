"""Failure detection without a GPU fault.

Every pipeline kernel waits on its tile copies with a bounded wait; on expiry a CTA records bit 0
of the library's fault word, drains its own copies and returns.  A copy that never lands cannot be
produced without a fault, so the diagnostic entry point runs the same bounded wait on an mbarrier
phase that nothing completes (a flag that nothing sets): the wait must expire after its limit, the
host must read the expiry, and the context must stay usable for ordinary calls.
"""
import time

import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bounded_wait_expires_is_reported_and_the_context_stays_usable(oracle_mod):
    mx.mxfp8_device_fault_word(clear=True)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert mx.mxfp8_selftest_bounded_wait(50_000_000, flag) == 0   # 50 ms
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert int(flag.item()) == 1
    assert 0.045 <= elapsed < 5.0, elapsed
    assert mx.mxfp8_device_fault_word(clear=True) & 1
    assert mx.mxfp8_device_fault_word() == 0
    # an ordinary call afterwards: bit-exact, and no fault recorded
    x_bits = wl.normal_bf16(96, 160, seed=1)
    r = mx.quantize(torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).cuda(), mx.E4M3)
    torch.cuda.synchronize()
    o = oracle_mod.quantize(x_bits, mx.E4M3)
    for g, w in zip(r[:4], o[:4]):
        assert np.array_equal(g.cpu().numpy(), w)
    assert mx.mxfp8_device_fault_word() == 0
