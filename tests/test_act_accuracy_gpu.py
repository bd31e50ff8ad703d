"""The kernels' fp32 activations, checked on every finite BF16 input.

The cast with an activation (and the backward fusion) computes act(x) (act'(x))
in fp32 with the hardware ex2 / rcp approximations; the oracle evaluates the
same functions exactly in double.  Since the kernels' value is a function of
the 16-bit input alone, the C ABI's diagnostic entry point
mxfp8_activation_values (the kernels' own device routines) is run on all 65280
finite BF16 values, and each is compared with the oracle's exact value:

  - ReLU, squared ReLU and their derivatives: bit-exact with the oracle's fp32.
  - GeLU, SiLU, QGeLU and their derivatives: within the bounds of
    tests/act_bounds.py (DELTA = 2^-20 times the condition factor of the fp32
    evaluation: 1 + |t| sigmoid(-t) for act, (1 + |t|) |s| (|1 + q| + |q|) for
    act' = s (1 + q)), plus SUB in fp32's subnormal range.

These bounds are what the parity tests of the activated casts use as the
windows within which a code may differ from the oracle's, so this test is what
makes those windows sound.

The same run checks the two properties the forward cast's column-scale shortcut
relies on (its scale of a 32x1 block is act(max x) when that is at least a bound
no negative input can reach): act is non-decreasing over the positive BF16
values in order, and |act(x)| stays below that bound for every negative x.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from act_bounds import DELTA, SUB, derivative_terms, forward_cond

pytestmark = pytest.mark.gpu

NEGATIVE_SIDE_BOUND = 0.2785 * 1.01   # the shortcut's bound for GeLU, SiLU, QGeLU

BITS = np.arange(65536, dtype=np.uint32).astype(np.uint16)
FINITE = BITS[(BITS & 0x7F80) != 0x7F80]


def bf16_values(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


def gpu_values(act, derivative):
    x = torch.from_numpy(FINITE.view(np.int16)).cuda()
    out = torch.full((FINITE.size,), float("nan"), dtype=torch.float32, device="cuda")
    st = mx.mxfp8_activation_values(x, FINITE.size, act, derivative, out)
    assert st == 0, mx.mxfp8_status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("act", ["relu", "srelu"])
@pytest.mark.parametrize("derivative", [0, 1])
def test_relu_family_bit_exact_on_every_input(oracle_mod, act, derivative):
    a = mx.binding.ACTIVATIONS[act]
    got = gpu_values(a, derivative)
    if derivative:
        ones = np.full(FINITE.shape, 0x3F80, np.uint16)          # dY = 1.0: the product is act'(x)
        want = oracle_mod.dactivate(ones, FINITE, a)
    else:
        want = oracle_mod.activate(FINITE, a)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("act", ["gelu", "silu", "qgelu"])
def test_forward_activation_error_bound_on_every_input(oracle_mod, act):
    a = mx.binding.ACTIVATIONS[act]
    got = gpu_values(a, 0).astype(np.float64)
    xv = bf16_values(FINITE)
    exact = np.array([oracle_mod.activation_f64(v, a) for v in xv])
    err = np.abs(got - exact)
    bound = DELTA * forward_cond(xv, a) * np.abs(exact) + SUB
    bad = np.flatnonzero(~(err <= bound))          # NaN counts as beyond the bound
    ratio = err / bound
    assert bad.size == 0, (f"{bad.size} inputs beyond the bound; worst error / bound {ratio.max():.3f} at "
                           f"x = {xv[np.argmax(ratio)]!r}")
    normal = np.abs(exact) > 2.0 ** -126
    rel = err[normal] / np.abs(exact[normal])
    print(f"{act}: largest error / bound {ratio.max():.3f}; largest relative error 2^{np.log2(rel.max()):.2f} "
          f"(x = {xv[normal][np.argmax(rel)]!r})")


@pytest.mark.parametrize("act", ["gelu", "silu", "qgelu"])
def test_derivative_error_bound_on_every_input(oracle_mod, act):
    a = mx.binding.ACTIVATIONS[act]
    got = gpu_values(a, 1).astype(np.float64)
    xv = bf16_values(FINITE)
    exact = np.array([oracle_mod.dactivation_f64(v, a) for v in xv])
    bound = DELTA * derivative_terms(xv, a) + SUB
    err = np.abs(got - exact)
    bad = np.flatnonzero(~(err <= bound))          # NaN counts as beyond the bound
    ratio = err / bound
    assert bad.size == 0, (f"{bad.size} inputs beyond the bound; worst error / bound {ratio.max():.3f} at "
                           f"x = {xv[np.argmax(ratio)]!r}: gpu {got[np.argmax(ratio)]!r}, exact {exact[np.argmax(ratio)]!r}")
    normal = np.abs(exact) > 2.0 ** -126
    print(f"d{act}: largest error / bound {ratio.max():.3f}; largest bound / |exact| over normal results "
          f"2^{np.log2(np.max(bound[normal] / np.abs(exact[normal]))):.2f}")


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
def test_forward_activation_shortcut_properties(act):
    """Non-decreasing over positive inputs in order; below the shortcut's bound on negative inputs."""
    a = mx.binding.ACTIVATIONS[act]
    got = gpu_values(a, 0)
    pos = (FINITE > 0) & (FINITE < 0x8000)             # positive finite values, ascending with the bits
    order = np.argsort(FINITE[pos].astype(np.int64))
    vals = got[pos][order].astype(np.float64)          # squared ReLU reaches +inf: compare, don't subtract
    assert np.all(vals[1:] >= vals[:-1])
    neg = FINITE >= 0x8000                              # -0 and the negative values
    worst = float(np.max(np.abs(got[neg])))
    if a in (1, 2):
        assert worst == 0.0
    else:
        assert worst < NEGATIVE_SIDE_BOUND, worst
