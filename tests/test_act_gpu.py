"""Fused activation before the cast (mxfp8_quantize_ex with `activation`), on the GPU.

ReLU and squared ReLU are exact in fp32, so FP8 codes and scales must be
bit-exact with the oracle.  GeLU, SiLU and QGeLU involve exp: the kernel's
fp32 value and the oracle's (the double value rounded once to fp32) can differ
by a few fp32 ulps, so where the exact value sits on a decision boundary the
two sides may legitimately decide differently.  A code may differ from the
oracle's only if the exact (double) scaled value lies within 2^-20 (relative)
of the midpoint between the two codes, or the fp32 value is subnormal (fewer
significant bits on both sides); a scale byte may differ by one only if the
block's exact amax lies within 2^-20 of the power-of-two boundary between the
two exponents, and then the block's codes are checked against the oracle's
rounding at the GPU's exponent.  At most 1e-4 of the codes may use the rule.

The derivatives are computed as s (1 + q) (q = x (1 - s) t' for dGeLU, x (1 - s) for dSiLU,
1.702 x (1 - s) for dQGeLU), and 1 + q cancels where act'(x) crosses zero: there an fp32
evaluation's relative error grows by the condition number kappa = 1 + |q| / |1 + q|, so the
backward fusion's checks allow kappa * 2^-20 for that element, and at most 3e-4 of its codes may
use the rule (a seeded 257x4112 dQGeLU case needed it for 1.09e-4).
"""
import math

import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FMAX = {0: 448.0, 1: 57344.0}
TOL = 2.0 ** -20


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def act_input(M, N, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N)) * np.exp2(rng.integers(-6, 6, (M, 1)))
    a[0, :32] = -np.abs(a[0, :32]) * 8          # a block that the activations squash to tiny values
    a[1, :64] = 0.0
    a[2, 32:64] = rng.standard_normal(32) * 1e-39
    a[5, 7] = 60.0
    return wl.to_bf16_bits(a)


def x_values(x_bits):
    return torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def check_codes(oracle_mod, gpu_codes, ref_codes, gpu_scales, ref_scales, y32, value64, exact, fmt, colwise,
                kappa=None):
    """Compare one direction; returns how many codes needed the boundary rule.

    y32: the oracle's fp32 values; value64(i, j): the exact (double) value of element (i, j);
    kappa: per-element condition numbers [M, N] widening the rule for codes (None: 1).
    """
    M, N = y32.shape
    if exact:
        assert np.array_equal(gpu_scales, ref_scales)
        assert np.array_equal(gpu_codes, ref_codes)
        return 0

    def block_of(i, j):   # element indices of the block holding (i, j)
        if colwise:
            r0 = (i // 32) * 32
            return [(r, j) for r in range(r0, min(r0 + 32, M))]
        c0 = (j // 32) * 32
        return [(i, c) for c in range(c0, min(c0 + 32, N))]

    used = 0
    expected = ref_codes.copy()
    # scale bytes that differ: exact amax must sit on the boundary between the two exponents
    for s_idx in np.argwhere(gpu_scales != ref_scales):
        s_idx = tuple(s_idx)
        eg, eo = int(gpu_scales[s_idx]), int(ref_scales[s_idx])
        assert abs(eg - eo) == 1, (s_idx, eg, eo)
        i, j = (s_idx[0] * 32, s_idx[1]) if colwise else (s_idx[0], s_idx[1] * 32)
        elems = block_of(i, j)
        amax64 = max(abs(value64(*e)) for e in elems)
        boundary = FMAX[fmt] * 2.0 ** (min(eg, eo) - 127)
        assert abs(amax64 - boundary) <= TOL * boundary, (s_idx, amax64, boundary)
        for e in elems:   # this block's codes at the GPU's exponent
            expected[e] = oracle_mod.fp8_encode(float(y32[e]) * 2.0 ** (127 - eg), fmt)
        used += len(elems)
    for e in np.argwhere(gpu_codes != expected):
        e = tuple(e)
        i, j = e
        sc = int(gpu_scales[i // 32, j] if colwise else gpu_scales[i, j // 32])
        v64 = value64(i, j) * 2.0 ** (127 - sc)
        dg = oracle_mod.fp8_decode(int(gpu_codes[e]), fmt)
        do = oracle_mod.fp8_decode(int(expected[e]), fmt)
        mid = (dg + do) / 2
        subnormal_y = abs(float(y32[e])) < 2.0 ** -126
        tol = TOL * (1.0 if kappa is None else float(kappa[e]))
        assert subnormal_y or abs(v64 - mid) <= tol * max(abs(v64), 2.0 ** -20), (e, v64, dg, do, tol)
        used += 1
    # the share of codes inside their window grows with the windows' width: kappa >= 1 widens them
    cap = 1e-4 if kappa is None else 3e-4
    assert used <= max(cap * M * N, 64), used
    return used


def dact_kappa(xv, a):
    """Condition number of 1 + q in the derivative's factored form (1 where it has none)."""
    if a in (1, 2):
        return None
    t = {3: 1.5957691216057308 * (xv + 0.044715 * xv ** 3), 4: xv, 5: 1.702 * xv}[a]
    with np.errstate(over="ignore"):
        oms = 1.0 / (1.0 + np.exp(t))                     # 1 - sigmoid(t)
    q = {3: xv * oms * 1.5957691216057308 * (1.0 + 3 * 0.044715 * xv ** 2), 4: xv * oms, 5: 1.702 * xv * oms}[a]
    with np.errstate(divide="ignore"):
        return 1.0 + np.abs(q) / np.maximum(np.abs(1.0 + q), 1e-300)


def act_checker(oracle_mod, x_bits, a):
    xv = x_values(x_bits)
    return oracle_mod.activate(x_bits, a), (lambda i, j: oracle_mod.activation_f64(xv[i, j], a))


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt", [0, 1])
def test_activation_parity(oracle_mod, act, fmt):
    M, N = 544, 1056
    x_bits = act_input(M, N, seed=len(act) * 7 + fmt)
    a = mx.binding.ACTIVATIONS[act]
    r = mx.quantize(dev(x_bits), fmt, activation=act, with_amax=True)
    torch.cuda.synchronize()
    o = oracle_mod.quantize_act(x_bits, fmt, a)
    y32, v64 = act_checker(oracle_mod, x_bits, a)
    exact = a in (1, 2)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, v64, exact, fmt, False)
    check_codes(oracle_mod, r.out_col.cpu().numpy(), o[2], r.scale_col.cpu().numpy(), o[3], y32, v64, exact, fmt, True)
    amax_ref = float(np.abs(oracle_mod.activate(x_bits, a)).max())
    if a in (1, 2):
        assert float(r.amax.item()) == amax_ref
    else:
        assert math.isclose(float(r.amax.item()), amax_ref, rel_tol=2 ** -20)


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_activation_swizzled_single_direction(oracle_mod, act):
    M, N = 256, 160
    x_bits = act_input(M, N, seed=99)
    a = mx.binding.ACTIVATIONS[act]
    r = mx.quantize(dev(x_bits), 0, rowwise=True, colwise=False, activation=act, swizzled=True)
    torch.cuda.synchronize()
    o = oracle_mod.quantize_act(x_bits, 0, a, rowwise=True, colwise=False)
    plain = r.scale_row.cpu().numpy()
    # unswizzle through the oracle's layout to compare with the plain scales
    want_swz = oracle_mod.swizzle_scales(o[1])
    if a == 1:
        assert np.array_equal(plain, want_swz) and np.array_equal(r.out_row.cpu().numpy(), o[0])
    else:
        assert np.mean(plain == want_swz) > 0.999
        assert np.mean(r.out_row.cpu().numpy() == o[0]) > 0.999


def test_activation_with_dbias_is_rejected():
    x = dev(act_input(64, 64, seed=1))
    with pytest.raises(mx.MXFP8Error):
        mx.quantize(x, 0, with_dbias=True, activation="relu")



# ---- backward fusion: dY * act'(X) ------------------------------------------------

@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt,shape", [(1, (544, 1056)), (0, (45, 80)), (1, (257, 4112))])
def test_dact_parity_with_dbias(oracle_mod, act, fmt, shape):
    M, N = shape
    a = mx.binding.ACTIVATIONS[act]
    dy_bits = wl.grad_bf16(M, N, seed=M + a)
    x_bits = act_input(M, N, seed=N + a) if M >= 8 else wl.normal_bf16(M, N, seed=a)
    r = mx.quantize_dact(dev(dy_bits), dev(x_bits), fmt, act, with_dbias=True)
    torch.cuda.synchronize()
    y32 = oracle_mod.dactivate(dy_bits, x_bits, a)
    o = oracle_mod.quantize_f32(y32, fmt, with_dbias=True)
    dyv, xv = x_values(dy_bits), x_values(x_bits)
    v64 = lambda i, j: dyv[i, j] * oracle_mod.dactivation_f64(xv[i, j], a)
    exact = a in (1, 2)
    kap = dact_kappa(xv, a)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, v64, exact, fmt, False,
                kap)
    check_codes(oracle_mod, r.out_col.cpu().numpy(), o[2], r.scale_col.cpu().numpy(), o[3], y32, v64, exact, fmt, True,
                kap)
    tol = 1e-5 * np.abs(y32.astype(np.float64)).sum(0) + 1e-30
    assert np.all(np.abs(r.dbias.cpu().numpy().astype(np.float64) - o[4]) <= tol)
