"""Fused activation before the cast (mxfp8_quantize_ex with `activation`), on the GPU.

ReLU and squared ReLU are exact in fp32, so FP8 codes and scales must be
bit-exact with the oracle.  GeLU, SiLU and QGeLU involve exp: the kernels
evaluate them in fp32 with the hardware ex2 / rcp approximations, the oracle
exactly in double rounded once to fp32, so where the exact value sits on a
rounding decision the two sides may legitimately decide differently.  The
rule below admits exactly those cases and no others.

The bound.  tests/test_act_accuracy_gpu.py proves, on every finite BF16 input,
that the kernels' fp32 act(x) and act'(x) are within the bounds of
tests/act_bounds.py: DELTA * cond * |exact| + SUB for act, with DELTA = 2^-20,
cond = 1 + |t| sigmoid(-t) the condition factor of the fp32 evaluation and SUB
= 2^-147 for results in fp32's subnormal range; DELTA * terms + SUB for act',
terms = (1 + |t|) |s| (|1 + q| + |q|) for act' = s (1 + q).  The backward
fusion's product dY * act'(X) scales that by |dY| and adds one fp32 rounding;
the oracle's fp32 value is within one rounding of the exact one.  So per
element both sides' values lie within
    w = DELTA cond |v| + SUB + 2^-23 |v| + 2^-149            (forward)
    w = |dY| (DELTA terms + SUB) + 2^-23 |v| + 2^-148        (backward)
of the exact value v, and a rounding decision between them lies within w of v
(all scaled by the block's 2^(127 - e)).

The rule.  A code may differ from the oracle's only if the exact scaled value
lies within w of the midpoint between the two codes.  A scale byte may differ
by one only if the block's exact amax lies within the block's largest w of the
power-of-two boundary between the two exponents.  The exponent rule's other
decision is amax == 0 (e = 127): a scale byte may be 127 on one side and any
value on the other only if every exact value of the block lies within its w of
zero, and the side with 127 then holds only zero codes.  In both cases the
block's codes are checked against the oracle's rounding at the GPU's exponent.  The number of
codes that used the rule may not exceed the number of elements whose exact
scaled value lies within w of a rounding decision, counted from the oracle's
values alone before the comparison (there is no fixed share).  Elements whose
window is wide (w > 2^-12 |v|: near a zero of act', or deep in the sigmoid's
tail) are counted and reported separately.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
from act_bounds import DELTA, SUB, derivative_terms, forward_cond
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

FMAX = {0: 448.0, 1: 57344.0}
ROUND = 2.0 ** -23          # the product's fp32 rounding plus the oracle's
WIDE = 2.0 ** -12           # windows wider than this (relative) are reported


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def act_input(M, N, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N)) * np.exp2(rng.integers(-6, 6, (M, 1)))
    a[0, :32] = -np.abs(a[0, :32]) * 8          # a block that the activations squash to tiny values
    a[1, :64] = 0.0
    a[2, 32:64] = rng.standard_normal(a[2, 32:64].shape) * 1e-39
    a[5, 7] = 60.0
    a[6, :32] = -rng.uniform(96.0, 112.0, a[6, :32].shape)   # SiLU / QGeLU of these are fp32-subnormal
    return wl.to_bf16_bits(a)


def x_values(x_bits):
    return torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()


def forward_window(oracle_mod, x_bits, a):
    """(exact values, absolute windows w) of the forward activation of BF16 x."""
    xv = x_values(x_bits)
    y64 = np.vectorize(lambda v: oracle_mod.activation_f64(v, a))(xv)
    return y64, (DELTA * forward_cond(xv, a) + ROUND) * np.abs(y64) + SUB + 2.0 ** -149


def backward_window(oracle_mod, dy_bits, x_bits, a):
    """(exact values, absolute windows w) of dY * act'(X)."""
    dyv, xv = x_values(dy_bits), x_values(x_bits)
    y64 = dyv * np.vectorize(lambda v: oracle_mod.dactivation_f64(v, a))(xv)
    return y64, np.abs(dyv) * (DELTA * derivative_terms(xv, a) + SUB) + ROUND * np.abs(y64) + 2.0 ** -148


def _decode_table(oracle_mod, fmt):
    return np.array([oracle_mod.fp8_decode(c, fmt) for c in range(128)])


def _scaled(y64, scales, colwise, M, N):
    e = np.repeat(scales, 32, axis=0)[:M] if colwise else np.repeat(scales, 32, axis=1)[:, :N]
    return np.exp2(127.0 - e.astype(np.float64))


def ambiguous_count(oracle_mod, ref_codes, ref_scales, y64, fmt, colwise, wabs):
    """Elements whose exact scaled value lies within its window of a rounding decision (the
    midpoint to a neighbouring code, or zero between +0 and -0), at the oracle's exponents."""
    M, N = ref_codes.shape
    D = _decode_table(oracle_mod, fmt)
    mult = _scaled(y64, ref_scales, colwise, M, N)
    a = np.abs(y64) * mult
    m = (ref_codes & 0x7F).astype(np.int64)
    top = 0x7E if fmt == 0 else 0x7B
    up = np.where(m < top, (D[m] + D[np.minimum(m + 1, 127)]) / 2, np.inf)
    down = np.where(m > 0, (D[m] + D[np.maximum(m - 1, 0)]) / 2, 0.0)
    dist = np.minimum(np.abs(a - up), np.abs(a - down))
    return int(np.count_nonzero(dist <= wabs * mult))


def check_codes(oracle_mod, gpu_codes, ref_codes, gpu_scales, ref_scales, y32, y64, wabs, fmt, colwise):
    """Compare one direction under the boundary rule; returns how many codes needed the rule.

    y32: the oracle's fp32 values [M, N]; y64: the exact (double) values; wabs: the absolute
    windows w [M, N] (None: the activation is exact, bytes must match).
    """
    M, N = y32.shape
    if wabs is None:
        assert np.array_equal(gpu_scales, ref_scales)
        assert np.array_equal(gpu_codes, ref_codes)
        return 0

    def block_of(i, j):   # element indices of the block holding (i, j)
        if colwise:
            r0 = (i // 32) * 32
            return [(r, j) for r in range(r0, min(r0 + 32, M))]
        c0 = (j // 32) * 32
        return [(i, c) for c in range(c0, min(c0 + 32, N))]

    wide = wabs > WIDE * np.abs(y64)
    used, used_wide = 0, 0
    expected = ref_codes.copy()
    # scale bytes that differ: exact amax must sit on the boundary between the two exponents
    for s_idx in np.argwhere(gpu_scales != ref_scales):
        s_idx = tuple(s_idx)
        eg, eo = int(gpu_scales[s_idx]), int(ref_scales[s_idx])
        i, j = (s_idx[0] * 32, s_idx[1]) if colwise else (s_idx[0], s_idx[1] * 32)
        elems = block_of(i, j)
        amax64 = max(abs(float(y64[e])) for e in elems)
        w = max(float(wabs[e]) for e in elems)
        if abs(eg - eo) == 1:
            boundary = FMAX[fmt] * 2.0 ** (min(eg, eo) - 127)
            assert abs(amax64 - boundary) <= w, (s_idx, amax64, boundary, w)
        else:   # amax == 0 on one side: every exact value within its window of zero
            assert 127 in (eg, eo), (s_idx, eg, eo)
            assert all(abs(float(y64[e])) <= float(wabs[e]) for e in elems), (s_idx, eg, eo, amax64)
            zero_side = gpu_codes if eg == 127 else ref_codes
            assert all(int(zero_side[e]) & 0x7F == 0 for e in elems), (s_idx, eg, eo)
        for e in elems:   # this block's codes at the GPU's exponent
            expected[e] = oracle_mod.fp8_encode(float(y32[e]) * 2.0 ** (127 - eg), fmt)
        used += len(elems)
    for e in np.argwhere(gpu_codes != expected):
        e = tuple(e)
        i, j = e
        sc = int(gpu_scales[i // 32, j] if colwise else gpu_scales[i, j // 32])
        mult = 2.0 ** (127 - sc)
        v64 = float(y64[e]) * mult
        dg = oracle_mod.fp8_decode(int(gpu_codes[e]), fmt)
        do = oracle_mod.fp8_decode(int(expected[e]), fmt)
        mid = (dg + do) / 2
        assert abs(v64 - mid) <= float(wabs[e]) * mult, (e, v64, dg, do, float(wabs[e]) * mult)
        used += 1
        used_wide += int(wide[e])
    if used:
        cap = ambiguous_count(oracle_mod, ref_codes, ref_scales, y64, fmt, colwise, wabs)
        cap += 32 * int(np.count_nonzero(gpu_scales != ref_scales))
        assert used <= cap, (used, cap)
    print(f"boundary rule: {used} of {M * N} codes (derived cap "
          f"{ambiguous_count(oracle_mod, ref_codes, ref_scales, y64, fmt, colwise, wabs)}); wide windows: "
          f"{int(np.count_nonzero(wide))} elements, {used_wide} of them needed the rule")
    return used


def forward_case(oracle_mod, x_bits, a):
    """The oracle's fp32 activations, and (exact values, windows) or (None, None) for ReLU / SReLU."""
    y32 = oracle_mod.activate(x_bits, a)
    if a in (1, 2):
        return y32, None, None
    y64, w = forward_window(oracle_mod, x_bits, a)
    return y32, y64, w


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt,shape", [(0, (544, 1056)), (1, (544, 1056)), (0, (97, 40))])
def test_activation_parity(oracle_mod, act, fmt, shape):
    M, N = shape
    x_bits = act_input(M, N, seed=len(act) * 7 + fmt)
    a = mx.binding.ACTIVATIONS[act]
    r = mx.quantize(dev(x_bits), fmt, activation=act, with_amax=True)
    torch.cuda.synchronize()
    o = oracle_mod.quantize_act(x_bits, fmt, a)
    y32, y64, w = forward_case(oracle_mod, x_bits, a)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, y64, w, fmt, False)
    check_codes(oracle_mod, r.out_col.cpu().numpy(), o[2], r.scale_col.cpu().numpy(), o[3], y32, y64, w, fmt, True)
    amax_gpu = float(r.amax.item())
    if a in (1, 2):
        assert amax_gpu == float(np.abs(y32).max())
    else:   # the largest |act| lies within the elements' windows
        assert np.max(np.abs(y64) - w) <= amax_gpu <= np.max(np.abs(y64) + w)


@pytest.mark.parametrize("act", ["relu", "gelu"])
def test_activation_swizzled_single_direction(oracle_mod, act):
    M, N = 256, 160
    x_bits = act_input(M, N, seed=99)
    a = mx.binding.ACTIVATIONS[act]
    r = mx.quantize(dev(x_bits), 0, rowwise=True, colwise=False, activation=act, swizzled=True)
    torch.cuda.synchronize()
    o = oracle_mod.quantize_act(x_bits, 0, a, rowwise=True, colwise=False)
    swz = r.scale_row.cpu().numpy()
    C = o[1].shape[1]
    # the swizzled plane read back into [M, C] through the oracle's layout function
    plain = np.array([[swz[oracle_mod.swizzle_offset(i, c, C)] for c in range(C)] for i in range(M)], np.uint8)
    pad = np.ones(swz.size, bool)
    pad[[oracle_mod.swizzle_offset(i, c, C) for i in range(M) for c in range(C)]] = False
    assert np.all(swz[pad] == 0)
    y32, y64, w = forward_case(oracle_mod, x_bits, a)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], plain, o[1], y32, y64, w, 0, False)


def test_activation_with_dbias_is_rejected():
    x = dev(act_input(64, 64, seed=1))
    with pytest.raises(mx.MXFP8Error):
        mx.quantize(x, 0, with_dbias=True, activation="relu")



# ---- backward fusion: dY * act'(X) ------------------------------------------------

@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt,shape", [(1, (544, 1056)), (0, (45, 80)), (1, (257, 4112)), (0, (70, 24))])
def test_dact_parity_with_dbias(oracle_mod, act, fmt, shape):
    M, N = shape
    a = mx.binding.ACTIVATIONS[act]
    dy_bits = wl.grad_bf16(M, N, seed=M + a)
    x_bits = act_input(M, N, seed=N + a) if M >= 8 else wl.normal_bf16(M, N, seed=a)
    r = mx.quantize_dact(dev(dy_bits), dev(x_bits), fmt, act, with_dbias=True)
    torch.cuda.synchronize()
    y32 = oracle_mod.dactivate(dy_bits, x_bits, a)
    o = oracle_mod.quantize_f32(y32, fmt, with_dbias=True)
    y64, w = (None, None) if a in (1, 2) else backward_window(oracle_mod, dy_bits, x_bits, a)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, y64, w, fmt, False)
    check_codes(oracle_mod, r.out_col.cpu().numpy(), o[2], r.scale_col.cpu().numpy(), o[3], y32, y64, w, fmt, True)
    tol = 1e-5 * np.abs(y32.astype(np.float64)).sum(0) + 1e-30
    assert np.all(np.abs(r.dbias.cpu().numpy().astype(np.float64) - o[4]) <= tol)


# ---- every BF16 value through the forward cast ---------------------------------------

_BITS = np.arange(65536, dtype=np.uint32).astype(np.uint16)
_FINITE = _BITS[(_BITS & 0x7F80) != 0x7F80]
# every finite BF16 value in bit order (ascending positives, then -0 and descending negatives),
# padded with +0 to 2048 runs of 32
RUNS = np.concatenate([_FINITE, np.zeros(65536 - _FINITE.size, np.uint16)]).reshape(2048, 32)


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt", [0, 1])
def test_column_scale_shortcut_on_every_input(act, fmt):
    """Each run of 32 consecutive BF16 values, laid out once as a 32x1 column block and once as a
    1x32 row block: the column pass (whose scale comes from act(max x) when that is large enough)
    must give the same scale and codes as the row pass (which takes max |act(x)| element by element)."""
    x_row = RUNS
    x_col = np.ascontiguousarray(RUNS.T)
    rr = mx.quantize(dev(x_row), fmt, activation=act)
    rc = mx.quantize(dev(x_col), fmt, activation=act)
    torch.cuda.synchronize()
    assert np.array_equal(rc.scale_col.cpu().numpy()[0], rr.scale_row.cpu().numpy()[:, 0])
    assert np.array_equal(rc.out_col.cpu().numpy(), rr.out_row.cpu().numpy().T)


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt", [0, 1])
def test_constant_blocks_give_equal_row_and_column_codes(act, fmt):
    """Every finite BF16 value fills its own 32x32 block: each 1x32 and each 32x1 block is constant,
    so both directions must give the same scale and the same code for it."""
    vals = np.concatenate([_FINITE, np.zeros(255 * 256 - _FINITE.size, np.uint16)]).reshape(255, 256)
    x = np.repeat(np.repeat(vals, 32, axis=0), 32, axis=1)          # [8160, 8192]
    r = mx.quantize(dev(x), fmt, activation=act)
    torch.cuda.synchronize()
    assert torch.equal(r.out_row, r.out_col)
    srow = r.scale_row.cpu().numpy()                                 # [8160, 256]
    scol = r.scale_col.cpu().numpy()                                 # [255, 8192]
    assert np.array_equal(srow[::32], scol[:, ::32])
    assert np.array_equal(srow, np.repeat(srow[::32], 32, axis=0))
    assert np.array_equal(scol, np.repeat(scol[:, ::32], 32, axis=1))


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt", [0, 1])
def test_every_bf16_value_rowwise_against_the_oracle(oracle_mod, act, fmt):
    """The rowwise cast of all finite BF16 values (runs of 32 in bit order) against the oracle.
    Squared ReLU overflows fp32 for |x| >= 2^64; those runs are replaced by zeros here (the oracle's
    exponent search is defined for finite values only)."""
    a = mx.binding.ACTIVATIONS[act]
    x = RUNS.copy()
    if a == 2:
        x[(x & 0x7F80) >= ((127 + 64) << 7)] = 0
    r = mx.quantize(dev(x), fmt, rowwise=True, colwise=False, activation=act)
    torch.cuda.synchronize()
    o = oracle_mod.quantize_act(x, fmt, a, rowwise=True, colwise=False)
    y32, y64, w = forward_case(oracle_mod, x, a)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, y64, w, fmt, False)


# ---- gated activations: act(a) * b for x = [a | b] --------------------------------------

def gated_input(M, N, seed):
    """x = [a | b]: a as for the activations (tails, zeros, subnormals), b N(0,1) with per-row
    exponents, a few zeros and subnormals."""
    a = act_input(M, N, seed) if M >= 8 else wl.normal_bf16(M, N, seed=seed)
    rng = np.random.Generator(np.random.PCG64(seed + 1))
    bv = rng.standard_normal((M, N)) * np.exp2(rng.integers(-8, 8, (M, 1)))
    bv.reshape(-1)[rng.integers(0, M * N, max(1, M * N // 200))] = 0.0
    bv.reshape(-1)[rng.integers(0, M * N, max(1, M * N // 200))] *= 1e-39
    return np.ascontiguousarray(np.concatenate([a, wl.to_bf16_bits(bv)], axis=1))


def gated_window(oracle_mod, x_bits, a):
    """(exact values, absolute windows w) of act(a) * b: the activation's window scaled by |b|,
    plus the product's fp32 rounding on both sides."""
    N = x_bits.shape[1] // 2
    av, bv = x_values(x_bits[:, :N]), x_values(x_bits[:, N:])
    act64 = np.vectorize(lambda v: oracle_mod.activation_f64(v, a))(av)
    y64 = act64 * bv
    w = np.abs(bv) * (DELTA * forward_cond(av, a) * np.abs(act64) + SUB) + ROUND * np.abs(y64) + 2.0 ** -148
    return y64, w


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt,shape", [(0, (544, 1056)), (1, (544, 1056)), (0, (45, 80)), (1, (257, 4112)),
                                       (0, (70, 24)), (1, (1, 8)), (0, (33, 8))])
def test_gated_parity(oracle_mod, act, fmt, shape):
    M, N = shape
    a = mx.binding.ACTIVATIONS[act]
    x_bits = gated_input(M, N, seed=M + 3 * a + fmt)
    r = mx.quantize_gated(dev(x_bits), fmt, act)
    torch.cuda.synchronize()
    y32 = oracle_mod.gate(x_bits, a)
    o = oracle_mod.quantize_f32(y32, fmt)
    y64, w = (None, None) if a in (1, 2) else gated_window(oracle_mod, x_bits, a)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, y64, w, fmt, False)
    check_codes(oracle_mod, r.out_col.cpu().numpy(), o[2], r.scale_col.cpu().numpy(), o[3], y32, y64, w, fmt, True)


@pytest.mark.parametrize("act", ["relu", "silu"])
@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_gated_single_direction(oracle_mod, act, rowwise, colwise):
    a = mx.binding.ACTIVATIONS[act]
    x_bits = gated_input(160, 72, seed=8)
    r = mx.quantize_gated(dev(x_bits), 1, act, rowwise=rowwise, colwise=colwise)
    torch.cuda.synchronize()
    y32 = oracle_mod.gate(x_bits, a)
    o = oracle_mod.quantize_f32(y32, 1, rowwise, colwise)
    y64, w = (None, None) if a == 1 else gated_window(oracle_mod, x_bits, a)
    if rowwise:
        assert r.out_col is None
        check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, y64, w, 1, False)
    else:
        assert r.out_row is None
        check_codes(oracle_mod, r.out_col.cpu().numpy(), o[2], r.scale_col.cpu().numpy(), o[3], y32, y64, w, 1, True)


def test_gated_noop_writes_nothing():
    x = dev(gated_input(96, 64, seed=3))
    u8 = dict(dtype=torch.uint8, device="cuda")
    outs = [torch.full((96, 64), 0x3C, **u8), torch.full((96, 2), 0x3C, **u8),
            torch.full((96, 64), 0x3C, **u8), torch.full((3, 64), 0x3C, **u8)]
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    assert mx.mxfp8_quantize_gated(x, 96, 64, 0, "silu", *outs, one, None) == 0
    torch.cuda.synchronize()
    assert all(bool((t == 0x3C).all()) for t in outs)


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt", [0, 1])
def test_gated_every_bf16_activation_input_rowwise(oracle_mod, act, fmt):
    """Every finite BF16 value as the activation's input a (runs of 32 in bit order), each run
    against a row of random linear inputs b, rowwise against the oracle.  |b| < 1 keeps every
    product finite (the activations of finite inputs are finite, squared ReLU below 2^64)."""
    a_code = mx.binding.ACTIVATIONS[act]
    a = RUNS.copy()
    if a_code == 2:
        a[(a & 0x7F80) >= ((127 + 64) << 7)] = 0
    rng = np.random.Generator(np.random.PCG64(fmt + 10 * a_code))
    mag = rng.uniform(0.5, 1.0, a.shape) * np.exp2(-rng.integers(1, 8, a.shape))
    b = wl.to_bf16_bits(mag * rng.choice([-1.0, 1.0], a.shape))
    x = np.ascontiguousarray(np.concatenate([a, b], axis=1))
    r = mx.quantize_gated(dev(x), fmt, act, rowwise=True, colwise=False)
    torch.cuda.synchronize()
    y32 = oracle_mod.gate(x, a_code)
    o = oracle_mod.quantize_f32(y32, fmt, True, False)
    y64, w = (None, None) if a_code in (1, 2) else gated_window(oracle_mod, x, a_code)
    check_codes(oracle_mod, r.out_row.cpu().numpy(), o[0], r.scale_row.cpu().numpy(), o[1], y32, y64, w, fmt, False)


# ---- gated backward: [g b act'(a) | g act(a)] --------------------------------------------

def dgated_windows(oracle_mod, g_bits, x_bits, a):
    """(exact da, window), (exact db, window): the derivative's and the activation's windows scaled
    by |g b| and |g| (g b is exact in fp32), plus one fp32 rounding on each side."""
    N = g_bits.shape[1]
    gv, av, bv = x_values(g_bits), x_values(x_bits[:, :N]), x_values(x_bits[:, N:])
    dact64 = np.vectorize(lambda v: oracle_mod.dactivation_f64(v, a))(av)
    act64 = np.vectorize(lambda v: oracle_mod.activation_f64(v, a))(av)
    da64, db64 = gv * bv * dact64, gv * act64
    wa = np.abs(gv * bv) * (DELTA * derivative_terms(av, a) + SUB) + ROUND * np.abs(da64) + 2.0 ** -148
    wb = np.abs(gv) * (DELTA * forward_cond(av, a) * np.abs(act64) + SUB) + ROUND * np.abs(db64) + 2.0 ** -148
    return (da64, wa), (db64, wb)


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("fmt,shape", [(1, (544, 1056)), (0, (45, 80)), (1, (257, 1032)), (0, (70, 24)),
                                       (1, (1, 8)), (0, (33, 8))])
def test_dgated_parity(oracle_mod, act, fmt, shape):
    M, N = shape
    a = mx.binding.ACTIVATIONS[act]
    g_bits = wl.grad_bf16(M, N, seed=M + 7 * a)
    x_bits = gated_input(M, N, seed=N + a + fmt)
    r = mx.quantize_dgated(dev(g_bits), dev(x_bits), fmt, act)
    torch.cuda.synchronize()
    da32, db32 = oracle_mod.dgate(g_bits, x_bits, a)
    Cn = -(-N // 32)
    wins = (None, None) if a in (1, 2) else dgated_windows(oracle_mod, g_bits, x_bits, a)
    for h, y32 in enumerate((da32, db32)):
        o = oracle_mod.quantize_f32(y32, fmt)
        y64, w = (None, None) if wins[0] is None else wins[h]
        cs, ss = slice(h * N, (h + 1) * N), slice(h * Cn, (h + 1) * Cn)
        check_codes(oracle_mod, r.out_row.cpu().numpy()[:, cs], o[0], r.scale_row.cpu().numpy()[:, ss], o[1],
                    y32, y64, w, fmt, False)
        check_codes(oracle_mod, r.out_col.cpu().numpy()[:, cs], o[2], r.scale_col.cpu().numpy()[:, cs], o[3],
                    y32, y64, w, fmt, True)


def test_dgated_matches_oracle_layout_and_noop(oracle_mod):
    """ReGLU (exact): the whole [M, 2N] outputs against the oracle's side-by-side layout; noop = 1
    writes nothing."""
    M, N = 96, 72
    g_bits = wl.grad_bf16(M, N, seed=3)
    x_bits = gated_input(M, N, seed=4)
    r = mx.quantize_dgated(dev(g_bits), dev(x_bits), 1, "relu")
    torch.cuda.synchronize()
    for got, want in zip(r[:4], oracle_mod.quantize_dgated(g_bits, x_bits, 1, 1)):
        assert np.array_equal(got.cpu().numpy(), want)
    u8 = dict(dtype=torch.uint8, device="cuda")
    outs = [torch.full((M, 2 * N), 0x3C, **u8), torch.full((M, 6), 0x3C, **u8),
            torch.full((M, 2 * N), 0x3C, **u8), torch.full((3, 2 * N), 0x3C, **u8)]
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    assert mx.mxfp8_quantize_dgated(dev(g_bits), dev(x_bits), M, N, 1, "silu", *outs, one, None) == 0
    torch.cuda.synchronize()
    assert all(bool((t == 0x3C).all()) for t in outs)


# ---- the gated cast over ragged row groups -----------------------------------------------

def run_gated_grouped(x_bits, offsets, fmt, act, prefill=0x3C, noop=None):
    total, N2 = x_bits.shape
    N = N2 // 2
    off = torch.from_numpy(np.asarray(offsets, np.int64)).cuda()
    srows = max(mx.grouped_scale_col_rows(np.maximum.accumulate(np.asarray(offsets, np.int64))), 1)
    u8 = dict(dtype=torch.uint8, device="cuda")
    outs = [torch.full((total, N), prefill, **u8), torch.full((total, -(-N // 32)), prefill, **u8),
            torch.full((total, N), prefill, **u8), torch.full((srows, N), prefill, **u8)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = mx.mxfp8_quantize_gated_grouped(dev(x_bits), total, N, off.numel() - 1, off, fmt, act, *outs, noop, err,
                                         None)
    assert st == 0, mx.mxfp8_status_string(st)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in outs], int(err.item())


GATED_GROUPS = [np.array([64, 0, 32, 416, 96], np.int64),                 # multiples of 32
                np.array([45, 0, 1, 31, 33, 96, 70, 127, 129, 13], np.int64)]   # ragged


@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("fmt,N", [(0, 96), (1, 1032)])
def test_gated_grouped_parity(oracle_mod, act, case, fmt, N):
    a = mx.binding.ACTIVATIONS[act]
    sizes = GATED_GROUPS[case]
    off = wl.offsets_from_sizes(sizes)
    x_bits = gated_input(int(off[-1]), N, seed=N + 5 * a + case)
    got, err = run_gated_grouped(x_bits, off, fmt, act)
    assert err == 0
    want = oracle_mod.quantize_gated_grouped(x_bits, off, fmt, a)
    if a in (1, 2):
        for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got, want):
            assert np.array_equal(g, w), name
        return
    # transcendental: each group under the boundary rule, its own blocks
    y32 = oracle_mod.gate(x_bits, a)
    y64, w = gated_window(oracle_mod, x_bits, a)
    s0 = 0
    for g in range(len(sizes)):
        lo, hi = int(off[g]), int(off[g + 1])
        if lo == hi:
            continue
        o = oracle_mod.quantize_f32(y32[lo:hi], fmt)
        nb = o[3].shape[0]
        check_codes(oracle_mod, got[0][lo:hi], o[0], got[1][lo:hi], o[1], y32[lo:hi], y64[lo:hi], w[lo:hi], fmt,
                    False)
        check_codes(oracle_mod, got[2][lo:hi], o[2], got[3][s0:s0 + nb], o[3], y32[lo:hi], y64[lo:hi], w[lo:hi],
                    fmt, True)
        s0 += nb


def test_gated_grouped_bad_offsets_and_noop():
    x_bits = gated_input(160, 64, seed=2)
    got, err = run_gated_grouped(x_bits, [0, 100, 50, 160], 0, "silu")
    assert err == 1 and all(np.all(t == 0x3C) for t in got)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    got, err = run_gated_grouped(x_bits, [0, 100, 160], 0, "silu", noop=one)
    assert err == 0 and all(np.all(t == 0x3C) for t in got)


def test_gated_and_dgated_empty_shapes():
    """M == 0 or N == 0: nothing to do, status OK, no launch."""
    before = mx.mxfp8_kernel_launch_count()
    assert mx.mxfp8_quantize_gated(None, 0, 64, 0, "silu", None, None, None, None, None, None) == 0
    assert mx.mxfp8_quantize_gated(None, 64, 0, 0, "silu", None, None, None, None, None, None) == 0
    assert mx.mxfp8_quantize_dgated(None, None, 0, 64, 1, "silu", None, None, None, None, None, None) == 0
    assert mx.mxfp8_kernel_launch_count() == before


# ---- the grouped cast with an activation ---------------------------------------------------

@pytest.mark.parametrize("act", ["relu", "srelu", "gelu", "silu", "qgelu"])
@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("fmt,N", [(0, 96), (1, 1032)])
def test_grouped_activated_parity(oracle_mod, act, case, fmt, N):
    a = mx.binding.ACTIVATIONS[act]
    sizes = GATED_GROUPS[case]
    off = wl.offsets_from_sizes(sizes)
    x_bits = act_input(int(off[-1]), N, seed=N + 3 * a + case)
    srows = mx.grouped_scale_col_rows(off)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mx.quantize_grouped(dev(x_bits), torch.from_numpy(off).cuda(), fmt, activation=act, err_flag=err,
                            scale_col_rows=srows)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = [t.cpu().numpy() for t in r[:4]]
    if a in (1, 2):
        for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got,
                              oracle_mod.quantize_grouped_act(x_bits, off, fmt, a)):
            assert np.array_equal(g, w), name
        return
    y32 = oracle_mod.activate(x_bits, a)
    y64, w = forward_window(oracle_mod, x_bits, a)
    s0 = 0
    for g in range(len(sizes)):
        lo, hi = int(off[g]), int(off[g + 1])
        if lo == hi:
            continue
        o = oracle_mod.quantize_f32(y32[lo:hi], fmt)
        nb = o[3].shape[0]
        check_codes(oracle_mod, got[0][lo:hi], o[0], got[1][lo:hi], o[1], y32[lo:hi], y64[lo:hi], w[lo:hi], fmt,
                    False)
        check_codes(oracle_mod, got[2][lo:hi], o[2], got[3][s0:s0 + nb], o[3], y32[lo:hi], y64[lo:hi], w[lo:hi],
                    fmt, True)
        s0 += nb


def test_grouped_activated_rejects_dbias_and_unknown_activation():
    x = dev(act_input(64, 64, seed=1))
    off = torch.tensor([0, 32, 64], dtype=torch.int64, device="cuda")
    with pytest.raises(ValueError):
        mx.quantize_grouped(x, off, 0, activation="gelu", with_dbias=True)
    u8 = dict(dtype=torch.uint8, device="cuda")
    o = [torch.empty((64, 64), **u8), torch.empty((64, 2), **u8), torch.empty((64, 64), **u8),
         torch.empty((2, 64), **u8)]
    assert mx.mxfp8_quantize_grouped_activated(x, 64, 64, 2, off, 0, 9, *o, None, None, None) == 4
    assert mx.mxfp8_quantize_grouped_activated(x, 64, 64, 2, off, 0, 0, *o, None, None, None) == 4


# ---- the grouped cast with per-group GEMM-ready scale planes ---------------------------------

def run_grouped_swizzled(x_bits, offsets, fmt, act, prefill=0x3C, noop=None):
    total, N = x_bits.shape
    off_np = np.asarray(offsets, np.int64)
    off = torch.from_numpy(off_np).cuda()
    u8 = dict(dtype=torch.uint8, device="cuda")
    rb = mx.mxfp8_grouped_swizzled_scale_bytes(np.maximum.accumulate(off_np), N, False)
    cb = mx.mxfp8_grouped_swizzled_scale_bytes(np.maximum.accumulate(off_np), N, True)
    outs = [torch.full((total, N), prefill, **u8), torch.full((max(rb, 1),), prefill, **u8),
            torch.full((total, N), prefill, **u8), torch.full((max(cb, 1),), prefill, **u8)]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = mx.mxfp8_quantize_grouped_swizzled(dev(x_bits), total, N, len(off_np) - 1, off, fmt, act, *outs, noop, err,
                                            None)
    assert st == 0, mx.mxfp8_status_string(st)
    torch.cuda.synchronize()
    got = [t.cpu().numpy() for t in outs]
    got[1], got[3] = got[1][:rb], got[3][:cb]
    return got, int(err.item())


@pytest.mark.parametrize("act", ["none", "relu", "srelu"])
@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("fmt,N", [(0, 96), (1, 1032)])
def test_grouped_swizzled_parity(oracle_mod, act, case, fmt, N):
    a = mx.binding.ACTIVATIONS[act]
    sizes = GATED_GROUPS[case]
    off = wl.offsets_from_sizes(sizes)
    x_bits = act_input(int(off[-1]), N, seed=N + 7 * a + case)
    got, err = run_grouped_swizzled(x_bits, off, fmt, act)
    assert err == 0
    want = oracle_mod.quantize_grouped_swizzled(x_bits, off, fmt, a)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got, want):
        assert g.shape == w.shape and np.array_equal(g, w), name


def _unswizzle(oracle_mod, plane, R, C):
    idx = np.array([[oracle_mod.swizzle_offset(r, c, C) for c in range(C)] for r in range(R)], np.int64)
    return plane[idx]


def test_grouped_swizzled_gelu_codes(oracle_mod):
    """A transcendental activation with per-group GEMM-ready planes: each group's planes read back
    through the oracle's layout function, its codes under the boundary rule."""
    sizes = np.array([45, 0, 83, 130], np.int64)
    off = wl.offsets_from_sizes(sizes)
    N, fmt, a = 72, 0, 3
    x_bits = act_input(int(off[-1]), N, seed=17)
    got, err = run_grouped_swizzled(x_bits, off, fmt, a)
    assert err == 0
    y32 = oracle_mod.activate(x_bits, a)
    y64, w = forward_window(oracle_mod, x_bits, a)
    Cn = -(-N // 32)
    rbase = cbase = 0
    for g in range(len(sizes)):
        lo, hi = int(off[g]), int(off[g + 1])
        if lo == hi:
            continue
        rows = hi - lo
        o = oracle_mod.quantize_f32(y32[lo:hi], fmt)
        rsz = -(-rows // 128) * 128 * (-(-Cn // 4) * 4)
        csz = -(-N // 128) * 128 * (-(-(-(-rows // 32)) // 4) * 4)
        srow = _unswizzle(oracle_mod, got[1][rbase:rbase + rsz], rows, Cn)
        scol = _unswizzle(oracle_mod, got[3][cbase:cbase + csz], N, -(-rows // 32)).T
        check_codes(oracle_mod, got[0][lo:hi], o[0], srow, o[1], y32[lo:hi], y64[lo:hi], w[lo:hi], fmt, False)
        check_codes(oracle_mod, got[2][lo:hi], o[2], np.ascontiguousarray(scol), o[3], y32[lo:hi], y64[lo:hi],
                    w[lo:hi], fmt, True)
        rbase += rsz
        cbase += csz
    assert rbase == got[1].size and cbase == got[3].size


def test_grouped_swizzled_noop_and_bad_offsets():
    x_bits = act_input(160, 64, seed=5)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    got, err = run_grouped_swizzled(x_bits, [0, 100, 160], 0, 0, noop=one)
    assert err == 0 and all(np.all(t == 0x3C) for t in got)
    got, err = run_grouped_swizzled(x_bits, [0, 100, 50, 160], 0, 0)
    assert err == 1 and all(np.all(t == 0x3C) for t in got)


def test_grouped_swizzled_through_the_binding(oracle_mod):
    off = wl.offsets_from_sizes(np.array([45, 0, 83, 130], np.int64))
    x_bits = act_input(int(off[-1]), 96, seed=29)
    t = mx.quantize_grouped(dev(x_bits), torch.from_numpy(off).cuda(), fmt=1, activation="relu", swizzled=True)
    want = oracle_mod.quantize_grouped_swizzled(x_bits, off, 1, 1)
    got = [t.out_row, t.scale_row, t.out_col, t.scale_col]
    for g, w in zip(got, want):
        assert np.array_equal(g.cpu().numpy(), w)
