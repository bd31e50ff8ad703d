"""Pins for the CPU oracle, against things other than the oracle itself.

* FP8 decode of all 256 codes against torch's float8 dtypes (a library routine).
* FP8 encode against torch's float32 -> float8 cast on in-range values, plus
  brute-force properties: round-trip of every finite code, ties-to-even at every
  midpoint, monotonicity, saturation.
* The block exponent against its defining inequality and against an integer
  closed form on the BF16 bits, for every finite positive BF16 value.
* Hand-worked blocks (tests/golden/hand_blocks.txt).
* Whole-matrix quantize against a brute-force nearest-code search on small
  matrices with M != N (catches a transposed operand or a wrong index).
* The round-trip error bound, the dbias column sum against math.fsum, and the
  grouped == flat invariant.
"""
import math
import os
import re

import numpy as np
import pytest
import torch

from mxfp8_block_scaled_04_gb300 import workloads as wl

E4M3, E5M2 = 0, 1
FMAX = {E4M3: 448.0, E5M2: 57344.0}
MBITS = {E4M3: 3, E5M2: 2}
EMIN = {E4M3: -6, E5M2: -14}
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_blocks.txt")


def torch_decode_table(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()


def is_finite_code(b, fmt):
    return math.isfinite(torch_decode_table(fmt)[b])


# ---- FP8 codec ----------------------------------------------------------------

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_every_code_matches_torch(oracle_mod, fmt):
    table = torch_decode_table(fmt)
    for b in range(256):
        got = oracle_mod.fp8_decode(b, fmt)
        want = table[b]
        if math.isnan(want):
            assert math.isnan(got), (fmt, b)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want), (fmt, b, got, want)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_roundtrips_every_finite_code(oracle_mod, fmt):
    table = torch_decode_table(fmt)
    for b in range(256):
        if math.isfinite(table[b]):
            assert oracle_mod.fp8_encode(table[b], fmt) == b, (fmt, b)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_midpoints_tie_to_even(oracle_mod, fmt):
    table = torch_decode_table(fmt)
    for sign in (0x00, 0x80):
        for c in range(0, 127):
            lo, hi = sign | c, sign | (c + 1)
            if not (math.isfinite(table[lo]) and math.isfinite(table[hi])):
                continue
            mid = (table[lo] + table[hi]) / 2
            even = lo if (c % 2 == 0) else hi   # codes differ only in the mantissa LSB chain
            assert oracle_mod.fp8_encode(mid, fmt) == even, (fmt, hex(lo), hex(hi))
            toward_hi = math.nextafter(mid, math.copysign(math.inf, mid))
            toward_lo = math.nextafter(mid, 0.0)
            assert oracle_mod.fp8_encode(toward_hi, fmt) == hi
            assert oracle_mod.fp8_encode(toward_lo, fmt) == lo


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_on_random_inrange(oracle_mod, fmt):
    rng = np.random.Generator(np.random.PCG64(123 + fmt))
    n = 40000
    mag = np.exp2(rng.uniform(math.log2(FMAX[fmt]) - 30, math.log2(FMAX[fmt]), n))
    v = (rng.choice([-1.0, 1.0], n) * mag).astype(np.float32)
    want = torch.from_numpy(v).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    got = np.array([oracle_mod.fp8_encode(float(t), fmt) for t in v], dtype=np.uint8)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_saturates_and_is_monotone(oracle_mod, fmt):
    top = 0x7E if fmt == E4M3 else 0x7B
    for v in (FMAX[fmt] * 1.0001, FMAX[fmt] * 1.07, 1e30, math.inf):
        assert oracle_mod.fp8_encode(v, fmt) == top
        assert oracle_mod.fp8_encode(-v, fmt) == top | 0x80
    rng = np.random.Generator(np.random.PCG64(7))
    v = np.sort(np.exp2(rng.uniform(-30, 20, 3000)))
    table = torch_decode_table(fmt)
    dec = [table[oracle_mod.fp8_encode(t, fmt)] for t in v]
    assert all(a <= b for a, b in zip(dec, dec[1:]))


# ---- block exponent ---------------------------------------------------------------

def all_positive_finite_bf16():
    bits = np.arange(1, 0x7F80, dtype=np.uint16)    # 0x0001 .. 0x7F7F
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return bits, vals


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block_exponent_defining_inequality(oracle_mod, fmt):
    bits, vals = all_positive_finite_bf16()
    fmax = FMAX[fmt]
    for a in vals:
        e = oracle_mod.block_exponent(a, fmt)
        assert 0 <= e <= 254
        k = e - 127
        assert a <= fmax * 2.0 ** k, (a, e)            # scaled amax never exceeds Fmax
        if e > 0:
            assert a > fmax * 2.0 ** (k - 1), (a, e)   # and k is the smallest such integer


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block_exponent_integer_form_on_bf16_bits(oracle_mod, fmt):
    # For a normal BF16 a = (1 + m/128) 2^(E-127): a <= 1.75 2^(emax+k) iff
    # k >= E-127-emax + [m/128 > 0.75]; a subnormal amax always clamps to 0.
    emax = 8 if fmt == E4M3 else 15
    bits, vals = all_positive_finite_bf16()
    for b, a in zip(bits.tolist(), vals):
        E, m = b >> 7, b & 0x7F
        want = max(0, E - emax + (1 if m > 0x60 else 0)) if E > 0 else 0
        assert oracle_mod.block_exponent(a, fmt) == want, (hex(b), a)
    assert oracle_mod.block_exponent(0.0, fmt) == 127


def test_e8m0_decode(oracle_mod):
    assert oracle_mod.e8m0_decode(127) == 1.0
    assert oracle_mod.e8m0_decode(0) == 2.0 ** -127
    assert oracle_mod.e8m0_decode(254) == 2.0 ** 127
    assert math.isnan(oracle_mod.e8m0_decode(255))


# ---- hand-worked blocks ---------------------------------------------------------

def parse_value(tok):
    """'1.0', '-0.0', '2**-130', '3*2**-133', '-2**-10' -> float."""
    m = re.fullmatch(r"(-?)(?:(\d+)\*)?2\*\*(-?\d+)", tok)
    if m:
        v = float(m.group(2) or 1) * 2.0 ** int(m.group(3))
        return -v if m.group(1) else v
    return float(tok)


def parse_golden():
    cases = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fmt_s, elems_s, e_s, bytes_s = [p.strip() for p in line.split("|")]
            elems, out = [], []
            for tok in elems_s.split(","):
                tok = tok.strip()
                if "**" in tok:
                    elems.append(parse_value(tok))
                else:
                    v, _, n = tok.partition("*")
                    elems += [parse_value(v)] * (int(n) if n else 1)
            for tok in bytes_s.split(","):
                h, _, n = tok.strip().partition("*")
                out += [int(h, 16)] * (int(n) if n else 1)
            assert len(elems) == 32 and len(out) == 32, line
            cases.append((E4M3 if fmt_s == "E4M3" else E5M2, elems, int(e_s), out))
    return cases


GOLDEN_CASES = parse_golden()


@pytest.mark.parametrize("case", range(len(GOLDEN_CASES)))
def test_hand_worked_blocks(oracle_mod, case):
    fmt, elems, e, want = GOLDEN_CASES[case]
    bits = wl.to_bf16_bits(np.array(elems, np.float64).reshape(1, 32))
    back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(back.ravel(), np.array(elems)), "fixture value is not an exact BF16"
    # Rowwise: the block is one row.  Colwise: the same block as one column.
    out_row, scale_row, _, _, _ = oracle_mod.quantize(np.tile(bits, (32, 1)), fmt)
    assert scale_row[0, 0] == e
    assert out_row[0].tolist() == want
    _, _, out_col, scale_col, _ = oracle_mod.quantize(np.tile(bits.reshape(32, 1), (1, 32)), fmt)
    assert scale_col[0, 0] == e
    assert out_col[:, 0].tolist() == want


# ---- whole matrices against a brute-force nearest-code search -------------------

def brute_force(x_bits, fmt):
    """Rowwise/colwise quantize by exhaustive search; independent of the oracle's code."""
    x = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    table = torch_decode_table(fmt)
    finite = np.array([b for b in range(256) if math.isfinite(table[b])])
    tv = table[finite]
    fmax = FMAX[fmt]

    def scale_of(amax):
        if amax == 0:
            return 127
        k = next(k for k in range(-300, 300) if amax <= fmax * 2.0 ** k)
        return min(max(k + 127, 0), 254)

    def encode(v):
        d = np.abs(tv - v)
        cand = finite[d == d.min()]
        same_sign = [b for b in cand if (b >> 7) == (1 if math.copysign(1, v) < 0 else 0)]
        cand = same_sign or list(cand)
        even = [b for b in cand if b % 2 == 0]
        return (even or cand)[0]

    M, N = x.shape
    out_row = np.zeros((M, N), np.uint8)
    scale_row = np.zeros((M, -(-N // 32)), np.uint8)
    out_col = np.zeros((M, N), np.uint8)
    scale_col = np.zeros((-(-M // 32), N), np.uint8)
    for i in range(M):
        for c in range(-(-N // 32)):
            blk = x[i, 32 * c:32 * c + 32]           # the last block may be shorter
            e = scale_of(np.abs(blk).max())
            scale_row[i, c] = e
            out_row[i, 32 * c:32 * c + len(blk)] = [encode(v * 2.0 ** (127 - e)) for v in blk]
    for r in range(-(-M // 32)):
        for j in range(N):
            blk = x[32 * r:32 * r + 32, j]
            e = scale_of(np.abs(blk).max())
            scale_col[r, j] = e
            out_col[32 * r:32 * r + len(blk), j] = [encode(v * 2.0 ** (127 - e)) for v in blk]
    return out_row, scale_row, out_col, scale_col


def structured_input(M, N, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N)) * np.exp2(rng.integers(-12, 12, (M, 1)))   # row scales differ
    a *= np.exp2(rng.integers(-6, 6, (1, N)))                                  # column scales differ
    a[0, :32] = 0.0
    a[:32, 0] = 0.0
    if M > 1:
        a[1, 32:64] = rng.standard_normal(a[1, 32:64].shape) * 1e-39          # subnormal block
    if M > 5 and N > 7:
        a[5, 7] = 3000.0
    if M % 32:   # the last, partial column blocks get their own outlier
        a[-1, -1] = -1500.0
    return wl.to_bf16_bits(a)


@pytest.mark.parametrize("fmt,M,N", [(E4M3, 64, 96), (E5M2, 96, 64), (E4M3, 45, 80), (E5M2, 71, 48),
                                     (E4M3, 7, 16), (E4M3, 33, 33)])
def test_quantize_matches_brute_force(oracle_mod, fmt, M, N):
    x = structured_input(M, N, seed=M + N + fmt)
    got = oracle_mod.quantize(x, fmt)[:4]
    want = brute_force(x, fmt)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), got, want):
        assert np.array_equal(g, w), name


# ---- bounds, dbias, grouped -----------------------------------------------------

@pytest.mark.parametrize("name", ["small_128x256"])
def test_roundtrip_error_bound(oracle_mod, name):
    w = wl.make(name)
    fmt = w["fmt"]
    x = torch.from_numpy(w["x"].view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    out_row, scale_row, out_col, scale_col, _ = oracle_mod.quantize(w["x"], fmt)
    table = torch_decode_table(fmt)
    for q, s in ((out_row, np.repeat(scale_row, 32, axis=1)), (out_col, np.repeat(scale_col, 32, axis=0))):
        sc = np.exp2(s.astype(np.float64) - 127)
        v = np.abs(x) / sc
        ex = np.maximum(np.floor(np.log2(np.where(v > 0, v, 1.0))), EMIN[fmt])
        half_ulp = np.exp2(ex - MBITS[fmt]) / 2
        assert np.all(np.abs(table[q] * sc - x) <= half_ulp * sc)
        assert np.all(v <= FMAX[fmt])


def test_dbias_matches_fsum(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(5))
    M, N = 96, 64
    a = rng.standard_normal((M, N))
    a[:, 0] = rng.integers(-50, 50, M)                 # exact small integers
    a[:, 1] = np.exp2(rng.integers(-10, 10, M))         # exact powers of two
    a[:, 2] = 1.0                                        # an fp32 running sum loses these ones
    a[0, 2] = 2.0 ** 24                                  # behind 2^24; the exact sum keeps them
    a[:, 3] *= np.exp2(rng.integers(-20, 20, M))         # wide exponent spread
    x = wl.to_bf16_bits(a)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    dbias = oracle_mod.quantize(x, E5M2, with_dbias=True)[4]
    want = np.array([math.fsum(xv[:, j]) for j in range(N)], np.float32)
    assert np.array_equal(dbias, want)
    assert dbias[0] == float(np.sum(xv[:, 0]))
    assert dbias[2] == np.float32(2.0 ** 24 + 95)


def test_grouped_equals_flat_and_rejects_bad_offsets(oracle_mod):
    sizes = wl.moe_group_sizes(8, 512, seed=3, forced_empty=2)
    off = wl.offsets_from_sizes(sizes)
    x = wl.moe_bf16(sizes, 96, seed=3)
    flat = oracle_mod.quantize(x, E4M3)[:4]
    grouped = oracle_mod.quantize_grouped(x, off, E4M3)
    for f, g in zip(flat, grouped):
        assert np.array_equal(f, g)
    for bad in ([0, 256, 128, 512], [0, 256, 480], [32, 512], [0, 16, 8, 512]):
        with pytest.raises(ValueError):
            oracle_mod.quantize_grouped(x, np.array(bad), E4M3)


def test_grouped_unaligned_groups_are_separate_flat_problems(oracle_mod):
    """Offsets that are not multiples of 32: every group is quantized on its own (its columnwise
    blocks start at its first row and its last block is partial), and its ceil(rows/32) columnwise
    scale rows follow those of the groups before it.  The flat oracle is pinned on its own above."""
    sizes = np.array([45, 0, 1, 31, 33, 96, 70], np.int64)
    off = wl.offsets_from_sizes(sizes)
    N = 72
    x = wl.moe_bf16(sizes, N, seed=11)
    for fmt in (E4M3, E5M2):
        o_row, s_row, o_col, s_col = oracle_mod.quantize_grouped(x, off, fmt)
        assert s_col.shape == (2 + 0 + 1 + 1 + 2 + 3 + 3, N) == (oracle_mod.grouped_scale_col_rows(off), N)
        s0 = 0
        for g in range(len(sizes)):
            a, b = off[g], off[g + 1]
            if a == b:
                continue
            f_row, f_srow, f_col, f_scol, _ = oracle_mod.quantize(x[a:b], fmt)
            assert np.array_equal(o_row[a:b], f_row) and np.array_equal(s_row[a:b], f_srow)
            assert np.array_equal(o_col[a:b], f_col)
            assert np.array_equal(s_col[s0:s0 + f_scol.shape[0]], f_scol)
            s0 += f_scol.shape[0]
        assert s0 == s_col.shape[0]


def test_grouped_partial_block_takes_its_own_rows_only(oracle_mod):
    """Hand-worked: group 0 has 45 rows, so its second columnwise block is rows 32..44 only.  Those
    rows hold 1.0 and the next group's rows hold 1000, which must not reach that block's scale:
    e = ceil(log2(1/448)) + 127 = 119 and 1.0 * 2^(127-119) = 256 -> E4M3 0x78; group 1's first
    block (1000) gets ceil(log2(1000/448)) + 127 = 129 at scale row ceil(45/32) = 2, and
    1000 * 2^-2 = 250 rounds to 256 in E4M3 (neighbours 240 and 256, tie-free) -> 0x78."""
    N = 32
    a = np.zeros((45 + 40, N))
    a[:32] = 0.5
    a[32:45] = 1.0
    a[45:] = 1000.0
    off = np.array([0, 45, 85], np.int64)
    _, _, o_col, s_col = oracle_mod.quantize_grouped(wl.to_bf16_bits(a), off, E4M3)
    assert s_col.shape == (2 + 2, N)
    assert np.all(s_col[0] == 118) and np.all(s_col[1] == 119) and np.all(s_col[2] == 129)
    assert np.all(o_col[32:45] == 0x78) and np.all(o_col[45:77] == 0x78)
    assert np.all(s_col[3] == 129)                     # rows 77..84: a block of 8 rows of 1000


def test_moe_sizes_recipe():
    sizes = wl.moe_group_sizes(64, 65536, seed=4)
    assert sizes.sum() == 65536 and np.all(sizes % 32 == 0)
    assert (sizes == 0).sum() >= 4


# ---- GEMM-ready scale layout and per-tensor amax -----------------------------------

SWZ_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "swizzle_offsets.txt")


def test_swizzle_offsets_hand_worked(oracle_mod):
    for line in open(SWZ_GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        shape, rc, off = [p.strip() for p in line.split("|")]
        R, C = map(int, shape.split())
        r, c = map(int, rc.split())
        assert oracle_mod.swizzle_offset(r, c, C) == int(off), line


@pytest.mark.parametrize("R,C", [(128, 4), (256, 8), (100, 5), (300, 13), (32, 1)])
def test_swizzle_equals_tile_transpose(oracle_mod, R, C):
    # The same layout written as a reshape/transpose of the zero-padded plain
    # matrix: [R/128, 4, 32, C/4, 4] (row tile, 32-row group, row in group,
    # column tile, column) -> order (row tile, column tile, row in group,
    # 32-row group, column).
    rng = np.random.Generator(np.random.PCG64(R * 31 + C))
    plain = rng.integers(1, 255, (R, C)).astype(np.uint8)
    Rp, Cp = -(-R // 128) * 128, -(-C // 4) * 4
    padded = np.zeros((Rp, Cp), np.uint8)
    padded[:R, :C] = plain
    want = padded.reshape(Rp // 128, 4, 32, Cp // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    got = oracle_mod.swizzle_scales(plain)
    assert np.array_equal(got, want)


def test_amax_matches_numpy(oracle_mod):
    x = structured_input(96, 160, seed=17)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert oracle_mod.amax(x) == np.float32(np.abs(xv).max())
    assert oracle_mod.amax(np.zeros((32, 32), np.uint16)) == 0.0


# ---- fused activation -----------------------------------------------------------

def torch_act64(x64, act):
    import torch.nn.functional as F
    t = torch.from_numpy(x64)
    if act == 1:
        return torch.relu(t).numpy()
    if act == 2:
        return (torch.relu(t) ** 2).numpy()
    if act == 3:
        return F.gelu(t, approximate="tanh").numpy()
    if act == 4:
        return F.silu(t).numpy()
    return (t * torch.sigmoid(1.702 * t)).numpy()


@pytest.mark.parametrize("act", [1, 2, 3, 4, 5])
def test_activation_matches_torch_float64(oracle_mod, act):
    x = structured_input(64, 96, seed=act)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    want = torch_act64(xv, act).astype(np.float32)       # library routine in fp64, rounded once
    got = oracle_mod.activate(x, act)
    if act in (1, 2):
        assert np.array_equal(got, want)                 # exact for ReLU and squared ReLU
    else:
        # torch evaluates GeLU as 0.5 x (1 + tanh(.)), which cancels for x << 0; the slack
        # 1e-15 |x| covers that and still catches any wrong constant or formula
        assert np.all(np.abs(got.astype(np.float64) - want) <= 2 ** -22 * np.abs(want) + 1e-15 * np.abs(xv) + 1e-38)
    assert np.all(got[xv < 0] >= (-0.3 if act > 2 else 0.0))


@pytest.mark.parametrize("shape", [(96, 64), (45, 80)])
def test_act_none_quantize_f32_equals_bf16_path(oracle_mod, shape):
    x = structured_input(*shape, seed=11)
    y = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).float().numpy()
    a = oracle_mod.quantize(x, 0, with_dbias=True)
    b = oracle_mod.quantize_f32(y, 0, with_dbias=True)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_relu_quantize_hand_checks(oracle_mod):
    # a row block of -1 and +2 with ReLU: values 0 and 2, amax 2 -> e = ceil(log2(2/448)) + 127 = 120;
    # 2 * 2^7 = 256 -> 0x78, zeros -> 0x00 (ReLU gives +0)
    x = wl.to_bf16_bits(np.tile(np.array([-1.0, 2.0] * 16), (32, 1)))
    o_row, s_row, _, _, _ = oracle_mod.quantize_act(x, 0, 1)
    assert s_row[0, 0] == 120 and o_row[0, :2].tolist() == [0x00, 0x78]


def test_grouped_dbias_is_per_group_fsum(oracle_mod):
    sizes = np.array([64, 0, 96, 32], np.int64)
    off = wl.offsets_from_sizes(sizes)
    x = wl.moe_bf16(sizes, 48, seed=6)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_mod.grouped_dbias(x, off)
    for g in range(len(sizes)):
        rows = xv[off[g]:off[g + 1]]
        want = np.array([math.fsum(rows[:, j]) for j in range(48)], np.float32)
        assert np.array_equal(got[g], want)
    assert np.all(got[1] == 0.0)
    # the groups' sums add up to the flat dbias (up to fp32 rounding of each)
    flat = oracle_mod.quantize(x, 0, False, False, with_dbias=True)[4]
    assert np.allclose(got.astype(np.float64).sum(0), flat, rtol=1e-6, atol=1e-30)
    with pytest.raises(ValueError):
        oracle_mod.grouped_dbias(x, np.array([0, 100, 64, 192]))
    # unaligned groups: each group's exact column sums as well
    off2 = np.array([0, 45, 45, 46, 192], np.int64)
    got2 = oracle_mod.grouped_dbias(x, off2)
    for g in range(4):
        rows = xv[off2[g]:off2[g + 1]]
        assert np.array_equal(got2[g], np.array([math.fsum(rows[:, j]) for j in range(48)], np.float32))



@pytest.mark.parametrize("act", [1, 2, 3, 4, 5])
def test_dactivation_matches_torch_autograd(oracle_mod, act):
    x = structured_input(32, 96, seed=act + 20)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    t = torch.from_numpy(xv.copy()).requires_grad_(True)
    import torch.nn.functional as F
    if act == 1:
        y = torch.relu(t)
    elif act == 2:
        y = torch.relu(t) ** 2
    elif act == 3:
        y = F.gelu(t, approximate="tanh")
    elif act == 4:
        y = F.silu(t)
    else:
        y = t * torch.sigmoid(1.702 * t)
    y.sum().backward()
    want = t.grad.numpy()
    got = np.array([oracle_mod.dactivation_f64(v, act) for v in xv.ravel()]).reshape(xv.shape)
    if act in (1, 2):
        want = np.where(xv > 0, want, 0.0)        # torch's relu'(0) = 0 as well
        assert np.array_equal(got, want)
    else:
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_dactivate_products_are_rounded_once(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(31))
    dy = wl.to_bf16_bits(rng.standard_normal((32, 64)))
    x = wl.to_bf16_bits(rng.standard_normal((32, 64)))
    dyv = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_mod.dactivate(dy, x, 2)                 # squared ReLU: dY * 2X, exact in fp32
    assert np.array_equal(got.astype(np.float64), np.where(xv > 0, dyv * 2 * xv, 0.0))
    got = oracle_mod.dactivate(dy, x, 1)
    assert np.array_equal(got.astype(np.float64), np.where(xv > 0, dyv, 0.0))



@pytest.mark.parametrize("act", [3, 4, 5])
def test_dactivation_sign_for_very_negative_inputs(oracle_mod, act):
    # for x below the activation's minimum the derivative is negative, however small:
    # its sign must survive underflow (a negative value that rounds to zero stays -0)
    for x in (-5.0, -12.0, -25.0, -100.0, -1e4):
        d = oracle_mod.dactivation_f64(x, act)
        assert d <= 0.0 and math.copysign(1.0, d) == -1.0, (act, x, d)
    assert oracle_mod.dactivation_f64(-0.5, 4) > 0.0 and oracle_mod.dactivation_f64(1.0, 3) > 1.0


# ---- gated activations: act(a) * b with x = [a | b] -----------------------------------

_BF16_FINITE = np.arange(65536, dtype=np.uint32).astype(np.uint16)
_BF16_FINITE = _BF16_FINITE[(_BF16_FINITE & 0x7F80) != 0x7F80]


@pytest.mark.parametrize("act", [1, 2, 3, 4, 5])
def test_gate_with_unit_linear_half_is_the_activation(oracle_mod, act):
    """b = 1 everywhere: act(a) * 1 rounds once to fp32 just as the activation alone, for every
    finite BF16 a; with b = 2^-3 the result is that value scaled exactly, wherever the scaled value
    is a normal fp32 number (an eighth of a subnormal is rounded again)."""
    a = _BF16_FINITE[: (_BF16_FINITE.size // 64) * 64].reshape(-1, 64)
    if act == 2:   # squared ReLU overflows fp32 for |a| >= 2^64
        a = np.where((a & 0x7F80) >= ((127 + 64) << 7), 0, a).astype(np.uint16)
    one = np.full_like(a, 0x3F80)
    got = oracle_mod.gate(np.concatenate([a, one], axis=1), act)
    assert np.array_equal(got.view(np.uint32), oracle_mod.activate(a, act).view(np.uint32))
    eighth = np.full_like(a, 0x3E00)                          # BF16 0.125
    got8 = oracle_mod.gate(np.concatenate([a, eighth], axis=1), act).astype(np.float64)
    ref = oracle_mod.activate(a, act).astype(np.float64) / 8
    normal = np.abs(ref) >= 2.0 ** -126
    assert np.array_equal(got8[normal], ref[normal])


def test_gate_hand_worked(oracle_mod):
    # a = [-2, 3, 0, 20], b = [5, -4, 7, 0.5]:
    #   ReGLU   [0, -12, 0, 10];  squared-ReLU GLU [0, -36, 0, 200];
    #   SwiGLU of a = 0 is 0; GeGLU(20) = 20 (sigmoid(603) is 1 in double) -> 20 * 0.5 = 10
    x = wl.to_bf16_bits(np.array([[-2.0, 3.0, 0.0, 20.0, 5.0, -4.0, 7.0, 0.5]]))
    assert oracle_mod.gate(x, 1).tolist() == [[0.0, -12.0, 0.0, 10.0]]
    assert oracle_mod.gate(x, 2).tolist() == [[0.0, -36.0, 0.0, 200.0]]
    assert oracle_mod.gate(x, 4)[0, 2] == 0.0 and oracle_mod.gate(x, 3)[0, 3] == 10.0
    # the halves are not interchangeable: with them swapped, ReGLU would give [-10, 0, 0, 10]
    assert oracle_mod.gate(x, 1)[0, 0] == 0.0


@pytest.mark.parametrize("act", [3, 4, 5])
def test_gate_matches_torch_float64(oracle_mod, act):
    import torch.nn.functional as F
    x = structured_input(48, 2 * 40, seed=20 + act)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    a, b = xv[:, :40], xv[:, 40:]
    if act == 3:
        want = F.gelu(a, approximate="tanh") * b
    elif act == 4:
        want = F.silu(a) * b
    else:
        want = a * torch.sigmoid(1.702 * a) * b
    want = want.numpy()
    got = oracle_mod.gate(x, act).astype(np.float64)
    assert np.all(np.abs(got - want) <= 2 ** -22 * np.abs(want) + 1e-15 * np.abs(a.numpy() * b.numpy()) + 1e-38)


def test_quantize_gated_is_the_cast_of_the_gate(oracle_mod):
    x = structured_input(64, 2 * 96, seed=5)
    for act in (1, 4):
        q = oracle_mod.quantize_gated(x, 1, act)
        r = oracle_mod.quantize_f32(oracle_mod.gate(x, act), 1)
        for u, v in zip(q, r[:4]):
            assert np.array_equal(u, v)


@pytest.mark.parametrize("act", [1, 2, 3, 4, 5])
def test_dgate_matches_torch_autograd(oracle_mod, act):
    """(da, db) of y = act(a) * b against torch autograd in float64 (the library's own derivative)."""
    import torch.nn.functional as F
    N = 40
    x = structured_input(32, 2 * N, seed=40 + act)
    g = structured_input(32, N, seed=50 + act)
    xv = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    gv = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    a = xv[:, :N].clone().requires_grad_(True)
    b = xv[:, N:].clone().requires_grad_(True)
    if act == 1:
        ya = torch.relu(a)
    elif act == 2:
        ya = torch.relu(a) ** 2
    elif act == 3:
        ya = F.gelu(a, approximate="tanh")
    elif act == 4:
        ya = F.silu(a)
    else:
        ya = a * torch.sigmoid(1.702 * a)
    (ya * b).backward(gv)
    da, db = oracle_mod.dgate(g, x, act)
    # one fp32 rounding on the oracle's side; torch's tanh-form GeLU derivative cancels for a << 0,
    # which the 1e-12 |g| (|b| + 1) slack covers (as in the derivative's own pin above)
    slack = 1e-12 * np.abs(gv.numpy()) * (np.abs(xv[:, N:].numpy()) + 1) + 1e-38
    for got, want in ((da, a.grad.numpy()), (db, b.grad.numpy())):
        if act in (1, 2):
            assert np.array_equal(got.astype(np.float64), want.astype(np.float32).astype(np.float64))
        else:
            assert np.all(np.abs(got.astype(np.float64) - want) <= 2 ** -23 * np.abs(want) + slack)


def test_dgate_hand_worked_and_layout(oracle_mod):
    # ReGLU: a = [-2, 3], b = [5, -4], g = [1, 2]: da = g b relu'(a) = [0, -8], db = g relu(a) = [0, 6]
    x = wl.to_bf16_bits(np.array([[-2.0, 3.0, 5.0, -4.0]]))
    g = wl.to_bf16_bits(np.array([[1.0, 2.0]]))
    da, db = oracle_mod.dgate(g, x, 1)
    assert da.tolist() == [[0.0, -8.0]] and db.tolist() == [[0.0, 6.0]]
    # N a multiple of 32: [da | db] quantized as one [M, 2N] tensor; otherwise side by side
    for N in (64, 40):
        xs = structured_input(64, 2 * N, seed=N)
        gs = structured_input(64, N, seed=N + 1)
        q = oracle_mod.quantize_dgated(gs, xs, 1, 4)
        da, db = oracle_mod.dgate(gs, xs, 4)
        both = oracle_mod.quantize_f32(np.concatenate([da, db], axis=1), 1)
        assert q[0].shape == (64, 2 * N) and q[1].shape == (64, 2 * -(-N // 32)) and q[3].shape == (2, 2 * N)
        if N % 32 == 0:
            for u, v in zip(q, both[:4]):
                assert np.array_equal(u, v)
        else:
            qa = oracle_mod.quantize_f32(da, 1)
            assert np.array_equal(q[1][:, :2], qa[1]) and np.array_equal(q[0][:, :N], qa[0])


def test_gated_grouped_is_per_group_gated_cast(oracle_mod):
    """The grouped gated cast: with 32-row-multiple groups it equals the gated cast of all rows
    (no block crosses a group); with ragged groups each group equals the gated cast of its rows."""
    N = 40
    for sizes, flat_equal in (([64, 0, 32, 96], True), ([45, 1, 0, 83, 31], False)):
        off = wl.offsets_from_sizes(np.array(sizes, np.int64))
        x = structured_input(int(off[-1]), 2 * N, seed=len(sizes))
        q = oracle_mod.quantize_gated_grouped(x, off, 1, 4)
        if flat_equal:
            for u, v in zip(q, oracle_mod.quantize_gated(x, 1, 4)):
                assert np.array_equal(u, v)
        s0 = 0
        for g in range(len(sizes)):
            a, b = off[g], off[g + 1]
            if a == b:
                continue
            f = oracle_mod.quantize_gated(x[a:b], 1, 4)
            assert np.array_equal(q[0][a:b], f[0]) and np.array_equal(q[1][a:b], f[1])
            assert np.array_equal(q[2][a:b], f[2]) and np.array_equal(q[3][s0:s0 + f[3].shape[0]], f[3])
            s0 += f[3].shape[0]
        assert s0 == q[3].shape[0]
    with pytest.raises(ValueError):
        oracle_mod.quantize_gated_grouped(x, np.array([0, 100, 50, 160]), 1, 4)


def test_grouped_activated_is_per_group_activated_cast(oracle_mod):
    """act(x) cast per group: aligned groups give the flat activated cast of all rows; ragged
    groups give each group's own activated cast."""
    N = 40
    for sizes, flat_equal in (([64, 0, 32, 96], True), ([45, 1, 0, 83, 31], False)):
        off = wl.offsets_from_sizes(np.array(sizes, np.int64))
        x = structured_input(int(off[-1]), N, seed=7 + len(sizes))
        q = oracle_mod.quantize_grouped_act(x, off, 0, 3)
        if flat_equal:
            for u, v in zip(q, oracle_mod.quantize_act(x, 0, 3)[:4]):
                assert np.array_equal(u, v)
        s0 = 0
        for g in range(len(sizes)):
            a, b = off[g], off[g + 1]
            if a == b:
                continue
            f = oracle_mod.quantize_act(x[a:b], 0, 3)
            assert np.array_equal(q[0][a:b], f[0]) and np.array_equal(q[2][a:b], f[2])
            assert np.array_equal(q[3][s0:s0 + f[3].shape[0]], f[3])
            s0 += f[3].shape[0]


def test_grouped_swizzled_planes(oracle_mod):
    """Per-group GEMM-ready planes: one group gives the flat call's swizzled planes; groups of
    128-row multiples give the flat rowwise plane (row tiles in order); ragged groups give each
    group's own swizzled planes, padded and concatenated."""
    N = 96
    x = structured_input(384, N, seed=31)
    flat = oracle_mod.quantize(x, 0)
    one = oracle_mod.quantize_grouped_swizzled(x, np.array([0, 384]), 0)
    assert np.array_equal(one[1], oracle_mod.swizzle_scales(flat[1]))
    assert np.array_equal(one[3], oracle_mod.swizzle_scales(np.ascontiguousarray(flat[3].T)))
    three = oracle_mod.quantize_grouped_swizzled(x, np.array([0, 128, 128, 384]), 0)
    assert np.array_equal(three[1], oracle_mod.swizzle_scales(flat[1]))
    ragged = oracle_mod.quantize_grouped_swizzled(x, np.array([0, 45, 45, 300, 384]), 0)
    # sizes: ceil(45/128) + ceil(255/128) + ceil(84/128) = 4 tiles of 128 x 4 (rowwise) and 4 x 128 (colwise)
    assert ragged[1].size == 4 * 128 * 4 and ragged[3].size == 4 * 4 * 128
    g1 = oracle_mod.quantize(x[45:300], 0)
    assert np.array_equal(ragged[1][512:512 + 1024], oracle_mod.swizzle_scales(g1[1]))
    assert np.array_equal(ragged[3][512:512 + 1024], oracle_mod.swizzle_scales(np.ascontiguousarray(g1[3].T)))
    assert np.array_equal(ragged[0], oracle_mod.quantize_grouped(x, np.array([0, 45, 45, 300, 384]), 0)[0])
