"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

FP8 and E8M0 bytes must be bit-exact.  dbias must satisfy
|gpu - oracle| <= 1e-5 * sum_i |x[i, j]| per column: the kernels add in fp32
in a fixed order (16 rows, their partner 16 rows, 4 row blocks per tile; then
8 tiles per warp and 16 warps at 16384 rows), at most ~42 roundings of
sum|x|, about 2.5e-6 relative, so 1e-5 leaves a 4x margin.

Every shape is compared element by element, the full-size workloads
(8192x28672, 16384x8192 with dbias on every column, the 64-expert 65536x7168
grouped call) included: the oracle runs on 32-aligned column slices on every
host core (tests/oracle_slices.py), which reassemble into its whole-matrix
result.  Only the 69632x65536 case past 2^32 elements is checked on sampled
32-row stripes and 32-column slices, which the oracle computes on their own (a
stripe of 32 rows holds complete rowwise and columnwise blocks).  Every output
sits between 4 KiB canary bands that must stay untouched.
"""
import numpy as np
import pytest
import torch

import mxfp8_block_scaled_04_gb300 as mx
import oracle_slices
from mxfp8_block_scaled_04_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

E4M3, E5M2 = 0, 1
GUARD = 4096
CANARY = 0xA5


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


class Guarded:
    """A device buffer with canary bands on both sides."""

    def __init__(self, shape, dtype=torch.uint8, fill=CANARY):
        n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        self.raw = torch.full((n + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.raw[GUARD:GUARD + n].fill_(fill)
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)

    def guards_intact(self):
        return bool((self.raw[:GUARD] == CANARY).all() and (self.raw[-GUARD:] == CANARY).all())


def run_quantize(x_bits, fmt, rowwise=True, colwise=True, with_dbias=False, noop=None, prefill=CANARY):
    M, N = x_bits.shape
    x = dev_bf16(x_bits)
    bufs = dict(
        out_row=Guarded((M, N), fill=prefill) if rowwise else None,
        scale_row=Guarded((M, -(-N // 32)), fill=prefill) if rowwise else None,
        out_col=Guarded((M, N), fill=prefill) if colwise else None,
        scale_col=Guarded((-(-M // 32), N), fill=prefill) if colwise else None,
        dbias=Guarded((N,), torch.float32, fill=prefill) if with_dbias else None,
    )
    ws = None
    if with_dbias:
        ws = torch.empty(max(mx.mxfp8_quantize_workspace_bytes(M, N, True), 16), dtype=torch.uint8, device="cuda")
    t = {k: (v.t if v is not None else None) for k, v in bufs.items()}
    before = mx.mxfp8_kernel_launch_count()
    st = mx.mxfp8_quantize(x, M, N, fmt, t["out_row"], t["scale_row"], t["out_col"], t["scale_col"],
                           t["dbias"], ws, noop, None)
    assert st == 0, mx.mxfp8_status_string(st)
    torch.cuda.synchronize()
    if M > 0 and N > 0:
        assert mx.mxfp8_kernel_launch_count() > before     # the CUDA kernel really ran
    for k, v in bufs.items():
        if v is not None:
            assert v.guards_intact(), f"{k}: canary band overwritten"
    host = {k: (v.t.cpu().numpy() if v is not None else None) for k, v in bufs.items()}
    return host


def assert_bytes_equal(got, want, name):
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches; first at {i}: gpu {got[i]:#04x} oracle {want[i]:#04x}")


def check_against_oracle(oracle_mod, x_bits, fmt, host, rowwise=True, colwise=True):
    o_row, s_row, o_col, s_col, _ = oracle_mod.quantize(x_bits, fmt, rowwise, colwise)
    if rowwise:
        assert_bytes_equal(host["scale_row"], s_row, "scale_row")
        assert_bytes_equal(host["out_row"], o_row, "out_row")
    if colwise:
        assert_bytes_equal(host["scale_col"], s_col, "scale_col")
        assert_bytes_equal(host["out_col"], o_col, "out_col")


def dbias_tolerance(x_bits):
    xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double()
    return 1e-5 * xv.abs().sum(dim=0).numpy()


def mixed_input(M, N, seed):
    """N(0,1) with per-row exponent spread, zeros, subnormals, outliers, powers of two."""
    rng = np.random.Generator(np.random.PCG64(seed))
    a = rng.standard_normal((M, N)) * np.exp2(rng.integers(-20, 20, (M, 1)))
    flat = a.reshape(-1)
    n = flat.size
    flat[rng.integers(0, n, n // 50)] = rng.standard_normal(n // 50) * 1e-39
    flat[rng.integers(0, n, n // 100)] = np.exp2(rng.integers(-30, 30, n // 100)) * rng.choice([-1, 1], n // 100)
    flat[rng.integers(0, n, n // 200)] = 0.0
    flat[rng.integers(0, n, n // 500)] = -0.0
    a[:32, :32] = 0.0
    if M >= 64 and N >= 64:
        a[32:64, 32:64] = rng.standard_normal((32, 32)) * 1e-39
    return wl.to_bf16_bits(a)


SHAPES = [(32, 32), (64, 96), (96, 160), (160, 96), (128, 256), (256, 384), (384, 224),
          (128, 8192), (544, 1056), (1024, 64)]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", SHAPES)
def test_parity_shapes(oracle_mod, shape, fmt):
    M, N = shape
    x = mixed_input(M, N, seed=M * 7 + N + fmt)
    host = run_quantize(x, fmt)
    check_against_oracle(oracle_mod, x, fmt, host)


def test_parity_small_workload(oracle_mod):
    w = wl.make("small_128x256")
    host = run_quantize(w["x"], w["fmt"])
    check_against_oracle(oracle_mod, w["x"], w["fmt"], host)


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_parity_single_direction(oracle_mod, rowwise, colwise):
    x = mixed_input(160, 288, seed=11)
    host = run_quantize(x, E4M3, rowwise=rowwise, colwise=colwise)
    check_against_oracle(oracle_mod, x, E4M3, host, rowwise, colwise)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", [(32, 32), (96, 160), (384, 224), (1056, 288)])
def test_parity_dbias(oracle_mod, shape, fmt):
    M, N = shape
    x = mixed_input(M, N, seed=3 * M + N)
    host = run_quantize(x, fmt, with_dbias=True)
    check_against_oracle(oracle_mod, x, fmt, host)
    want = oracle_mod.quantize(x, fmt, False, False, with_dbias=True)[4]
    assert np.all(np.abs(host["dbias"].astype(np.float64) - want) <= dbias_tolerance(x))


def test_dbias_exact_columns(oracle_mod):
    rng = np.random.Generator(np.random.PCG64(9))
    M, N = 512, 64
    a = rng.integers(-64, 64, (M, N)).astype(np.float64)      # sums are exact in fp32
    a[:, 1] = np.exp2(rng.integers(-8, 8, M))
    x = wl.to_bf16_bits(a)
    host = run_quantize(x, E5M2, with_dbias=True)
    want = oracle_mod.quantize(x, E5M2, False, False, with_dbias=True)[4]
    assert np.array_equal(host["dbias"], want)


@pytest.mark.parametrize("with_dbias", [False, True])
def test_noop_flag(oracle_mod, with_dbias):
    x = mixed_input(256, 384, seed=5)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    zero = torch.zeros(1, dtype=torch.float32, device="cuda")
    host = run_quantize(x, E5M2, with_dbias=with_dbias, noop=one, prefill=0x3C)
    for k, v in host.items():
        if v is not None:
            assert np.all(v.view(np.uint8) == 0x3C), f"{k} written despite noop"
    host = run_quantize(x, E5M2, with_dbias=with_dbias, noop=zero, prefill=0x3C)
    check_against_oracle(oracle_mod, x, E5M2, host)


def test_empty_rows_dbias_zero():
    x = np.zeros((0, 64), np.uint16)
    host = run_quantize(x, E4M3, with_dbias=True, prefill=0x3C)
    assert np.all(host["dbias"] == 0.0)


# ---- grouped -------------------------------------------------------------------

def run_grouped(x_bits, offsets, fmt, noop=None, prefill=CANARY):
    total, N = x_bits.shape
    x = dev_bf16(x_bits)
    off = torch.from_numpy(np.asarray(offsets, np.int64)).cuda()
    srows = max(mx.grouped_scale_col_rows(np.maximum.accumulate(np.asarray(offsets, np.int64))), 1)
    bufs = dict(out_row=Guarded((total, N), fill=prefill), scale_row=Guarded((total, -(-N // 32)), fill=prefill),
                out_col=Guarded((total, N), fill=prefill), scale_col=Guarded((srows, N), fill=prefill))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = mx.mxfp8_quantize_grouped(x, total, N, off.numel() - 1, off, fmt, bufs["out_row"].t,
                                   bufs["scale_row"].t, bufs["out_col"].t, bufs["scale_col"].t,
                                   None, noop, err, None)
    assert st == 0, mx.mxfp8_status_string(st)
    torch.cuda.synchronize()
    for k, v in bufs.items():
        assert v.guards_intact(), k
    return {k: v.t.cpu().numpy() for k, v in bufs.items()}, int(err.item())


@pytest.mark.parametrize("N", [96, 160, 512])
def test_parity_grouped(oracle_mod, N):
    sizes = np.array([64, 0, 32, 416, 0, 0, 128, 96, 160, 32], np.int64)
    off = wl.offsets_from_sizes(sizes)
    x = wl.moe_bf16(sizes, N, seed=N)
    host, err = run_grouped(x, off, E4M3)
    assert err == 0
    o = oracle_mod.quantize_grouped(x, off, E4M3)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"),
                          (host["out_row"], host["scale_row"], host["out_col"], host["scale_col"]), o):
        assert_bytes_equal(g, w, name)


UNALIGNED_SIZES = [
    np.array([45, 0, 1, 31, 33, 96, 70, 127, 129, 0, 13], np.int64),   # partial blocks everywhere
    np.array([1] * 40 + [300], np.int64),                                 # many one-row groups
    np.array([0, 200, 0], np.int64),                                      # one group, empties around it
    np.array([17, 15], np.int64),                                         # both groups inside one block
]


@pytest.mark.parametrize("case", range(len(UNALIGNED_SIZES)))
@pytest.mark.parametrize("fmt,N", [(E4M3, 96), (E5M2, 160), (E4M3, 40), (E5M2, 1032)])
def test_parity_grouped_unaligned_offsets(oracle_mod, case, fmt, N):
    """Groups that are not multiples of 32 rows: each is its own flat problem, whose last
    columnwise block must not take in the next group's rows (which the tile loads with it)."""
    sizes = UNALIGNED_SIZES[case]
    off = wl.offsets_from_sizes(sizes)
    x = wl.moe_bf16(sizes, N, seed=int(sizes.sum()) + N)
    host, err = run_grouped(x, off, fmt)
    assert err == 0
    o = oracle_mod.quantize_grouped(x, off, fmt)
    for name, w in zip(("out_row", "scale_row", "out_col", "scale_col"), o):
        assert_bytes_equal(host[name], w, name)


def test_parity_grouped_unaligned_next_group_dominates(oracle_mod):
    """The rows after a group's partial last block are 1000x larger: any leak into that block's
    amax changes its scale byte."""
    sizes = np.array([45, 83, 1, 64], np.int64)
    off = wl.offsets_from_sizes(sizes)
    a = np.random.Generator(np.random.PCG64(3)).standard_normal((int(sizes.sum()), 128))
    a[45:128] *= 1000.0
    a[129:] *= 1000.0
    x = wl.to_bf16_bits(a)
    host, err = run_grouped(x, off, E4M3)
    assert err == 0
    o = oracle_mod.quantize_grouped(x, off, E4M3)
    for name, w in zip(("out_row", "scale_row", "out_col", "scale_col"), o):
        assert_bytes_equal(host[name], w, name)


@pytest.mark.parametrize("offsets,valid", [
    ([0, 16, 928], True),           # valid: groups of 16 and 912 rows (each its own flat problem)
    ([0, 16, 8, 928], False),       # decreasing
    ([0, 512, 256, 928], False),    # decreasing
    ([0, 512, 896], False),         # last entry != total rows
    ([32, 928], False),             # first entry != 0
    ([0, 480, 928], True),          # valid: 480 and 448 rows
])
def test_grouped_offsets_validation(offsets, valid):
    x = wl.normal_bf16(928, 96, seed=1)
    host, err = run_grouped(x, offsets, E4M3, prefill=0x3C)
    if valid:
        assert err == 0
        return
    assert err == 1
    for k, v in host.items():
        assert np.all(v == 0x3C), f"{k} written despite invalid offsets"


def test_grouped_noop():
    sizes = np.array([64, 96], np.int64)
    x = wl.moe_bf16(sizes, 128, seed=2)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    host, err = run_grouped(x, wl.offsets_from_sizes(sizes), E4M3, noop=one, prefill=0x3C)
    assert err == 0
    for k, v in host.items():
        assert np.all(v == 0x3C), k


def test_no_device_fault_recorded():
    assert mx.mxfp8_device_fault_word() == 0


# ---- full-size workloads: every byte against the oracle ---------------------------

def test_parity_act_4096_full(oracle_mod):
    w = wl.make("act_4096x4096")
    host = run_quantize(w["x"], w["fmt"])
    check_against_oracle(oracle_mod, w["x"], w["fmt"], host)


def stripes_to_check(M, rng, must=()):
    n = M // 32
    picks = {0, n - 1, *must}
    picks |= set(rng.integers(0, n, 6).tolist())
    return sorted(p for p in picks if 0 <= p < n)


def check_stripes(oracle_mod, x_bits, fmt, out, stripes):
    N = x_bits.shape[1]
    for s in stripes:
        r0 = 32 * s
        xs = np.ascontiguousarray(x_bits[r0:r0 + 32])
        o_row, s_row, o_col, s_col, _ = oracle_mod.quantize(xs, fmt)
        assert_bytes_equal(out["out_row"][r0:r0 + 32].cpu().numpy(), o_row, f"out_row stripe {s}")
        assert_bytes_equal(out["scale_row"][r0:r0 + 32].cpu().numpy(), s_row, f"scale_row stripe {s}")
        assert_bytes_equal(out["out_col"][r0:r0 + 32].cpu().numpy(), o_col, f"out_col stripe {s}")
        assert_bytes_equal(out["scale_col"][s:s + 1].cpu().numpy(), s_col, f"scale_col stripe {s}")
    assert N % 32 == 0


def quantize_device(x_bits, fmt, with_dbias=False, noop=None):
    x = dev_bf16(x_bits)
    return x, mx.quantize(x, fmt, with_dbias=with_dbias, noop=noop)


def check_whole(got, want):
    for name, g, o in zip(("out_row", "scale_row", "out_col", "scale_col"), got, want):
        assert_bytes_equal(g, o, name)


def test_parity_fc1_8192x28672_full(oracle_mod):
    """The throughput shape: every FP8 byte and every scale byte of both directions."""
    w = wl.make("fc1_8192x28672")
    host = run_quantize(w["x"], w["fmt"])
    want = oracle_slices.quantize(oracle_mod, w["x"], w["fmt"])
    check_whole([host[k] for k in ("out_row", "scale_row", "out_col", "scale_col")], want)
    assert int(host["scale_row"].max()) <= 254 and int(host["scale_col"].max()) <= 254
    torch.cuda.empty_cache()


def test_parity_grad_16384x8192_full_with_dbias(oracle_mod):
    """E5M2 gradient with fused dbias: every byte of both directions, dbias on all 8192 columns,
    then the same call with noop = 1 on a zeroed input leaves every output as it was."""
    w = wl.make("grad_16384x8192")
    x_bits, fmt = w["x"], w["fmt"]
    M, N = x_bits.shape
    host = run_quantize(x_bits, fmt, with_dbias=True)
    want = oracle_slices.quantize(oracle_mod, x_bits, fmt, with_dbias=True)
    check_whole([host[k] for k in ("out_row", "scale_row", "out_col", "scale_col")], want)
    assert np.all(np.abs(host["dbias"].astype(np.float64) - want[4]) <= dbias_tolerance(x_bits))
    del host, want
    # noop = 1 at full size: nothing changes
    x, r = quantize_device(x_bits, fmt, with_dbias=True)
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    before = [t.clone() for t in (r.out_row, r.scale_row, r.out_col, r.scale_col, r.dbias)]
    ws = torch.empty(mx.mxfp8_quantize_workspace_bytes(M, N, True), dtype=torch.uint8, device="cuda")
    xin = torch.zeros_like(x)
    st = mx.mxfp8_quantize(xin, M, N, fmt, r.out_row, r.scale_row, r.out_col, r.scale_col, r.dbias, ws, one, None)
    assert st == 0
    torch.cuda.synchronize()
    for a, b in zip(before, (r.out_row, r.scale_row, r.out_col, r.scale_col, r.dbias)):
        assert torch.equal(a, b)
    del x, r, before, xin, ws
    torch.cuda.empty_cache()


def test_parity_beyond_2_32_elements_with_dbias(oracle_mod):
    """69632 x 65536 (4.56e9 elements, ~19 GB on the device): byte offsets into both FP8 planes pass
    2^31 and 2^32, the columnwise scale plane holds 1.4e8 bytes, and the dbias workspace 544 tiles.
    Checked on sampled 32-row stripes and 32-column slices (a whole compare would hold ~30 GB on the host)."""
    M, N, fmt = 69632, 65536, E5M2
    x_bits = wl.banded_bf16(M, N, seed=32)
    x, r = quantize_device(x_bits, fmt, with_dbias=True)
    torch.cuda.synchronize()
    rng = np.random.Generator(np.random.PCG64(32))
    # stripes holding byte offsets 2^31 and 2^32 of the FP8 planes, and the last one
    must = (0, (1 << 31) // N // 32, (1 << 32) // N // 32, M // 32 - 1)
    check_stripes(oracle_mod, x_bits, fmt, r._asdict(), stripes_to_check(M, rng, must=must))
    dbias = r.dbias.cpu().numpy()
    for j0 in sorted({0, N - 32, *(32 * rng.integers(0, N // 32, 2)).tolist()}):
        xs = np.ascontiguousarray(x_bits[:, j0:j0 + 32])
        _, _, o_col, s_col, db = oracle_mod.quantize(xs, fmt, rowwise=False, colwise=True, with_dbias=True)
        assert_bytes_equal(r.out_col[:, j0:j0 + 32].cpu().numpy(), o_col, f"out_col cols {j0}")
        assert_bytes_equal(r.scale_col[:, j0:j0 + 32].cpu().numpy(), s_col, f"scale_col cols {j0}")
        assert np.all(np.abs(dbias[j0:j0 + 32].astype(np.float64) - db) <= dbias_tolerance(xs)), j0
    del x, r, x_bits
    torch.cuda.empty_cache()


def test_parity_moe_64x65536x7168_full(oracle_mod):
    """The 64-expert grouped workload in one launch: every byte against the oracle's grouped call."""
    w = wl.make("moe_64x65536x7168")
    x_bits, off = w["x"], w["offsets"]
    host, err = run_grouped(x_bits, off, w["fmt"])
    assert err == 0
    want = oracle_slices.quantize_grouped(oracle_mod, x_bits, off, w["fmt"])
    check_whole([host[k] for k in ("out_row", "scale_row", "out_col", "scale_col")], want)
    torch.cuda.empty_cache()


# ---- shapes that are not multiples of 32 ------------------------------------------

RAGGED = [(45, 80), (71, 48), (1, 16), (33, 16), (130, 144), (1000, 1040), (257, 4112), (31, 4096)]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", RAGGED)
def test_parity_ragged_shapes(oracle_mod, shape, fmt):
    M, N = shape
    x = mixed_input(M, N, seed=M * 13 + N + fmt)
    host = run_quantize(x, fmt)
    check_against_oracle(oracle_mod, x, fmt, host)


# N a multiple of 8 but not of 16: FP8 rows only 8-byte aligned, each row's last segment 8 columns
NARROW = [(64, 8), (45, 24), (96, 40), (33, 8), (257, 1032), (130, 136), (1000, 2056)]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", NARROW)
def test_parity_n_multiple_of_8(oracle_mod, shape, fmt):
    M, N = shape
    x = mixed_input(M, N, seed=M * 17 + N + fmt)
    host = run_quantize(x, fmt, with_dbias=True)
    check_against_oracle(oracle_mod, x, fmt, host)
    want = oracle_mod.quantize(x, fmt, False, False, with_dbias=True)[4]
    assert np.all(np.abs(host["dbias"].astype(np.float64) - want) <= dbias_tolerance(x))


@pytest.mark.parametrize("rowwise,colwise", [(True, False), (False, True)])
def test_parity_n_multiple_of_8_single_direction(oracle_mod, rowwise, colwise):
    x = mixed_input(160, 40, seed=41)
    host = run_quantize(x, E4M3, rowwise=rowwise, colwise=colwise)
    check_against_oracle(oracle_mod, x, E4M3, host, rowwise, colwise)


@pytest.mark.parametrize("N", [24, 40, 1032])
def test_parity_grouped_n_multiple_of_8(oracle_mod, N):
    sizes = np.array([64, 0, 32, 224, 96], np.int64)
    off = wl.offsets_from_sizes(sizes)
    x = wl.moe_bf16(sizes, N, seed=N + 5)
    host, err = run_grouped(x, off, E5M2)
    assert err == 0
    o = oracle_mod.quantize_grouped(x, off, E5M2)
    for name, w in zip(("out_row", "scale_row", "out_col", "scale_col"), o):
        assert_bytes_equal(host[name], w, name)


@pytest.mark.parametrize("shape", [(45, 80), (1000, 1040)])
def test_parity_ragged_dbias(oracle_mod, shape):
    M, N = shape
    x = mixed_input(M, N, seed=M + 3 * N)
    host = run_quantize(x, E5M2, with_dbias=True)
    check_against_oracle(oracle_mod, x, E5M2, host)
    want = oracle_mod.quantize(x, E5M2, False, False, with_dbias=True)[4]
    assert np.all(np.abs(host["dbias"].astype(np.float64) - want) <= dbias_tolerance(x))



# ---- grouped dbias ------------------------------------------------------------------

@pytest.mark.parametrize("N", [96, 160, 512])
def test_grouped_dbias(oracle_mod, N):
    sizes = np.array([64, 0, 32, 416, 0, 0, 128, 96, 160, 32], np.int64)
    off = wl.offsets_from_sizes(sizes)
    x_bits = wl.moe_bf16(sizes, N, seed=N + 1)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mx.quantize_grouped(dev_bf16(x_bits), torch.from_numpy(off).cuda(), E5M2, err_flag=err, with_dbias=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    o = oracle_mod.quantize_grouped(x_bits, off, E5M2)
    for name, g, w in zip(("out_row", "scale_row", "out_col", "scale_col"), r[:4], o):
        assert_bytes_equal(g.cpu().numpy(), w, name)
    want = oracle_mod.grouped_dbias(x_bits, off)
    xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().abs().numpy()
    got = r.dbias.cpu().numpy()
    for g in range(len(sizes)):
        tol = 1e-5 * xv[off[g]:off[g + 1]].sum(0)
        assert np.all(np.abs(got[g].astype(np.float64) - want[g]) <= tol), g
    assert np.all(got[1] == 0.0) and np.all(got[4] == 0.0)


@pytest.mark.parametrize("case", ["512_groups", "512_unaligned_groups", "one_group", "long_and_empty"])
def test_grouped_dbias_group_layouts(oracle_mod, case):
    """Per-group sums across the reduce's 16 contiguous tile ranges: many small groups, one group
    spanning every range, and long groups between empty ones, with N not a multiple of 32."""
    rng = np.random.Generator(np.random.PCG64(len(case)))
    if case == "512_groups":
        sizes, N = 32 * rng.choice([0, 1, 3, 4, 5, 17], size=512), 48
    elif case == "512_unaligned_groups":
        sizes, N = rng.choice([0, 1, 7, 31, 33, 100, 129, 600], size=512), 48
    elif case == "one_group":
        sizes, N = np.array([8192], np.int64), 80
    else:
        sizes, N = np.array([0, 2080, 0, 0, 32, 4096, 0, 1024, 0], np.int64), 112
    sizes = sizes.astype(np.int64)
    off = wl.offsets_from_sizes(sizes)
    x_bits = wl.moe_bf16(sizes, N, seed=7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    r = mx.quantize_grouped(dev_bf16(x_bits), torch.from_numpy(off).cuda(), E4M3, err_flag=err, with_dbias=True)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    want = oracle_mod.grouped_dbias(x_bits, off)
    xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).double().abs().numpy()
    got = r.dbias.cpu().numpy().astype(np.float64)
    for g in range(len(sizes)):
        tol = 1e-5 * xv[off[g]:off[g + 1]].sum(0)
        assert np.all(np.abs(got[g] - want[g]) <= tol), g
        if sizes[g] == 0:
            assert np.all(got[g] == 0.0), g
    if case == "512_unaligned_groups":
        for name, gq, w in zip(("out_row", "scale_row", "out_col", "scale_col"), r[:4],
                               oracle_mod.quantize_grouped(x_bits, off, E4M3)):
            assert_bytes_equal(gq.cpu().numpy(), w, name)


def test_grouped_dbias_bad_offsets_write_nothing():
    x = dev_bf16(wl.normal_bf16(928, 96, seed=1))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    off = torch.tensor([0, 929, 928], dtype=torch.int64, device="cuda")   # decreasing
    dbias = torch.full((2, 96), 3.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(mx.mxfp8_quantize_grouped_dbias_workspace_bytes(928, 96, 2), dtype=torch.uint8, device="cuda")
    u8 = dict(dtype=torch.uint8, device="cuda")
    outs = [torch.full((928, 96), 0x3C, **u8), torch.full((928, 3), 0x3C, **u8),
            torch.full((928, 96), 0x3C, **u8), torch.full((29, 96), 0x3C, **u8)]
    st = mx.mxfp8_quantize_grouped_dbias(x, 928, 96, 2, off, E4M3, *outs, dbias, ws, None, err, None)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 1
    assert bool((dbias == 3.0).all()) and all(bool((t == 0x3C).all()) for t in outs)


def test_parity_moe_64x65536x7168_unaligned_full(oracle_mod):
    """The MoE workload's shape with ragged token counts that are not multiples of 32 (Zipf split
    of single rows): every byte against the oracle, per-group dbias within 1e-5 * sum|x|."""
    sizes = wl.moe_group_sizes(64, 65536, seed=9, unit=1)
    assert np.any(sizes % 32 != 0)
    off = wl.offsets_from_sizes(sizes)
    x_bits = wl.moe_bf16(sizes, 7168, seed=9)
    r = mx.quantize_grouped(dev_bf16(x_bits), torch.from_numpy(off).cuda(), E4M3, with_dbias=True,
                            scale_col_rows=mx.grouped_scale_col_rows(off))
    torch.cuda.synchronize()
    want_q = oracle_slices.quantize_grouped(oracle_mod, x_bits, off, E4M3)
    check_whole([t.cpu().numpy() for t in r[:4]], want_q)
    want = oracle_slices.grouped_dbias(oracle_mod, x_bits, off)
    got = r.dbias.cpu().numpy().astype(np.float64)
    xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).float().abs()
    for g in range(len(off) - 1):
        tol = 1e-5 * xv[off[g]:off[g + 1]].double().sum(0).numpy()
        assert np.all(np.abs(got[g] - want[g]) <= tol), g
    del r
    torch.cuda.empty_cache()


def test_parity_moe_64x65536x7168_unaligned_swizzled_full(oracle_mod):
    """The ragged MoE shape with one GEMM-ready plane pair per expert: every code against the
    oracle's grouped call, and each expert's slice of both concatenated planes against the
    oracle's swizzle of that expert's own scales (padding zero); expert g's planes follow the
    sum_{h<g} ceil(rows_h/128) tile rows of the experts before it."""
    sizes = wl.moe_group_sizes(64, 65536, seed=11, unit=1)
    off = wl.offsets_from_sizes(sizes)
    N = 7168
    x_bits = wl.moe_bf16(sizes, N, seed=11)
    r = mx.quantize_grouped(dev_bf16(x_bits), torch.from_numpy(off).cuda(), E4M3, swizzled=True)
    torch.cuda.synchronize()
    got = [t.cpu().numpy() for t in r[:4]]
    want = oracle_slices.quantize_grouped(oracle_mod, x_bits, off, E4M3)
    assert np.array_equal(got[0], want[0]) and np.array_equal(got[2], want[2])
    Cn, rb, cb, s0 = -(-N // 32), 0, 0, 0
    for g in range(len(off) - 1):
        rows = int(off[g + 1] - off[g])
        if rows == 0:
            continue
        srow = oracle_mod.swizzle_scales(want[1][off[g]:off[g + 1]])
        sc = -(-rows // 32)
        scol = oracle_mod.swizzle_scales(np.ascontiguousarray(want[3][s0:s0 + sc].T))
        assert np.array_equal(got[1][rb:rb + srow.size], srow), g
        assert np.array_equal(got[3][cb:cb + scol.size], scol), g
        rb, cb, s0 = rb + srow.size, cb + scol.size, s0 + sc
    assert rb == got[1].size and cb == got[3].size
    del r
    torch.cuda.empty_cache()


def test_grouped_dbias_moe_64x65536x7168_full(oracle_mod):
    w = wl.make("moe_64x65536x7168")
    x_bits, off = w["x"], w["offsets"]
    r = mx.quantize_grouped(dev_bf16(x_bits), torch.from_numpy(off).cuda(), E4M3, with_dbias=True)
    torch.cuda.synchronize()
    want = oracle_slices.grouped_dbias(oracle_mod, x_bits, off)
    got = r.dbias.cpu().numpy().astype(np.float64)
    xv = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).float().abs()
    for g in range(len(off) - 1):
        tol = 1e-5 * xv[off[g]:off[g + 1]].double().sum(0).numpy()
        assert np.all(np.abs(got[g] - want[g]) <= tol), g
    want_q = oracle_slices.quantize_grouped(oracle_mod, x_bits, off, E4M3)
    check_whole([t.cpu().numpy() for t in r[:4]], want_q)
    del r
    torch.cuda.empty_cache()
