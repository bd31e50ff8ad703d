"""Host-side checks of the C ABI; no GPU needed (no compute calls are made).

Every rejection below is decided on the host before the library touches the
device, so these run on a machine without a GPU.
"""
import ctypes
import os
import re

import pytest

import mxfp8_block_scaled_04_gb300 as mx

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mxfp8.h")

OK, NULL, SHAPE, ALIGN, FORMAT, WORKSPACE, DEVICE, LAUNCH, GROUPS = range(9)
A = 1 << 20     # a fake, 16-byte aligned address: never dereferenced by these calls


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\s*\*?\s*(mxfp8_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("mxfp8_quantize", "mxfp8_quantize_grouped", "mxfp8_quantize_workspace_bytes",
              "mxfp8_quantize_grouped_workspace_bytes", "mxfp8_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(cuda_lib):
    for name in declared_functions():
        assert hasattr(cuda_lib, name), name
        assert ctypes.cast(getattr(cuda_lib, name), ctypes.c_void_p).value


def test_status_strings(cuda_lib):
    for s in range(9):
        assert mx.mxfp8_status_string(s)
    assert mx.mxfp8_status_string(99) == "unknown status"


def test_workspace_bytes(cuda_lib):
    assert mx.mxfp8_quantize_workspace_bytes(16384, 8192, False) == 0
    assert mx.mxfp8_quantize_workspace_bytes(16384, 8192, True) == 128 * 8192 * 4
    assert mx.mxfp8_quantize_workspace_bytes(96, 64, True) == 1 * 64 * 4
    assert mx.mxfp8_quantize_workspace_bytes(160, 64, True) == 2 * 64 * 4
    assert mx.mxfp8_quantize_workspace_bytes(100, 64, True) == 1 * 64 * 4  # any M
    assert mx.mxfp8_quantize_workspace_bytes(100, 72, True) == 1 * 72 * 4     # N a multiple of 8
    assert mx.mxfp8_quantize_workspace_bytes(100, 68, True) == 0          # N not a multiple of 8
    assert mx.mxfp8_quantize_grouped_workspace_bytes(65536, 7168, 64) == 0


def q(x=A, M=64, N=64, fmt=0, orow=A, srow=A, ocol=A, scol=A, dbias=None, ws=None, noop=None):
    return mx.mxfp8_quantize(x, M, N, fmt, orow, srow, ocol, scol, dbias, ws, noop, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=2), FORMAT), (dict(fmt=-1), FORMAT),
    (dict(N=100), SHAPE), (dict(N=36), SHAPE), (dict(N=4), SHAPE), (dict(M=-32), SHAPE), (dict(N=1 << 31), SHAPE),
    (dict(x=None), NULL), (dict(orow=None), NULL), (dict(scol=None), NULL),
    (dict(orow=None, srow=None, ocol=None, scol=None), NULL),
    (dict(x=A + 8), ALIGN), (dict(orow=A + 4), ALIGN), (dict(ocol=A + 8), ALIGN), (dict(scol=A + 2), ALIGN),
    (dict(dbias=A + 2, ws=A), ALIGN), (dict(dbias=A, ws=A + 4), ALIGN),
    (dict(dbias=A), WORKSPACE),
])
def test_quantize_rejections(cuda_lib, kw, status):
    assert q(**kw) == status


def test_scale_row_needs_no_alignment_and_unaligned_pair_checks_pass_host_stage(cuda_lib):
    # scale_row is written byte by byte: any address passes the host checks, so
    # the call proceeds to the device stage, which fails without a usable GPU
    # (or with a fake pointer) and reports MXFP8_ERR_DEVICE.
    assert q(srow=A + 1) == DEVICE


def g(x=A, total=128, N=64, G=2, off=A, fmt=0, orow=A, srow=A, ocol=A, scol=A, err=None):
    return mx.mxfp8_quantize_grouped(x, total, N, G, off, fmt, orow, srow, ocol, scol, None, None, err, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=3), FORMAT), (dict(total=-32), SHAPE), (dict(N=36), SHAPE), (dict(total=1 << 31), SHAPE),
    (dict(G=0), GROUPS), (dict(G=mx.MAX_GROUPS + 1), GROUPS), (dict(off=None), GROUPS),
    (dict(x=None), NULL), (dict(orow=None), NULL), (dict(orow=None, srow=None, ocol=None, scol=None), NULL),
    (dict(x=A + 2), ALIGN), (dict(off=A + 4), ALIGN), (dict(err=A + 2), ALIGN),
])
def test_grouped_rejections(cuda_lib, kw, status):
    assert g(**kw) == status


def test_grouped_any_row_count_passes_host_checks(cuda_lib):
    # offsets are read only on the device, so total_rows that is not a multiple of 32 goes on to
    # the device stage (which fails here without a usable GPU)
    assert g(total=45) == DEVICE and g(total=1) == DEVICE and g(total=0) == DEVICE


def test_grouped_scale_col_rows():
    assert mx.grouped_scale_col_rows([0, 45, 45, 46, 192]) == 2 + 0 + 1 + 5
    assert mx.grouped_scale_col_rows([0, 64, 96, 512]) == 512 // 32
    assert mx.grouped_scale_col_rows([0, 0]) == 0


def test_binding_wrappers_reject_bad_tensors(cuda_lib):
    import torch
    with pytest.raises(ValueError):
        mx.quantize(torch.zeros(64, 64, dtype=torch.float32))
    with pytest.raises(ValueError):
        mx.quantize(torch.zeros(64, 64, dtype=torch.bfloat16).t())


def h(x=A, M=64, N=64, fmt=0, orow=A, srow=A, ocol=A, scol=A, dbias=None, staging=A, nbytes=1 << 30):
    return mx.mxfp8_quantize_host(x, M, N, fmt, orow, srow, ocol, scol, dbias, staging, nbytes, 0)


@pytest.mark.parametrize("kw,status", [
    (dict(fmt=5), FORMAT), (dict(M=0), SHAPE), (dict(N=36), SHAPE),
    (dict(x=None), NULL), (dict(staging=None), NULL), (dict(orow=None), NULL),
    (dict(orow=None, srow=None, ocol=None, scol=None), NULL),
    (dict(staging=A + 16), ALIGN), (dict(nbytes=1024), WORKSPACE),
])
def test_host_pipeline_rejections(cuda_lib, kw, status):
    assert h(**kw) == status


def test_host_staging_bytes(cuda_lib):
    # 8192 x 28672: chunks of at most 512 rows (32 MiB of BF16 rounded down to 128 rows),
    # three slots of 512 * 28672 * (2 + 1 + 1) bytes plus both scale planes
    per_slot = 512 * 28672 * 2 + 2 * 512 * 28672 + 512 * 28672 // 32 + 16 * 28672
    assert mx.mxfp8_quantize_host_staging_bytes(8192, 28672, False) == 3 * per_slot
    with_db = mx.mxfp8_quantize_host_staging_bytes(8192, 28672, True)
    assert with_db == 3 * per_slot + 64 * 28672 * 4 + 28672 * 4
    assert mx.mxfp8_quantize_host_staging_bytes(0, 64, False) == 0


def test_config_struct_layout_matches_the_c_header(tmp_path):
    # compile a probe against include/mxfp8.h and compare sizeof/offsetof with the ctypes mirror
    import subprocess
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mxfp8.h"\n'
                   '#define F(f) printf(" %zu", offsetof(mxfp8_quantize_config_t, f));\n'
                   'int main(void){ printf("%zu", sizeof(mxfp8_quantize_config_t));\n'
                   'F(x) F(M) F(N) F(fp8_fmt) F(out_row) F(scale_row) F(out_col) F(scale_col) F(dbias) F(workspace)'
                   ' F(noop) F(scale_layout) F(amax) F(activation) F(reserved) return 0; }\n')
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-I", os.path.dirname(HEADER), str(src), "-o", str(exe)], check=True)
    c_vals = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    C = mx.QuantizeConfig
    py_vals = [ctypes.sizeof(C)] + [getattr(C, f).offset for f, _ in C._fields_]
    assert c_vals == py_vals


def test_scale_bytes(cuda_lib):
    assert mx.mxfp8_scale_bytes(8192, 896, mx.SCALES_PLAIN) == 8192 * 896
    assert mx.mxfp8_scale_bytes(8192, 896, mx.SCALES_SWIZZLED) == 8192 * 896
    assert mx.mxfp8_scale_bytes(96, 5, mx.SCALES_SWIZZLED) == 128 * 8
    assert mx.mxfp8_scale_bytes(96, 5, 7) == 0


def test_ex_rejections(cuda_lib):
    assert mx.mxfp8_quantize_ex(None, 0) == NULL
    cfg = mx.make_config(A, 64, 64, 0, A, A, A, A, scale_layout=2)
    assert mx.mxfp8_quantize_ex(cfg, 0) == FORMAT
    cfg = mx.make_config(A, 64, 64, 0, A, A, A, A, scale_layout=1)
    cfg.reserved[3] = 1
    assert mx.mxfp8_quantize_ex(cfg, 0) == FORMAT
    assert mx.mxfp8_quantize_ex(mx.make_config(A, 64, 36, 0, A, A, A, A, scale_layout=1), 0) == SHAPE
    assert mx.mxfp8_quantize_ex(mx.make_config(A, 64, 64, 0, None, A, A, A, scale_layout=1), 0) == NULL
    assert mx.mxfp8_quantize_ex(mx.make_config(A, 64, 64, 0, A, A, A, A, scale_layout=1, amax=A + 2), 0) == ALIGN
    assert mx.mxfp8_quantize_ex(mx.make_config(A, 64, 64, 0, A, A, A, A, activation=6), 0) == FORMAT
    assert mx.mxfp8_quantize_ex(mx.make_config(A, 64, 64, 0, A, A, A, A, dbias=A, workspace=A,
                                               activation="gelu"), 0) == FORMAT
    # swizzled scale planes need no alignment: an odd scale pointer reaches the device stage
    assert mx.mxfp8_quantize_ex(mx.make_config(A, 64, 64, 0, A, A + 1, A, A + 1, scale_layout=1), 0) == DEVICE


def test_ragged_shapes_pass_host_checks(cuda_lib):
    # M not a multiple of 32 and N a multiple of 8 are valid shapes: with fake
    # pointers the call gets past every host check and stops at the device stage
    assert q(M=45, N=80) == DEVICE
    assert q(M=1, N=16) == DEVICE
    assert q(M=33, N=8) == DEVICE
    assert q(M=7, N=40) == DEVICE


def test_grouped_dbias_host_checks(cuda_lib):
    def gd(dbias=A, ws=A, **kw):
        args = dict(x=A, total=128, N=64, G=2, off=A, fmt=0)
        args.update(kw)
        return mx.mxfp8_quantize_grouped_dbias(args["x"], args["total"], args["N"], args["G"], args["off"],
                                               args["fmt"], A, A, A, A, dbias, ws, None, None, 0)
    assert gd(dbias=None) == NULL
    assert gd(ws=None) == WORKSPACE
    assert gd(total=-1) == SHAPE
    assert gd(total=40) == DEVICE      # any row count passes the host checks (groups may be unaligned)
    assert gd(G=0) == GROUPS
    assert gd(dbias=A + 2) == ALIGN
    assert gd() == DEVICE
    assert mx.mxfp8_quantize_grouped_dbias_workspace_bytes(65536, 7168, 64) == 768 + (512 + 64) * 7168 * 4
    assert mx.mxfp8_quantize_grouped_dbias_workspace_bytes(65536, 7168, 0) == 0


def test_dact_host_checks(cuda_lib):
    def d(**kw):
        a = dict(g=A, x=A, M=64, N=64, fmt=0, act=3, dbias=None, ws=None)
        a.update(kw)
        return mx.mxfp8_quantize_dact(a["g"], a["x"], a["M"], a["N"], a["fmt"], a["act"], A, A, A, A,
                                      a["dbias"], a["ws"], None, 0)
    assert d(act=0) == FORMAT and d(act=6) == FORMAT and d(fmt=2) == FORMAT
    assert d(N=36) == SHAPE
    assert d(x=None) == NULL and d(g=None) == NULL
    assert d(x=A + 8) == ALIGN
    assert d(dbias=A) == WORKSPACE
    assert d() == DEVICE


def test_gated_host_checks(cuda_lib):
    def gt(**kw):
        a = dict(x=A, M=64, N=64, fmt=0, act=4, orow=A, srow=A, ocol=A, scol=A)
        a.update(kw)
        return mx.mxfp8_quantize_gated(a["x"], a["M"], a["N"], a["fmt"], a["act"], a["orow"], a["srow"],
                                       a["ocol"], a["scol"], None, 0)
    assert gt(act=0) == FORMAT and gt(act=6) == FORMAT and gt(fmt=2) == FORMAT
    assert gt(N=36) == SHAPE and gt(M=-1) == SHAPE and gt(N=1 << 30) == SHAPE
    assert gt(x=None) == NULL and gt(orow=None) == NULL and gt(orow=None, srow=None, ocol=None, scol=None) == NULL
    assert gt(x=A + 8) == ALIGN and gt(ocol=A + 8) == ALIGN
    assert gt() == DEVICE and gt(N=40) == DEVICE      # N a multiple of 8: b starts 16-byte aligned
    import torch
    with pytest.raises(ValueError):
        mx.quantize_gated(torch.zeros(4, 6, dtype=torch.bfloat16)[:, :5].contiguous())


def test_grouped_activated_host_checks(cuda_lib):
    def ga(**kw):
        a = dict(x=A, total=128, N=64, G=2, off=A, fmt=0, act=3)
        a.update(kw)
        return mx.mxfp8_quantize_grouped_activated(a["x"], a["total"], a["N"], a["G"], a["off"], a["fmt"], a["act"],
                                                   A, A, A, A, None, None, 0)
    assert ga(act=0) == FORMAT and ga(act=6) == FORMAT and ga(fmt=2) == FORMAT
    assert ga(N=36) == SHAPE and ga(G=0) == GROUPS and ga(x=None) == NULL and ga(x=A + 8) == ALIGN
    assert ga() == DEVICE and ga(total=45) == DEVICE


def test_grouped_swizzled_host_checks(cuda_lib):
    def gs(**kw):
        a = dict(x=A, total=128, N=64, G=2, off=A, fmt=0, act=0, srow=A, scol=A)
        a.update(kw)
        return mx.mxfp8_quantize_grouped_swizzled(a["x"], a["total"], a["N"], a["G"], a["off"], a["fmt"], a["act"],
                                                  A, a["srow"], A, a["scol"], None, None, 0)
    assert gs(act=6) == FORMAT and gs(act=-1) == FORMAT and gs(fmt=2) == FORMAT
    assert gs(N=36) == SHAPE and gs(G=0) == GROUPS and gs(off=None) == GROUPS
    assert gs(x=None) == NULL and gs(x=A + 8) == ALIGN
    assert gs() == DEVICE and gs(total=45) == DEVICE and gs(act=3) == DEVICE
    # plane sizes: ceil(rows_g / 128) tiles per group, 128 x ceil(ceil(N/32)/4)*4 (rowwise) or
    # ceil(N/128)*128 x 4 (columnwise) bytes per tile
    assert mx.mxfp8_grouped_swizzled_scale_bytes([0, 45, 45, 300], 96, False) == 3 * 128 * 4
    assert mx.mxfp8_grouped_swizzled_scale_bytes([0, 45, 45, 300], 96, True) == 3 * 128 * 4
    assert mx.mxfp8_grouped_swizzled_scale_bytes([0, 129], 1032, False) == 2 * 128 * 36
    assert mx.mxfp8_grouped_swizzled_scale_bytes([0, 129], 1032, True) == 2 * 1152 * 4
    assert mx.mxfp8_grouped_swizzled_scale_bytes([0, 50, 40], 64, False) == 0      # decreasing
    assert mx.mxfp8_grouped_swizzled_scale_bytes([1, 50], 64, False) == 0          # not starting at 0
    assert mx.mxfp8_grouped_swizzled_scale_bytes([0, 50], 36, False) == 0          # N % 8


def test_gated_grouped_host_checks(cuda_lib):
    def gg(**kw):
        a = dict(x=A, total=128, N=64, G=2, off=A, fmt=0, act=4, orow=A, srow=A, ocol=A, scol=A, err=None)
        a.update(kw)
        return mx.mxfp8_quantize_gated_grouped(a["x"], a["total"], a["N"], a["G"], a["off"], a["fmt"], a["act"],
                                               a["orow"], a["srow"], a["ocol"], a["scol"], None, a["err"], 0)
    assert gg(fmt=3) == FORMAT and gg(act=0) == FORMAT
    assert gg(N=36) == SHAPE and gg(total=-1) == SHAPE
    assert gg(G=0) == GROUPS and gg(G=mx.MAX_GROUPS + 1) == GROUPS and gg(off=None) == GROUPS
    assert gg(x=None) == NULL and gg(orow=None) == NULL
    assert gg(x=A + 8) == ALIGN and gg(off=A + 4) == ALIGN and gg(err=A + 2) == ALIGN
    assert gg() == DEVICE and gg(total=45) == DEVICE


def test_dgated_host_checks(cuda_lib):
    def dg(**kw):
        a = dict(g=A, x=A, M=64, N=64, fmt=1, act=4, orow=A, srow=A, ocol=A, scol=A)
        a.update(kw)
        return mx.mxfp8_quantize_dgated(a["g"], a["x"], a["M"], a["N"], a["fmt"], a["act"], a["orow"], a["srow"],
                                        a["ocol"], a["scol"], None, 0)
    assert dg(act=0) == FORMAT and dg(act=6) == FORMAT and dg(fmt=2) == FORMAT
    assert dg(N=36) == SHAPE and dg(M=-1) == SHAPE and dg(N=1 << 30) == SHAPE
    assert dg(g=None) == NULL and dg(x=None) == NULL and dg(scol=None) == NULL
    assert dg(g=A + 8) == ALIGN and dg(x=A + 8) == ALIGN and dg(orow=A + 8) == ALIGN
    assert dg() == DEVICE and dg(N=40) == DEVICE
    import torch
    with pytest.raises(ValueError):
        mx.quantize_dgated(torch.zeros(4, 8, dtype=torch.bfloat16), torch.zeros(4, 8, dtype=torch.bfloat16))


def test_selftest_bounded_wait_rejections(cuda_lib):
    assert mx.mxfp8_selftest_bounded_wait(1_000_000, None) == NULL
    assert mx.mxfp8_selftest_bounded_wait(0, A) == SHAPE
    assert mx.mxfp8_selftest_bounded_wait(-5, A) == SHAPE
    assert mx.mxfp8_selftest_bounded_wait(10_000_000_001, A) == SHAPE


def test_noalloc_status_order_matches_quantize(cuda_lib):
    """The no-allocation call reports a bad format before a NULL dbias or an oversized shape, and
    the generic shape rules before its own scratch limit, as mxfp8_quantize orders its checks."""
    from mxfp8_block_scaled_04_gb300 import binding
    A = 1 << 20
    assert binding.mxfp8_quantize_dbias_noalloc(A, 64, 64, 7, A, A, A, A, None, None, None) == 4        # FORMAT
    assert binding.mxfp8_quantize_dbias_noalloc(A, 32768, 16384, 7, A, A, A, A, A, None, None) == 4     # FORMAT
    assert binding.mxfp8_quantize_dbias_noalloc(A, 64, 20, 0, A, A, A, A, None, None, None) == 2        # SHAPE
    assert binding.mxfp8_quantize_dbias_noalloc(A, 1 << 31, 64, 0, A, A, A, A, A, None, None) == 2      # SHAPE
    assert binding.mxfp8_quantize_dbias_noalloc(A, 64, 64, 0, A, A, A, A, None, None, None) == 1        # NULL dbias
    assert binding.mxfp8_quantize_dbias_noalloc(A, 32768, 16384, 0, A, A, A, A, A, None, None) == 2     # beyond 8 MiB


def test_grouped_host_rejections(cuda_lib):
    import torch
    good = torch.tensor([0, 45, 45, 128], dtype=torch.int64)

    def gh(x=A, total=128, N=64, off=good, G=3, fmt=0, act=0, orow=A, srow=A, ocol=A, scol=A, staging=A,
           nbytes=1 << 30):
        return mx.mxfp8_quantize_grouped_host(x, total, N, G, off, fmt, act, orow, srow, ocol, scol, staging,
                                              nbytes, 0)
    assert gh(fmt=2) == FORMAT and gh(act=6) == FORMAT and gh(act=-1) == FORMAT
    assert gh(total=0) == SHAPE and gh(N=36) == SHAPE
    assert gh(G=0) == GROUPS and gh(off=None) == GROUPS and gh(G=mx.MAX_GROUPS + 1) == GROUPS
    # the offsets are read on the host: a bad vector is rejected before any device work
    assert gh(off=torch.tensor([0, 50, 40, 128])) == GROUPS
    assert gh(off=torch.tensor([1, 50, 60, 128])) == GROUPS
    assert gh(off=torch.tensor([0, 50, 60, 127])) == GROUPS
    assert gh(x=None) == NULL and gh(staging=None) == NULL and gh(orow=None) == NULL
    assert gh(orow=None, srow=None, ocol=None, scol=None) == NULL
    assert gh(staging=A + 16) == ALIGN and gh(nbytes=1024) == WORKSPACE
    assert gh() == DEVICE and gh(act=3) == DEVICE and gh(orow=None, srow=None) == DEVICE


def _plan_checks(off, total, N):
    b = mx.mxfp8_grouped_host_chunks(off, total, N)
    R = max(128, (32 << 20) // (2 * N) // 128 * 128)
    assert b[0] == 0 and b[-1] == total and all(x < y for x, y in zip(b, b[1:]))
    for x in b[1:-1]:
        g = max(i for i in range(len(off) - 1) if off[i] <= x < off[i + 1])
        assert (x - off[g]) % 32 == 0                     # a cut group keeps its own 32-row blocks
    assert all(y - x <= R + 31 for x, y in zip(b, b[1:]))  # fits a staging slot of R + 32 rows
    # the pieces' columnwise scale rows add up to the group's: sum_g ceil(rows_g / 32)
    pieces = 0
    for x, y in zip(b, b[1:]):
        for g in range(len(off) - 1):
            a, e = min(max(off[g], x), y), min(max(off[g + 1], x), y)
            pieces += -(-(e - a) // 32)
    assert pieces == mx.grouped_scale_col_rows(off)
    return b


@pytest.mark.parametrize("seed", range(6))
def test_grouped_host_chunk_plan(cuda_lib, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    N = int(rng.choice([64, 1032, 7168, 16384]))
    G = int(rng.integers(1, 200))
    sizes = rng.integers(0, 3000, G)
    sizes[rng.random(G) < 0.2] = 0
    sizes[0] += 1
    off = [0] + np.cumsum(sizes).tolist()
    b = _plan_checks(off, off[-1], N)
    assert len(b) >= 2


def test_grouped_host_chunk_plan_edges(cuda_lib):
    _plan_checks([0, 1], 1, 64)                              # one row
    _plan_checks([0, 100000], 100000, 7168)                  # one group cut many times
    _plan_checks([0, 45, 45, 3000, 3001, 9000, 16384], 16384, 7168)
    _plan_checks([0] + [37 * i for i in range(1, 513)], 37 * 512, 4096)   # 512 groups, none 32-aligned
    # rows wider than 128 KiB: chunks of 128 rows and no ramp at either end
    assert _plan_checks([0, 5000], 5000, 200000) == list(range(0, 5000, 128)) + [5000]
    _plan_checks([0, 45, 3000, 9000], 9000, 300000)
    _plan_checks([0, 128], 128, 300000)
    assert mx.lib().mxfp8_grouped_host_chunks(None, 1, 10, 64, None, 0) == -1
    with pytest.raises(ValueError):
        mx.mxfp8_grouped_host_chunks([0, 5, 3], 3, 64)


def test_ex_host_rejections(cuda_lib):
    def cfg(**kw):
        a = dict(x=A, M=64, N=64, fmt=0, orow=A, srow=A, ocol=A, scol=A, dbias=None, ws=None, noop=None,
                 layout=mx.SCALES_SWIZZLED, amax=A, act=3)
        a.update(kw)
        return mx.make_config(a["x"], a["M"], a["N"], a["fmt"], a["orow"], a["srow"], a["ocol"], a["scol"],
                              a["dbias"], a["ws"], a["noop"], a["layout"], a["amax"], a["act"])

    def eh(staging=A, nbytes=1 << 30, **kw):
        return mx.mxfp8_quantize_ex_host(cfg(**kw), staging, nbytes, 0)
    assert mx.lib().mxfp8_quantize_ex_host(None, A, 1 << 30, None) == NULL
    c = cfg()
    c.reserved[2] = 1
    assert mx.mxfp8_quantize_ex_host(c, A, 1 << 30, 0) == FORMAT
    assert eh(layout=2) == FORMAT and eh(act=6) == FORMAT and eh(act=1, dbias=A) == FORMAT
    assert eh(ws=A) == FORMAT and eh(noop=A) == FORMAT          # no workspace or noop with host buffers
    assert eh(fmt=2) == FORMAT and eh(M=0) == SHAPE and eh(N=36) == SHAPE
    assert eh(x=None) == NULL and eh(staging=None) == NULL and eh(orow=None) == NULL
    assert eh(staging=A + 16) == ALIGN and eh(nbytes=1024) == WORKSPACE
    assert eh() == DEVICE and eh(act=0, amax=None) == DEVICE
    # staging: GEMM-ready slots are at least the plain ones; amax adds one 256-byte line
    plain = mx.mxfp8_quantize_ex_host_staging_bytes(cfg(layout=mx.SCALES_PLAIN, amax=None))
    assert plain == mx.mxfp8_quantize_host_staging_bytes(64, 64, 0)
    assert mx.mxfp8_quantize_ex_host_staging_bytes(cfg(layout=mx.SCALES_PLAIN)) == plain + 256
    assert mx.mxfp8_quantize_ex_host_staging_bytes(cfg(amax=None)) >= plain
    assert mx.mxfp8_quantize_ex_host_staging_bytes(None) == 0


@pytest.mark.parametrize("which", ["dact", "gated", "dgated"])
def test_two_input_host_rejections(cuda_lib, which):
    def call(inp=A, M=64, N=64, fmt=0, act=3, orow=A, srow=A, ocol=A, scol=A, staging=A, nbytes=1 << 30):
        if which == "dact":
            return mx.mxfp8_quantize_dact_host(inp, A, M, N, fmt, act, orow, srow, ocol, scol, None, staging,
                                               nbytes, 0)
        if which == "gated":
            return mx.mxfp8_quantize_gated_host(inp, M, N, fmt, act, orow, srow, ocol, scol, staging, nbytes, 0)
        return mx.mxfp8_quantize_dgated_host(inp, A, M, N, fmt, act, orow, srow, ocol, scol, staging, nbytes, 0)
    assert call(fmt=2) == FORMAT and call(act=0) == FORMAT and call(act=6) == FORMAT
    assert call(M=0) == SHAPE and call(N=36) == SHAPE
    assert call(inp=None) == NULL and call(staging=None) == NULL and call(orow=None) == NULL
    assert call(orow=None, srow=None, ocol=None, scol=None) == NULL
    assert call(staging=A + 16) == ALIGN and call(nbytes=1024) == WORKSPACE
    assert call() == DEVICE and call(ocol=None, scol=None) == DEVICE
    size = {"dact": lambda M, N: mx.mxfp8_quantize_dact_host_staging_bytes(M, N, False),
            "gated": mx.mxfp8_quantize_gated_host_staging_bytes,
            "dgated": mx.mxfp8_quantize_dgated_host_staging_bytes}[which]
    assert size(0, 64) == 0 and size(64, 36) == 0 and size(64, 64) > 0
    assert size(65536, 1024) > size(128, 1024)             # slots hold one chunk: at most ~32 MiB of input
