"""CPU oracle for MXFP8 block-scaled quantization (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it, and the two share no code.

The arithmetic lives in ``mxfp8_oracle.c`` (plain scalar C, exact double
evaluation); this module compiles it with gcc and wraps it with numpy arrays.
See the header of ``mxfp8_oracle.c`` for what each function computes and which
page passage it follows.  NaN/Inf inputs are outside the contract (parity
unpinned for them).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
BLOCK = 32

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u8, u16p, u8p = ctypes.c_uint8, ctypes.POINTER(ctypes.c_uint16), ctypes.POINTER(ctypes.c_uint8)
            i64, i64p, f32p = ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_float)
            lib.mxo_bf16_to_double.restype = ctypes.c_double
            lib.mxo_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.mxo_fp8_decode.restype = ctypes.c_double
            lib.mxo_fp8_decode.argtypes = [u8, ctypes.c_int]
            lib.mxo_fp8_encode.restype = u8
            lib.mxo_fp8_encode.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.mxo_fp8_max.restype = ctypes.c_double
            lib.mxo_fp8_max.argtypes = [ctypes.c_int]
            lib.mxo_block_exponent.restype = ctypes.c_int
            lib.mxo_block_exponent.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.mxo_e8m0_decode.restype = ctypes.c_double
            lib.mxo_e8m0_decode.argtypes = [u8]
            lib.mxo_quantize.restype = ctypes.c_int
            lib.mxo_quantize.argtypes = [u16p, i64, i64, ctypes.c_int, u8p, u8p, u8p, u8p, f32p]
            lib.mxo_quantize_grouped.restype = ctypes.c_int
            lib.mxo_quantize_grouped.argtypes = [u16p, i64, i64, ctypes.c_int, i64p, ctypes.c_int,
                                                 u8p, u8p, u8p, u8p]
            lib.mxo_swizzled_bytes.restype = i64
            lib.mxo_swizzled_bytes.argtypes = [i64, i64]
            lib.mxo_swizzle_offset.restype = i64
            lib.mxo_swizzle_offset.argtypes = [i64, i64, i64]
            lib.mxo_swizzle_scales.restype = None
            lib.mxo_swizzle_scales.argtypes = [u8p, i64, i64, u8p]
            lib.mxo_amax.restype = ctypes.c_float
            lib.mxo_amax.argtypes = [u16p, i64, i64]
            lib.mxo_grouped_dbias.restype = ctypes.c_int
            lib.mxo_grouped_dbias.argtypes = [u16p, i64, i64, ctypes.c_int, i64p, f32p]
            lib.mxo_dactivation_f64.restype = ctypes.c_double
            lib.mxo_dactivation_f64.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.mxo_dactivate.restype = None
            lib.mxo_dactivate.argtypes = [u16p, u16p, i64, ctypes.c_int, f32p]
            lib.mxo_activation_f64.restype = ctypes.c_double
            lib.mxo_activation_f64.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.mxo_activation.restype = ctypes.c_float
            lib.mxo_activation.argtypes = [ctypes.c_double, ctypes.c_int]
            lib.mxo_quantize_f32.restype = ctypes.c_int
            lib.mxo_quantize_f32.argtypes = [f32p, i64, i64, ctypes.c_int, u8p, u8p, u8p, u8p, f32p]
            lib.mxo_activate.restype = None
            lib.mxo_activate.argtypes = [u16p, i64, ctypes.c_int, f32p]
            lib.mxo_dgate.restype = None
            lib.mxo_dgate.argtypes = [u16p, u16p, i64, i64, ctypes.c_int, f32p, f32p]
            lib.mxo_gate.restype = None
            lib.mxo_gate.argtypes = [u16p, i64, i64, ctypes.c_int, f32p]
            _lib = lib
    return _lib


def _ptr(a, ctype):
    return None if a is None else a.ctypes.data_as(ctypes.POINTER(ctype))


# ---- scalar helpers ---------------------------------------------------------

def bf16_to_float(bits: int) -> float:
    return _load().mxo_bf16_to_double(int(bits) & 0xFFFF)


def fp8_decode(byte: int, fmt: int) -> float:
    return _load().mxo_fp8_decode(int(byte) & 0xFF, fmt)


def fp8_encode(v: float, fmt: int) -> int:
    return int(_load().mxo_fp8_encode(float(v), fmt))


def fp8_max(fmt: int) -> float:
    return _load().mxo_fp8_max(fmt)


def block_exponent(amax: float, fmt: int) -> int:
    return int(_load().mxo_block_exponent(float(amax), fmt))


def e8m0_decode(e: int) -> float:
    return _load().mxo_e8m0_decode(int(e) & 0xFF)


# ---- array entry points -------------------------------------------------------

def quantize(x_bits: np.ndarray, fmt: int, rowwise: bool = True, colwise: bool = True,
             with_dbias: bool = False):
    """Quantize BF16 bits ``x_bits`` (uint16 [M,N], row-major).

    Returns ``(out_row, scale_row, out_col, scale_col, dbias)``; entries for a
    direction that was not requested are None.  Shapes: out_* [M,N] uint8,
    scale_row [M,ceil(N/32)], scale_col [ceil(M/32),N] uint8, dbias [N] float32
    (a last, partial block takes its amax over the elements it has).
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N = x.shape
    out_row = np.empty((M, N), np.uint8) if rowwise else None
    scale_row = np.empty((M, -(-N // BLOCK)), np.uint8) if rowwise else None
    out_col = np.empty((M, N), np.uint8) if colwise else None
    scale_col = np.empty((-(-M // BLOCK), N), np.uint8) if colwise else None
    dbias = np.empty((N,), np.float32) if with_dbias else None
    rc = _load().mxo_quantize(_ptr(x, ctypes.c_uint16), M, N, fmt,
                              _ptr(out_row, ctypes.c_uint8), _ptr(scale_row, ctypes.c_uint8),
                              _ptr(out_col, ctypes.c_uint8), _ptr(scale_col, ctypes.c_uint8),
                              _ptr(dbias, ctypes.c_float))
    if rc != 0:
        raise ValueError(f"oracle: M={M}, N={N} must be non-negative")
    return out_row, scale_row, out_col, scale_col, dbias


def quantize_grouped(x_bits: np.ndarray, offsets: np.ndarray, fmt: int):
    """Grouped quantize: rows [offsets[g], offsets[g+1]) are group g, each its own flat problem.

    Returns ``(out_row, scale_row, out_col, scale_col)``: the row-indexed outputs at
    each group's rows; ``scale_col`` has ``grouped_scale_col_rows(offsets)`` rows, group
    g's ``ceil(rows_g/32)`` after those of the groups before it (with every offset a
    multiple of 32 this is the flat call's layout on the concatenated rows).  Raises
    ValueError on invalid offsets.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    total, N = x.shape
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    G = off.shape[0] - 1
    out_row = np.zeros((total, N), np.uint8)
    scale_row = np.zeros((total, -(-N // BLOCK)), np.uint8)
    out_col = np.zeros((total, N), np.uint8)
    scale_col = np.zeros((max(grouped_scale_col_rows(off), 0), N), np.uint8)
    rc = _load().mxo_quantize_grouped(_ptr(x, ctypes.c_uint16), total, N, G, _ptr(off, ctypes.c_int64), fmt,
                                      _ptr(out_row, ctypes.c_uint8), _ptr(scale_row, ctypes.c_uint8),
                                      _ptr(out_col, ctypes.c_uint8), _ptr(scale_col, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("oracle: invalid group offsets")
    return out_row, scale_row, out_col, scale_col


def grouped_scale_col_rows(offsets) -> int:
    """Rows of a grouped call's columnwise scale plane: sum over groups of ceil(rows_g / 32)."""
    off = np.asarray(offsets, dtype=np.int64)
    return int(np.sum(-(-np.diff(off) // BLOCK))) if off.size > 1 else 0


def swizzle_offset(r: int, c: int, C: int) -> int:
    """Byte offset of scale (r, c) of an R x C scale matrix in the GEMM-ready layout."""
    return int(_load().mxo_swizzle_offset(r, c, C))


def swizzle_scales(plain: np.ndarray) -> np.ndarray:
    """Plain scales [R, C] (uint8) -> GEMM-ready layout (1-D uint8, zero padded)."""
    p = np.ascontiguousarray(plain, dtype=np.uint8)
    R, C = p.shape
    out = np.empty(int(_load().mxo_swizzled_bytes(R, C)), np.uint8)
    _load().mxo_swizzle_scales(_ptr(p, ctypes.c_uint8), R, C, _ptr(out, ctypes.c_uint8))
    return out


def amax(x_bits: np.ndarray) -> float:
    """max |x| over a BF16 matrix (uint16 bits), as fp32."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N = x.shape
    return float(_load().mxo_amax(_ptr(x, ctypes.c_uint16), M, N))


ACT_NONE, ACT_RELU, ACT_SRELU, ACT_GELU, ACT_SILU, ACT_QGELU = range(6)


def activate(x_bits: np.ndarray, act: int) -> np.ndarray:
    """fp32 activation of a BF16 matrix (see mxo_activation for the formulas)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    y = np.empty(x.shape, np.float32)
    _load().mxo_activate(_ptr(x, ctypes.c_uint16), x.size, act, _ptr(y, ctypes.c_float))
    return y


def quantize_f32(y: np.ndarray, fmt: int, rowwise: bool = True, colwise: bool = True, with_dbias: bool = False):
    """Quantize fp32 values [M,N]; returns (out_row, scale_row, out_col, scale_col, dbias) as quantize()."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    M, N = y.shape
    out_row = np.empty((M, N), np.uint8) if rowwise else None
    scale_row = np.empty((M, -(-N // BLOCK)), np.uint8) if rowwise else None
    out_col = np.empty((M, N), np.uint8) if colwise else None
    scale_col = np.empty((-(-M // BLOCK), N), np.uint8) if colwise else None
    dbias = np.empty((N,), np.float32) if with_dbias else None
    rc = _load().mxo_quantize_f32(_ptr(y, ctypes.c_float), M, N, fmt, _ptr(out_row, ctypes.c_uint8),
                                  _ptr(scale_row, ctypes.c_uint8), _ptr(out_col, ctypes.c_uint8),
                                  _ptr(scale_col, ctypes.c_uint8), _ptr(dbias, ctypes.c_float))
    if rc != 0:
        raise ValueError("oracle: M, N must be non-negative")
    return out_row, scale_row, out_col, scale_col, dbias


def quantize_act(x_bits: np.ndarray, fmt: int, act: int, rowwise: bool = True, colwise: bool = True,
                 with_dbias: bool = False):
    """Activation in fp32, then the MXFP8 cast of the fp32 values."""
    return quantize_f32(activate(x_bits, act), fmt, rowwise, colwise, with_dbias)


def gate(x_bits: np.ndarray, act: int) -> np.ndarray:
    """fp32 act(a) * b of a BF16 matrix [M, 2N] with a = its first N columns, b = its last N (mxo_gate)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N2 = x.shape
    if N2 % 2:
        raise ValueError("oracle: a gated input has an even number of columns")
    y = np.empty((M, N2 // 2), np.float32)
    _load().mxo_gate(_ptr(x, ctypes.c_uint16), M, N2 // 2, act, _ptr(y, ctypes.c_float))
    return y


def quantize_gated(x_bits: np.ndarray, fmt: int, act: int, rowwise: bool = True, colwise: bool = True):
    """The MXFP8 cast of act(a) * b for a gated input [M, 2N] (no dbias)."""
    return quantize_f32(gate(x_bits, act), fmt, rowwise, colwise)[:4]


def _grouped_f32(y: np.ndarray, offsets, fmt: int):
    """quantize_f32 of each group's rows of y, laid out as quantize_grouped lays out its groups."""
    off = np.asarray(offsets, dtype=np.int64)
    total, N = y.shape
    if off.size < 2 or off[0] != 0 or off[-1] != total or np.any(np.diff(off) < 0):
        raise ValueError("oracle: invalid group offsets")
    out_row = np.zeros((total, N), np.uint8)
    scale_row = np.zeros((total, -(-N // BLOCK)), np.uint8)
    out_col = np.zeros((total, N), np.uint8)
    scale_col = np.zeros((grouped_scale_col_rows(off), N), np.uint8)
    s0 = 0
    for g in range(off.size - 1):
        a, b = int(off[g]), int(off[g + 1])
        if a == b:
            continue
        o_r, s_r, o_c, s_c, _ = quantize_f32(y[a:b], fmt)
        out_row[a:b], scale_row[a:b], out_col[a:b] = o_r, s_r, o_c
        scale_col[s0:s0 + s_c.shape[0]] = s_c
        s0 += s_c.shape[0]
    return out_row, scale_row, out_col, scale_col


def quantize_grouped_swizzled(x_bits: np.ndarray, offsets, fmt: int, act: int = 0):
    """The grouped cast (of act(x) when act != 0) with each group's scale planes in the GEMM-ready
    layout: group g's rowwise plane is swizzle_scales of its [rows_g, ceil(N/32)] scales, its
    columnwise plane swizzle_scales of the transposed [N, ceil(rows_g/32)] scales; the planes of the
    groups are concatenated in group order.  Returns (out_row, scale_row, out_col, scale_col)."""
    off = np.asarray(offsets, dtype=np.int64)
    y = activate(x_bits, act) if act else None
    if act:
        o_r, _, o_c, _ = _grouped_f32(y, off, fmt)
    else:
        o_r, _, o_c, _ = quantize_grouped(x_bits, off, fmt)
    rows_planes, col_planes = [], []
    for g in range(off.size - 1):
        a, b = int(off[g]), int(off[g + 1])
        if a == b:
            continue
        q = quantize_f32(y[a:b], fmt) if act else quantize(x_bits[a:b], fmt)
        rows_planes.append(swizzle_scales(q[1]))
        col_planes.append(swizzle_scales(np.ascontiguousarray(q[3].T)))
    cat = lambda ps: np.concatenate(ps) if ps else np.zeros(0, np.uint8)
    return o_r, cat(rows_planes), o_c, cat(col_planes)


def quantize_gated_grouped(x_bits: np.ndarray, offsets, fmt: int, act: int):
    """The gated cast over row groups, each group its own flat problem (as quantize_grouped):
    row-indexed outputs at the group's rows, the group's ceil(rows/32) columnwise scale rows after
    those of the groups before it.  ValueError for offsets quantize_grouped rejects."""
    if x_bits.shape[1] % 2:
        raise ValueError("oracle: a gated input has an even number of columns")
    off = np.asarray(offsets, dtype=np.int64)
    if off.size < 2 or off[-1] != x_bits.shape[0]:
        raise ValueError("oracle: invalid group offsets")
    return _grouped_f32(gate(x_bits, act), off, fmt)


def quantize_grouped_act(x_bits: np.ndarray, offsets, fmt: int, act: int):
    """The grouped cast of the fp32 activations act(x) (see activate), each group its own flat problem."""
    return _grouped_f32(activate(x_bits, act), offsets, fmt)


def dgate(g_bits: np.ndarray, x_bits: np.ndarray, act: int):
    """fp32 (da, db) = (g * b * act'(a), g * act(a)) for g [M, N] and x = [a | b] [M, 2N] (mxo_dgate)."""
    g = np.ascontiguousarray(g_bits, dtype=np.uint16)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, N = g.shape
    if x.shape != (M, 2 * N):
        raise ValueError("oracle: x must be [M, 2N] for a gradient g of [M, N]")
    da = np.empty((M, N), np.float32)
    db = np.empty((M, N), np.float32)
    _load().mxo_dgate(_ptr(g, ctypes.c_uint16), _ptr(x, ctypes.c_uint16), M, N, act,
                      _ptr(da, ctypes.c_float), _ptr(db, ctypes.c_float))
    return da, db


def quantize_dgated(g_bits: np.ndarray, x_bits: np.ndarray, fmt: int, act: int, rowwise: bool = True,
                    colwise: bool = True):
    """The MXFP8 cast of the gated input's gradient [da | db]: da and db are quantized as two
    [M, N] tensors and laid side by side, codes [M, 2N], scale_row [M, 2 ceil(N/32)] (da's
    blocks, then db's), scale_col [ceil(M/32), 2N]."""
    da, db = dgate(g_bits, x_bits, act)
    qa = quantize_f32(da, fmt, rowwise, colwise)
    qb = quantize_f32(db, fmt, rowwise, colwise)
    return tuple(None if u is None else np.ascontiguousarray(np.concatenate([u, v], axis=1))
                 for u, v in zip(qa[:4], qb[:4]))


def activation_f64(v: float, act: int) -> float:
    """Exact-as-double activation of one value (no fp32 rounding)."""
    return float(_load().mxo_activation_f64(float(v), act))


def grouped_dbias(x_bits: np.ndarray, offsets: np.ndarray) -> np.ndarray:
    """Per-group column sums [G, N] float32 of a grouped input; ValueError on invalid offsets."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    total, N = x.shape
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    G = off.shape[0] - 1
    out = np.empty((G, N), np.float32)
    if _load().mxo_grouped_dbias(_ptr(x, ctypes.c_uint16), total, N, G, _ptr(off, ctypes.c_int64),
                                 _ptr(out, ctypes.c_float)) != 0:
        raise ValueError("oracle: invalid group offsets")
    return out


def dactivation_f64(v: float, act: int) -> float:
    """Exact-as-double derivative act'(v) (see mxo_dactivation_f64)."""
    return float(_load().mxo_dactivation_f64(float(v), act))


def dactivate(dy_bits: np.ndarray, x_bits: np.ndarray, act: int) -> np.ndarray:
    """fp32 dY * act'(X) for BF16 matrices of equal shape."""
    dy = np.ascontiguousarray(dy_bits, dtype=np.uint16)
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert dy.shape == x.shape
    y = np.empty(x.shape, np.float32)
    _load().mxo_dactivate(_ptr(dy, ctypes.c_uint16), _ptr(x, ctypes.c_uint16), x.size, act, _ptr(y, ctypes.c_float))
    return y


def quantize_dact(dy_bits: np.ndarray, x_bits: np.ndarray, fmt: int, act: int, rowwise: bool = True,
                  colwise: bool = True, with_dbias: bool = False):
    """The MXFP8 cast of dY * act'(X) (and its column sums as dbias)."""
    return quantize_f32(dactivate(dy_bits, x_bits, act), fmt, rowwise, colwise, with_dbias)
