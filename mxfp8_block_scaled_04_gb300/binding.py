"""Python binding of the C ABI in include/mxfp8.h (ctypes; marshalling only).

The functions named ``mxfp8_*`` mirror the C entry points one for one: they
take torch tensors (or raw integer device addresses, or None for NULL) and
return the C status code.  ``quantize`` / ``quantize_grouped`` allocate the
outputs with torch and raise :class:`MXFP8Error` on a non-OK status.  Every
step of the computation runs in the CUDA library; there is no fallback, and
the first call fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Optional

import torch

E4M3 = 0
E5M2 = 1
BLOCK = 32
MAX_GROUPS = 512

STATUS_NAMES = {
    0: "MXFP8_OK", 1: "MXFP8_ERR_NULL", 2: "MXFP8_ERR_SHAPE", 3: "MXFP8_ERR_ALIGN",
    4: "MXFP8_ERR_FORMAT", 5: "MXFP8_ERR_WORKSPACE", 6: "MXFP8_ERR_DEVICE",
    7: "MXFP8_ERR_LAUNCH", 8: "MXFP8_ERR_GROUPS",
}

SCALES_PLAIN = 0
SCALES_SWIZZLED = 1
NOALLOC_SCRATCH_BYTES = 8 << 20   # MXFP8_NOALLOC_SCRATCH_BYTES in include/mxfp8.h


class QuantizeConfig(ctypes.Structure):
    """Mirror of mxfp8_quantize_config_t (include/mxfp8.h)."""
    _fields_ = [("x", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("fp8_fmt", ctypes.c_int),
                ("out_row", ctypes.c_void_p), ("scale_row", ctypes.c_void_p), ("out_col", ctypes.c_void_p),
                ("scale_col", ctypes.c_void_p), ("dbias", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("noop", ctypes.c_void_p), ("scale_layout", ctypes.c_int), ("amax", ctypes.c_void_p),
                ("activation", ctypes.c_int), ("reserved", ctypes.c_int * 5)]


ACTIVATIONS = {"none": 0, "relu": 1, "srelu": 2, "gelu": 3, "silu": 4, "qgelu": 5}


LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmxfp8.so")
_lock = threading.Lock()
_lib = None


class MXFP8Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({mxfp8_status_string(status)})")


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"MXFP8 CUDA library not found at {LIB_PATH}; build it with "
                    "`python -m mxfp8_block_scaled_04_gb300.build` (there is no CPU fallback)")
            L = ctypes.CDLL(LIB_PATH)
            vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
            L.mxfp8_quantize_workspace_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_workspace_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize.restype = i32
            L.mxfp8_quantize.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_grouped_workspace_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_grouped_workspace_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize_grouped.restype = i32
            L.mxfp8_quantize_grouped.argtypes = [vp, i64, i64, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_grouped_dbias_workspace_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_grouped_dbias_workspace_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize_grouped_dbias.restype = i32
            L.mxfp8_quantize_grouped_dbias.argtypes = [vp, i64, i64, i32, vp, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_dact.restype = i32
            L.mxfp8_quantize_dact.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_gated.restype = i32
            L.mxfp8_quantize_gated.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_grouped_activated.restype = i32
            L.mxfp8_quantize_grouped_activated.argtypes = [vp, i64, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp,
                                                           vp]
            L.mxfp8_quantize_grouped_swizzled.restype = i32
            L.mxfp8_quantize_grouped_swizzled.argtypes = [vp, i64, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
            L.mxfp8_grouped_swizzled_scale_bytes.restype = ctypes.c_size_t
            L.mxfp8_grouped_swizzled_scale_bytes.argtypes = [ctypes.POINTER(ctypes.c_int64), i32, i64, i32]
            L.mxfp8_quantize_gated_grouped.restype = i32
            L.mxfp8_quantize_gated_grouped.argtypes = [vp, i64, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_dgated.restype = i32
            L.mxfp8_quantize_dgated.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp]
            L.mxfp8_quantize_host_staging_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_host_staging_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize_host.restype = i32
            L.mxfp8_quantize_host.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
            L.mxfp8_quantize_dact_host_staging_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_dact_host_staging_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize_dact_host.restype = i32
            L.mxfp8_quantize_dact_host.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, vp,
                                                   ctypes.c_size_t, vp]
            L.mxfp8_quantize_gated_host_staging_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_gated_host_staging_bytes.argtypes = [i64, i64]
            L.mxfp8_quantize_gated_host.restype = i32
            L.mxfp8_quantize_gated_host.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
            L.mxfp8_quantize_dgated_host_staging_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_dgated_host_staging_bytes.argtypes = [i64, i64]
            L.mxfp8_quantize_dgated_host.restype = i32
            L.mxfp8_quantize_dgated_host.argtypes = [vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, vp,
                                                     ctypes.c_size_t, vp]
            L.mxfp8_quantize_ex_host_staging_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_ex_host_staging_bytes.argtypes = [ctypes.POINTER(QuantizeConfig)]
            L.mxfp8_quantize_ex_host.restype = i32
            L.mxfp8_quantize_ex_host.argtypes = [ctypes.POINTER(QuantizeConfig), vp, ctypes.c_size_t, vp]
            L.mxfp8_quantize_grouped_host_staging_bytes.restype = ctypes.c_size_t
            L.mxfp8_quantize_grouped_host_staging_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize_grouped_host.restype = i32
            L.mxfp8_quantize_grouped_host.argtypes = [vp, i64, i64, i32, vp, i32, i32, vp, vp, vp, vp, vp,
                                                      ctypes.c_size_t, vp]
            L.mxfp8_grouped_host_chunks.restype = i64
            L.mxfp8_grouped_host_chunks.argtypes = [vp, i32, i64, i64, vp, i64]
            L.mxfp8_scale_bytes.restype = ctypes.c_size_t
            L.mxfp8_scale_bytes.argtypes = [i64, i64, i32]
            L.mxfp8_quantize_ex.restype = i32
            L.mxfp8_quantize_ex.argtypes = [ctypes.POINTER(QuantizeConfig), vp]
            L.mxfp8_status_string.restype = ctypes.c_char_p
            L.mxfp8_status_string.argtypes = [i32]
            L.mxfp8_kernel_launch_count.restype = ctypes.c_uint64
            L.mxfp8_kernel_launch_count.argtypes = []
            L.mxfp8_device_fault_word.restype = i32
            L.mxfp8_device_fault_word.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
            L.mxfp8_selftest_bounded_wait.restype = i32
            L.mxfp8_selftest_bounded_wait.argtypes = [i64, vp, vp]
            L.mxfp8_activation_values.restype = i32
            L.mxfp8_activation_values.argtypes = [vp, i64, i32, i32, vp, vp]
            _lib = L
    return _lib


def _addr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        return a.data_ptr() if a.numel() > 0 or a.data_ptr() else None
    return int(a)


def _stream(s) -> Optional[int]:
    if s is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


# ---- one-for-one C entry points --------------------------------------------------

def mxfp8_quantize_workspace_bytes(M: int, N: int, with_dbias: bool) -> int:
    return int(lib().mxfp8_quantize_workspace_bytes(M, N, int(bool(with_dbias))))


def mxfp8_quantize(x, M, N, fp8_fmt, out_row, scale_row, out_col, scale_col,
                   dbias=None, workspace=None, noop=None, stream=None) -> int:
    return int(lib().mxfp8_quantize(_addr(x), M, N, fp8_fmt, _addr(out_row), _addr(scale_row),
                                    _addr(out_col), _addr(scale_col), _addr(dbias), _addr(workspace),
                                    _addr(noop), _stream(stream)))


def mxfp8_quantize_grouped_workspace_bytes(total_rows: int, N: int, num_groups: int) -> int:
    return int(lib().mxfp8_quantize_grouped_workspace_bytes(total_rows, N, num_groups))


def mxfp8_quantize_grouped(x, total_rows, N, num_groups, offsets, fp8_fmt, out_row, scale_row,
                           out_col, scale_col, workspace=None, noop=None, err_flag=None, stream=None) -> int:
    return int(lib().mxfp8_quantize_grouped(_addr(x), total_rows, N, num_groups, _addr(offsets), fp8_fmt,
                                            _addr(out_row), _addr(scale_row), _addr(out_col),
                                            _addr(scale_col), _addr(workspace), _addr(noop),
                                            _addr(err_flag), _stream(stream)))


def mxfp8_quantize_grouped_dbias_workspace_bytes(total_rows: int, N: int, num_groups: int) -> int:
    return int(lib().mxfp8_quantize_grouped_dbias_workspace_bytes(total_rows, N, num_groups))


def mxfp8_quantize_grouped_dbias(x, total_rows, N, num_groups, offsets, fp8_fmt, out_row, scale_row, out_col,
                                 scale_col, dbias, workspace, noop=None, err_flag=None, stream=None) -> int:
    return int(lib().mxfp8_quantize_grouped_dbias(_addr(x), total_rows, N, num_groups, _addr(offsets), fp8_fmt,
                                                  _addr(out_row), _addr(scale_row), _addr(out_col),
                                                  _addr(scale_col), _addr(dbias), _addr(workspace), _addr(noop),
                                                  _addr(err_flag), _stream(stream)))


def mxfp8_quantize_dact(grad, act_input, M, N, fp8_fmt, activation, out_row, scale_row, out_col, scale_col,
                        dbias=None, workspace=None, noop=None, stream=None) -> int:
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_dact(_addr(grad), _addr(act_input), M, N, fp8_fmt, int(activation),
                                         _addr(out_row), _addr(scale_row), _addr(out_col), _addr(scale_col),
                                         _addr(dbias), _addr(workspace), _addr(noop), _stream(stream)))


def mxfp8_quantize_gated(x, M, N, fp8_fmt, activation, out_row, scale_row, out_col, scale_col,
                         noop=None, stream=None) -> int:
    """The cast of act(a) * b for x = [a | b] (bf16 [M, 2N]); see include/mxfp8.h."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_gated(_addr(x), M, N, fp8_fmt, int(activation), _addr(out_row),
                                          _addr(scale_row), _addr(out_col), _addr(scale_col), _addr(noop),
                                          _stream(stream)))


def mxfp8_quantize_grouped_activated(x, total_rows, N, num_groups, offsets, fp8_fmt, activation, out_row,
                                     scale_row, out_col, scale_col, noop=None, err_flag=None, stream=None) -> int:
    """The grouped cast of act(x); see include/mxfp8.h."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_grouped_activated(_addr(x), total_rows, N, num_groups, _addr(offsets), fp8_fmt,
                                                      int(activation), _addr(out_row), _addr(scale_row),
                                                      _addr(out_col), _addr(scale_col), _addr(noop), _addr(err_flag),
                                                      _stream(stream)))


def mxfp8_quantize_grouped_swizzled(x, total_rows, N, num_groups, offsets, fp8_fmt, activation, out_row, scale_row,
                                    out_col, scale_col, noop=None, err_flag=None, stream=None) -> int:
    """The grouped cast with per-group GEMM-ready scale planes; see include/mxfp8.h."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_grouped_swizzled(_addr(x), total_rows, N, num_groups, _addr(offsets), fp8_fmt,
                                                     int(activation), _addr(out_row), _addr(scale_row),
                                                     _addr(out_col), _addr(scale_col), _addr(noop), _addr(err_flag),
                                                     _stream(stream)))


def mxfp8_grouped_swizzled_scale_bytes(host_offsets, N: int, colwise: bool) -> int:
    """Bytes of one per-group GEMM-ready scale plane for host offsets [G+1]."""
    off = torch.as_tensor(host_offsets, dtype=torch.int64, device="cpu").contiguous()
    ptr = ctypes.cast(off.data_ptr(), ctypes.POINTER(ctypes.c_int64))
    return int(lib().mxfp8_grouped_swizzled_scale_bytes(ptr, off.numel() - 1, N, int(bool(colwise))))


def mxfp8_quantize_gated_grouped(x, total_rows, N, num_groups, offsets, fp8_fmt, activation, out_row, scale_row,
                                 out_col, scale_col, noop=None, err_flag=None, stream=None) -> int:
    """The gated cast over ragged row groups in one launch; see include/mxfp8.h."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_gated_grouped(_addr(x), total_rows, N, num_groups, _addr(offsets), fp8_fmt,
                                                  int(activation), _addr(out_row), _addr(scale_row), _addr(out_col),
                                                  _addr(scale_col), _addr(noop), _addr(err_flag), _stream(stream)))


def mxfp8_quantize_dgated(grad, x, M, N, fp8_fmt, activation, out_row, scale_row, out_col, scale_col,
                          noop=None, stream=None) -> int:
    """The cast of [g b act'(a) | g act(a)] for x = [a | b]; see include/mxfp8.h."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_dgated(_addr(grad), _addr(x), M, N, fp8_fmt, int(activation), _addr(out_row),
                                           _addr(scale_row), _addr(out_col), _addr(scale_col), _addr(noop),
                                           _stream(stream)))


def mxfp8_quantize_host_staging_bytes(M: int, N: int, with_dbias: bool) -> int:
    return int(lib().mxfp8_quantize_host_staging_bytes(M, N, int(bool(with_dbias))))


def mxfp8_quantize_host(x_host, M, N, fp8_fmt, out_row_host, scale_row_host, out_col_host, scale_col_host,
                        dbias_host, staging, staging_bytes, stream=None) -> int:
    return int(lib().mxfp8_quantize_host(_addr(x_host), M, N, fp8_fmt, _addr(out_row_host), _addr(scale_row_host),
                                         _addr(out_col_host), _addr(scale_col_host), _addr(dbias_host),
                                         _addr(staging), int(staging_bytes), _stream(stream)))


def _act(activation) -> int:
    return ACTIVATIONS[activation.lower()] if isinstance(activation, str) else int(activation)


def mxfp8_quantize_dact_host_staging_bytes(M: int, N: int, with_dbias: bool) -> int:
    return int(lib().mxfp8_quantize_dact_host_staging_bytes(M, N, int(bool(with_dbias))))


def mxfp8_quantize_dact_host(grad_host, act_input_host, M, N, fp8_fmt, activation, out_row_host, scale_row_host,
                             out_col_host, scale_col_host, dbias_host, staging, staging_bytes, stream=None) -> int:
    return int(lib().mxfp8_quantize_dact_host(_addr(grad_host), _addr(act_input_host), M, N, fp8_fmt,
                                              _act(activation), _addr(out_row_host), _addr(scale_row_host),
                                              _addr(out_col_host), _addr(scale_col_host), _addr(dbias_host),
                                              _addr(staging), int(staging_bytes), _stream(stream)))


def mxfp8_quantize_gated_host_staging_bytes(M: int, N: int) -> int:
    return int(lib().mxfp8_quantize_gated_host_staging_bytes(M, N))


def mxfp8_quantize_gated_host(x_host, M, N, fp8_fmt, activation, out_row_host, scale_row_host, out_col_host,
                              scale_col_host, staging, staging_bytes, stream=None) -> int:
    return int(lib().mxfp8_quantize_gated_host(_addr(x_host), M, N, fp8_fmt, _act(activation), _addr(out_row_host),
                                               _addr(scale_row_host), _addr(out_col_host), _addr(scale_col_host),
                                               _addr(staging), int(staging_bytes), _stream(stream)))


def mxfp8_quantize_dgated_host_staging_bytes(M: int, N: int) -> int:
    return int(lib().mxfp8_quantize_dgated_host_staging_bytes(M, N))


def mxfp8_quantize_dgated_host(grad_host, x_host, M, N, fp8_fmt, activation, out_row_host, scale_row_host,
                               out_col_host, scale_col_host, staging, staging_bytes, stream=None) -> int:
    return int(lib().mxfp8_quantize_dgated_host(_addr(grad_host), _addr(x_host), M, N, fp8_fmt, _act(activation),
                                                _addr(out_row_host), _addr(scale_row_host), _addr(out_col_host),
                                                _addr(scale_col_host), _addr(staging), int(staging_bytes),
                                                _stream(stream)))


def mxfp8_quantize_ex_host_staging_bytes(cfg: QuantizeConfig) -> int:
    return int(lib().mxfp8_quantize_ex_host_staging_bytes(ctypes.byref(cfg) if cfg is not None else None))


def mxfp8_quantize_ex_host(cfg: QuantizeConfig, staging, staging_bytes, stream=None) -> int:
    """mxfp8_quantize_ex with host buffers (the config's pointers are host addresses)."""
    return int(lib().mxfp8_quantize_ex_host(ctypes.byref(cfg) if cfg is not None else None, _addr(staging),
                                            int(staging_bytes), _stream(stream)))


def mxfp8_quantize_grouped_host_staging_bytes(total_rows: int, N: int, num_groups: int) -> int:
    return int(lib().mxfp8_quantize_grouped_host_staging_bytes(total_rows, N, num_groups))


def mxfp8_quantize_grouped_host(x_host, total_rows, N, num_groups, host_offsets, fp8_fmt, activation, out_row_host,
                                scale_row_host, out_col_host, scale_col_host, staging, staging_bytes,
                                stream=None) -> int:
    """The grouped cast with host buffers; ``host_offsets`` a CPU int64 tensor or address."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_quantize_grouped_host(_addr(x_host), total_rows, N, num_groups, _addr(host_offsets),
                                                 fp8_fmt, int(activation), _addr(out_row_host),
                                                 _addr(scale_row_host), _addr(out_col_host), _addr(scale_col_host),
                                                 _addr(staging), int(staging_bytes), _stream(stream)))


def mxfp8_grouped_host_chunks(host_offsets, total_rows: int, N: int) -> list:
    """Chunk boundaries the grouped host call uses for these host offsets (a list of rows)."""
    off = torch.as_tensor(host_offsets, dtype=torch.int64, device="cpu").contiguous()
    G = off.numel() - 1
    n = int(lib().mxfp8_grouped_host_chunks(off.data_ptr(), G, total_rows, N, None, 0))
    if n < 0:
        raise ValueError("invalid offsets or shape")
    out = torch.empty((n,), dtype=torch.int64)
    lib().mxfp8_grouped_host_chunks(off.data_ptr(), G, total_rows, N, out.data_ptr(), n)
    return out.tolist()


def mxfp8_scale_bytes(rows: int, scale_cols: int, scale_layout: int = SCALES_PLAIN) -> int:
    return int(lib().mxfp8_scale_bytes(rows, scale_cols, scale_layout))


def mxfp8_quantize_ex(cfg: QuantizeConfig, stream=None) -> int:
    return int(lib().mxfp8_quantize_ex(ctypes.byref(cfg) if cfg is not None else None, _stream(stream)))


def make_config(x, M, N, fp8_fmt, out_row=None, scale_row=None, out_col=None, scale_col=None, dbias=None,
                workspace=None, noop=None, scale_layout=SCALES_PLAIN, amax=None, activation=0) -> QuantizeConfig:
    """A QuantizeConfig from tensors / addresses / None (marshalling only)."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return QuantizeConfig(_addr(x), M, N, fp8_fmt, _addr(out_row), _addr(scale_row), _addr(out_col),
                          _addr(scale_col), _addr(dbias), _addr(workspace), _addr(noop), scale_layout,
                          _addr(amax), int(activation), (ctypes.c_int * 5)())


def mxfp8_status_string(status: int) -> str:
    return lib().mxfp8_status_string(int(status)).decode()


def mxfp8_kernel_launch_count() -> int:
    return int(lib().mxfp8_kernel_launch_count())


def mxfp8_device_fault_word(clear: bool = False) -> int:
    out = ctypes.c_uint(0)
    st = lib().mxfp8_device_fault_word(ctypes.byref(out), int(bool(clear)))
    if st != 0:
        raise MXFP8Error(st, "mxfp8_device_fault_word")
    return int(out.value)


# ---- torch conveniences ----------------------------------------------------------

def mxfp8_selftest_bounded_wait(limit_ns: int, timed_out, stream=None) -> int:
    """Diagnostic: a bounded wait on a phase nothing completes (device int32 ``timed_out`` gets 1)."""
    return int(lib().mxfp8_selftest_bounded_wait(int(limit_ns), _addr(timed_out), _stream(stream)))


def mxfp8_activation_values(x, n, activation, derivative, out, stream=None) -> int:
    """Diagnostic: the kernels' fp32 act(x) (derivative 0) or act'(x) (1) for device bf16 ``x`` [n]."""
    if isinstance(activation, str):
        activation = ACTIVATIONS[activation.lower()]
    return int(lib().mxfp8_activation_values(_addr(x), int(n), int(activation), int(derivative), _addr(out),
                                             _stream(stream)))


class MXFP8Tensor(NamedTuple):
    """Quantized outputs; a direction that was not requested is None."""
    out_row: Optional[torch.Tensor]     # uint8 [M, N]
    scale_row: Optional[torch.Tensor]   # uint8 [M, N/32] (E8M0), or the swizzled plane (1-D)
    out_col: Optional[torch.Tensor]     # uint8 [M, N]
    scale_col: Optional[torch.Tensor]   # uint8 [M/32, N] (E8M0), or the swizzled plane (1-D)
    dbias: Optional[torch.Tensor]       # float32 [N]
    amax: Optional[torch.Tensor] = None  # float32 [1]: max |x|


def _fmt(fmt) -> int:
    if isinstance(fmt, str):
        return {"e4m3": E4M3, "e5m2": E5M2}[fmt.lower()]
    return int(fmt)


def _alloc(x: torch.Tensor, rowwise: bool, colwise: bool, scale_col_rows: Optional[int] = None,
           scales: bool = True):
    """FP8 planes and (with ``scales``) plain scale planes for x [M, N]."""
    M, N = x.shape
    dev = x.device
    u8 = torch.uint8
    sc = -(-M // BLOCK) if scale_col_rows is None else scale_col_rows
    return (torch.empty((M, N), dtype=u8, device=dev) if rowwise else None,
            torch.empty((M, -(-N // BLOCK)), dtype=u8, device=dev) if rowwise and scales else None,
            torch.empty((M, N), dtype=u8, device=dev) if colwise else None,
            torch.empty((sc, N), dtype=u8, device=dev) if colwise and scales else None)


def grouped_scale_col_rows(offsets) -> int:
    """Rows of a grouped call's columnwise scale plane: the sum over groups of ceil(rows_g / 32)
    (total_rows / 32 when every offset is a multiple of 32).  ``offsets`` on the host."""
    off = torch.as_tensor(offsets, dtype=torch.int64, device="cpu")
    return int(((off[1:] - off[:-1]).clamp(min=0) + BLOCK - 1).div(BLOCK, rounding_mode="floor").sum())


def quantize(x: torch.Tensor, fmt=E4M3, rowwise: bool = True, colwise: bool = True,
             with_dbias: bool = False, noop: Optional[torch.Tensor] = None,
             workspace: Optional[torch.Tensor] = None, stream=None, swizzled: bool = False,
             with_amax: bool = False, activation="none") -> MXFP8Tensor:
    """MXFP8-quantize a contiguous CUDA bf16 tensor [M, N] (any M, N a multiple of 8).

    ``swizzled`` writes both scale planes in the GEMM-ready layout (1-D tensors of
    mxfp8_scale_bytes bytes); ``with_amax`` also returns max |x| as a float32 [1];
    ``activation`` ("relu", "srelu", "gelu", "silu", "qgelu") is applied before the cast.
    """
    act = ACTIVATIONS[activation.lower()] if isinstance(activation, str) else int(activation)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D torch.bfloat16 tensor")
    M, N = x.shape
    f = _fmt(fmt)
    if swizzled:
        u8 = dict(dtype=torch.uint8, device=x.device)
        out_row = torch.empty((M, N), **u8) if rowwise else None
        scale_row = torch.empty((mxfp8_scale_bytes(M, -(-N // BLOCK), SCALES_SWIZZLED),), **u8) if rowwise else None
        out_col = torch.empty((M, N), **u8) if colwise else None
        scale_col = torch.empty((mxfp8_scale_bytes(N, -(-M // BLOCK), SCALES_SWIZZLED),), **u8) if colwise else None
    else:
        out_row, scale_row, out_col, scale_col = _alloc(x, rowwise, colwise)
    dbias = torch.empty((N,), dtype=torch.float32, device=x.device) if with_dbias else None
    amax = torch.empty((1,), dtype=torch.float32, device=x.device) if with_amax else None
    if with_dbias and workspace is None:
        nbytes = mxfp8_quantize_workspace_bytes(M, N, True)
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=x.device)
    if swizzled or with_amax or act:
        cfg = make_config(x, M, N, f, out_row, scale_row, out_col, scale_col, dbias,
                          workspace if with_dbias else None, noop,
                          SCALES_SWIZZLED if swizzled else SCALES_PLAIN, amax, act)
        st = mxfp8_quantize_ex(cfg, stream)
    else:
        st = mxfp8_quantize(x, M, N, f, out_row, scale_row, out_col, scale_col, dbias,
                            workspace if with_dbias else None, noop, stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, dbias, amax)


def quantize_host(x: torch.Tensor, fmt=E4M3, rowwise: bool = True, colwise: bool = True,
                  with_dbias: bool = False, staging: Optional[torch.Tensor] = None, stream=None,
                  swizzled: bool = False, with_amax: bool = False, activation="none") -> MXFP8Tensor:
    """Quantize a host (CPU, ideally pinned) bf16 tensor; outputs are pinned host tensors.

    The copies and kernels are pipelined by the library.  The outputs are ready
    once ``stream`` (default: the current CUDA stream) has been synchronised.
    ``swizzled``, ``with_amax`` and ``activation`` are the options of ``quantize``.
    """
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous() or x.is_cuda:
        raise ValueError("x must be a contiguous 2-D torch.bfloat16 host tensor")
    M, N = x.shape
    pin = dict(pin_memory=True)
    u8 = torch.uint8
    layout = SCALES_SWIZZLED if swizzled else SCALES_PLAIN
    out_row = torch.empty((M, N), dtype=u8, **pin) if rowwise else None
    out_col = torch.empty((M, N), dtype=u8, **pin) if colwise else None
    if swizzled:
        scale_row = torch.empty((mxfp8_scale_bytes(M, -(-N // BLOCK), layout),), dtype=u8, **pin) if rowwise else None
        scale_col = torch.empty((mxfp8_scale_bytes(N, -(-M // BLOCK), layout),), dtype=u8, **pin) if colwise else None
    else:
        scale_row = torch.empty((M, -(-N // BLOCK)), dtype=u8, **pin) if rowwise else None
        scale_col = torch.empty((-(-M // BLOCK), N), dtype=u8, **pin) if colwise else None
    dbias = torch.empty((N,), dtype=torch.float32, **pin) if with_dbias else None
    amax = torch.empty((1,), dtype=torch.float32, **pin) if with_amax else None
    act = ACTIVATIONS[activation.lower()] if isinstance(activation, str) else int(activation)
    if not (swizzled or with_amax or act):
        need = mxfp8_quantize_host_staging_bytes(M, N, with_dbias)
        if staging is None:
            staging = torch.empty((max(need, 256),), dtype=u8, device="cuda")
        st = mxfp8_quantize_host(x, M, N, _fmt(fmt), out_row, scale_row, out_col, scale_col, dbias,
                                 staging, staging.numel(), stream)
        if st != 0:
            raise MXFP8Error(st, "mxfp8_quantize_host")
        return MXFP8Tensor(out_row, scale_row, out_col, scale_col, dbias)
    cfg = make_config(x, M, N, _fmt(fmt), out_row, scale_row, out_col, scale_col, dbias, None, None, layout,
                      amax, act)
    need = mxfp8_quantize_ex_host_staging_bytes(cfg)
    if staging is None:
        staging = torch.empty((max(need, 256),), dtype=u8, device="cuda")
    st = mxfp8_quantize_ex_host(cfg, staging, staging.numel(), stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_ex_host")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, dbias, amax)


def quantize_grouped_host(x: torch.Tensor, offsets: torch.Tensor, fmt=E4M3, activation="none",
                          rowwise: bool = True, colwise: bool = True, staging: Optional[torch.Tensor] = None,
                          stream=None) -> MXFP8Tensor:
    """The grouped cast of a host (CPU, ideally pinned) bf16 tensor with host int64 offsets [G+1];
    outputs are pinned host tensors, ready once ``stream`` has been synchronised."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous() or x.is_cuda:
        raise ValueError("x must be a contiguous 2-D torch.bfloat16 host tensor")
    off = torch.as_tensor(offsets, dtype=torch.int64, device="cpu").contiguous()
    total, N = x.shape
    G = off.numel() - 1
    pin = dict(pin_memory=True)
    u8 = torch.uint8
    out_row = torch.empty((total, N), dtype=u8, **pin) if rowwise else None
    scale_row = torch.empty((total, -(-N // BLOCK)), dtype=u8, **pin) if rowwise else None
    out_col = torch.empty((total, N), dtype=u8, **pin) if colwise else None
    scale_col = torch.empty((grouped_scale_col_rows(off), N), dtype=u8, **pin) if colwise else None
    need = mxfp8_quantize_grouped_host_staging_bytes(total, N, G)
    if staging is None:
        staging = torch.empty((max(need, 256),), dtype=u8, device="cuda")
    st = mxfp8_quantize_grouped_host(x, total, N, G, off, _fmt(fmt), activation, out_row, scale_row, out_col,
                                     scale_col, staging, staging.numel(), stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_grouped_host")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, None)


def _host_bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous() or t.is_cuda:
        raise ValueError(f"{name} must be a contiguous 2-D torch.bfloat16 host tensor")


def _host_outputs(M: int, W: int, SR: int, rowwise: bool, colwise: bool):
    pin = dict(dtype=torch.uint8, pin_memory=True)
    return (torch.empty((M, W), **pin) if rowwise else None, torch.empty((M, SR), **pin) if rowwise else None,
            torch.empty((M, W), **pin) if colwise else None, torch.empty((-(-M // BLOCK), W), **pin) if colwise else None)


def quantize_dact_host(grad: torch.Tensor, act_input: torch.Tensor, fmt=E4M3, activation="gelu",
                       rowwise: bool = True, colwise: bool = True, with_dbias: bool = False, stream=None) -> MXFP8Tensor:
    """quantize_dact with host (CPU, ideally pinned) inputs; pinned host outputs, ready once ``stream``
    has been synchronised."""
    _host_bf16(grad, "grad")
    _host_bf16(act_input, "act_input")
    if grad.shape != act_input.shape:
        raise ValueError("grad and act_input must have the same shape")
    M, N = grad.shape
    outs = _host_outputs(M, N, -(-N // BLOCK), rowwise, colwise)
    dbias = torch.empty((N,), dtype=torch.float32, pin_memory=True) if with_dbias else None
    need = mxfp8_quantize_dact_host_staging_bytes(M, N, with_dbias)
    staging = torch.empty((max(need, 256),), dtype=torch.uint8, device="cuda")
    st = mxfp8_quantize_dact_host(grad, act_input, M, N, _fmt(fmt), activation, *outs, dbias, staging,
                                  staging.numel(), stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_dact_host")
    return MXFP8Tensor(*outs, dbias)


def quantize_gated_host(x: torch.Tensor, fmt=E4M3, activation="silu", rowwise: bool = True, colwise: bool = True,
                        stream=None) -> MXFP8Tensor:
    """quantize_gated with a host [M, 2N] input; pinned host outputs."""
    _host_bf16(x, "x")
    M, N2 = x.shape
    if N2 % 2:
        raise ValueError("a gated input has an even number of columns")
    N = N2 // 2
    outs = _host_outputs(M, N, -(-N // BLOCK), rowwise, colwise)
    need = mxfp8_quantize_gated_host_staging_bytes(M, N)
    staging = torch.empty((max(need, 256),), dtype=torch.uint8, device="cuda")
    st = mxfp8_quantize_gated_host(x, M, N, _fmt(fmt), activation, *outs, staging, staging.numel(), stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_gated_host")
    return MXFP8Tensor(*outs, None)


def quantize_dgated_host(grad: torch.Tensor, x: torch.Tensor, fmt=E5M2, activation="silu", rowwise: bool = True,
                         colwise: bool = True, stream=None) -> MXFP8Tensor:
    """quantize_dgated with host inputs (grad [M, N], x [M, 2N]); pinned host outputs [M, 2N]."""
    _host_bf16(grad, "grad")
    _host_bf16(x, "x")
    M, N = grad.shape
    if x.shape != (M, 2 * N):
        raise ValueError("x must be [M, 2N] for grad [M, N]")
    outs = _host_outputs(M, 2 * N, 2 * -(-N // BLOCK), rowwise, colwise)
    need = mxfp8_quantize_dgated_host_staging_bytes(M, N)
    staging = torch.empty((max(need, 256),), dtype=torch.uint8, device="cuda")
    st = mxfp8_quantize_dgated_host(grad, x, M, N, _fmt(fmt), activation, *outs, staging, staging.numel(), stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_dgated_host")
    return MXFP8Tensor(*outs, None)


def quantize_dact(grad: torch.Tensor, act_input: torch.Tensor, fmt=E4M3, activation="gelu",
                  rowwise: bool = True, colwise: bool = True, with_dbias: bool = False,
                  noop: Optional[torch.Tensor] = None, stream=None) -> MXFP8Tensor:
    """The cast of grad * act'(act_input) (both contiguous CUDA bf16 [M, N]), dbias optional."""
    for t in (grad, act_input):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
            raise ValueError("grad and act_input must be contiguous 2-D torch.bfloat16 tensors")
    if grad.shape != act_input.shape:
        raise ValueError("grad and act_input must have the same shape")
    M, N = grad.shape
    out_row, scale_row, out_col, scale_col = _alloc(grad, rowwise, colwise)
    dbias = torch.empty((N,), dtype=torch.float32, device=grad.device) if with_dbias else None
    ws = (torch.empty((max(mxfp8_quantize_workspace_bytes(M, N, True), 16),), dtype=torch.uint8,
                      device=grad.device) if with_dbias else None)
    st = mxfp8_quantize_dact(grad, act_input, M, N, _fmt(fmt), activation, out_row, scale_row, out_col,
                             scale_col, dbias, ws, noop, stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_dact")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, dbias)


def quantize_gated(x: torch.Tensor, fmt=E4M3, activation="silu", rowwise: bool = True, colwise: bool = True,
                   noop: Optional[torch.Tensor] = None, stream=None) -> MXFP8Tensor:
    """The cast of act(a) * b for a contiguous CUDA bf16 x = [a | b] of shape [M, 2N].

    ``activation`` "silu" gives SwiGLU, "gelu" GeGLU, "relu" ReGLU, "srelu" the squared-ReLU
    GLU, "qgelu" QGeGLU; the outputs are [M, N].
    """
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D torch.bfloat16 tensor")
    if x.shape[1] % 2:
        raise ValueError("a gated input has an even number of columns")
    M, N = x.shape[0], x.shape[1] // 2
    out_row, scale_row, out_col, scale_col = _alloc(x[:, :N], rowwise, colwise)
    st = mxfp8_quantize_gated(x, M, N, _fmt(fmt), activation, out_row, scale_row, out_col, scale_col, noop, stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_gated")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, None)


def quantize_gated_grouped(x: torch.Tensor, offsets: torch.Tensor, fmt=E4M3, activation="silu",
                           rowwise: bool = True, colwise: bool = True, noop: Optional[torch.Tensor] = None,
                           err_flag: Optional[torch.Tensor] = None, stream=None,
                           scale_col_rows: Optional[int] = None) -> MXFP8Tensor:
    """The gated cast of x = [a | b] (bf16 [total_rows, 2N]) over the row groups of ``offsets``
    (a CUDA int64 prefix vector [G+1]); scale_col rows as for quantize_grouped."""
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D torch.bfloat16 tensor")
    if x.shape[1] % 2:
        raise ValueError("a gated input has an even number of columns")
    if offsets.dtype != torch.int64 or offsets.dim() != 1 or not offsets.is_contiguous():
        raise ValueError("offsets must be a contiguous 1-D torch.int64 tensor")
    total, N = x.shape[0], x.shape[1] // 2
    G = offsets.numel() - 1
    if colwise and scale_col_rows is None:
        scale_col_rows = grouped_scale_col_rows(offsets.cpu())
    out_row, scale_row, out_col, scale_col = _alloc(x[:, :N], rowwise, colwise, scale_col_rows)
    st = mxfp8_quantize_gated_grouped(x, total, N, G, offsets, _fmt(fmt), activation, out_row, scale_row, out_col,
                                      scale_col, noop, err_flag, stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_gated_grouped")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, None)


def quantize_dgated(grad: torch.Tensor, x: torch.Tensor, fmt=E5M2, activation="silu", rowwise: bool = True,
                    colwise: bool = True, noop: Optional[torch.Tensor] = None, stream=None) -> MXFP8Tensor:
    """The cast of the gradient of x = [a | b] for y = act(a) * b, given grad = dL/dy [M, N].

    Returns codes [M, 2N] (da | db), scale_row [M, 2 ceil(N/32)] (da's blocks, then db's),
    scale_col [ceil(M/32), 2N].
    """
    for t in (grad, x):
        if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_contiguous():
            raise ValueError("grad and x must be contiguous 2-D torch.bfloat16 tensors")
    M, N = grad.shape
    if x.shape != (M, 2 * N):
        raise ValueError("x must be [M, 2N] for grad of shape [M, N]")
    u8 = dict(dtype=torch.uint8, device=grad.device)
    out_row = torch.empty((M, 2 * N), **u8) if rowwise else None
    scale_row = torch.empty((M, 2 * (-(-N // BLOCK))), **u8) if rowwise else None
    out_col = torch.empty((M, 2 * N), **u8) if colwise else None
    scale_col = torch.empty((-(-M // BLOCK), 2 * N), **u8) if colwise else None
    st = mxfp8_quantize_dgated(grad, x, M, N, _fmt(fmt), activation, out_row, scale_row, out_col, scale_col,
                               noop, stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_dgated")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, None)


def quantize_grouped(x: torch.Tensor, offsets: torch.Tensor, fmt=E4M3, rowwise: bool = True,
                     colwise: bool = True, noop: Optional[torch.Tensor] = None,
                     err_flag: Optional[torch.Tensor] = None, stream=None, with_dbias: bool = False,
                     scale_col_rows: Optional[int] = None, activation="none",
                     swizzled: bool = False) -> MXFP8Tensor:
    """Grouped quantize; ``offsets`` is a CUDA int64 prefix vector [G+1] (kept on the device).

    Every group is quantized as its own flat problem; ``scale_col`` has
    ``grouped_scale_col_rows(offsets)`` rows, group g's after those of the groups before it.
    Pass ``scale_col_rows`` when it is known on the host; otherwise it is computed from a
    host copy of ``offsets`` (one device-to-host read).  ``with_dbias`` also returns the
    per-group column sums as float32 [G, N]; ``activation`` ("relu", "srelu", "gelu", "silu",
    "qgelu") casts act(x) instead (no dbias then).  ``swizzled`` writes each group's scale planes
    in the GEMM-ready layout (1-D uint8 tensors; see include/mxfp8.h; no dbias), which reads a host
    copy of ``offsets``.
    """
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_contiguous():
        raise ValueError("x must be a contiguous 2-D torch.bfloat16 tensor")
    if offsets.dtype != torch.int64 or offsets.dim() != 1 or not offsets.is_contiguous():
        raise ValueError("offsets must be a contiguous 1-D torch.int64 tensor")
    total, N = x.shape
    G = offsets.numel() - 1
    act = ACTIVATIONS[activation.lower()] if isinstance(activation, str) else int(activation)
    if act and with_dbias:
        raise ValueError("an activation does not combine with dbias")
    if swizzled and with_dbias:
        raise ValueError("the swizzled grouped call has no dbias")
    if colwise and scale_col_rows is None and not swizzled:
        scale_col_rows = grouped_scale_col_rows(offsets.cpu())
    out_row, scale_row, out_col, scale_col = _alloc(x, rowwise, colwise, scale_col_rows or 0, scales=not swizzled)
    if swizzled:
        host_off = offsets.cpu()
        u8 = dict(dtype=torch.uint8, device=x.device)
        if rowwise:
            scale_row = torch.empty((max(mxfp8_grouped_swizzled_scale_bytes(host_off, N, False), 1),), **u8)
        if colwise:
            scale_col = torch.empty((max(mxfp8_grouped_swizzled_scale_bytes(host_off, N, True), 1),), **u8)
        dbias = None
        st = mxfp8_quantize_grouped_swizzled(x, total, N, G, offsets, _fmt(fmt), act, out_row, scale_row, out_col,
                                             scale_col, noop, err_flag, stream)
    elif act:
        dbias = None
        st = mxfp8_quantize_grouped_activated(x, total, N, G, offsets, _fmt(fmt), act, out_row, scale_row, out_col,
                                              scale_col, noop, err_flag, stream)
    elif with_dbias:
        dbias = torch.empty((G, N), dtype=torch.float32, device=x.device)
        ws = torch.empty((max(mxfp8_quantize_grouped_dbias_workspace_bytes(total, N, G), 16),), dtype=torch.uint8,
                         device=x.device)
        st = mxfp8_quantize_grouped_dbias(x, total, N, G, offsets, _fmt(fmt), out_row, scale_row, out_col,
                                          scale_col, dbias, ws, noop, err_flag, stream)
    else:
        dbias = None
        st = mxfp8_quantize_grouped(x, total, N, G, offsets, _fmt(fmt), out_row, scale_row,
                                    out_col, scale_col, None, noop, err_flag, stream)
    if st != 0:
        raise MXFP8Error(st, "mxfp8_quantize_grouped")
    return MXFP8Tensor(out_row, scale_row, out_col, scale_col, dbias)


def mxfp8_quantize_dbias_noalloc(x, M, N, fp8_fmt, out_row, scale_row, out_col, scale_col,
                                 dbias, noop=None, stream=None) -> int:
    """mxfp8_quantize with dbias and no workspace argument (for callers that cannot allocate).

    The C entry point keeps the dbias workspace in an 8 MiB static device array;
    see include/mxfp8.h for its limits and its sharing rule.
    """
    f = lib().mxfp8_quantize_dbias_noalloc
    if f.argtypes is None:
        vp = ctypes.c_void_p
        f.restype = ctypes.c_int
        f.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp]
    return int(f(_addr(x), M, N, fp8_fmt, _addr(out_row), _addr(scale_row), _addr(out_col), _addr(scale_col),
                 _addr(dbias), _addr(noop), _stream(stream)))
