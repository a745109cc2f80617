"""ctypes binding of ``libgconv.so`` -- argument marshalling only.

Function names match the C ABI in ``include/gconv.h``.  Every device-side
step runs in the library's CUDA kernels; this module only turns Python values
(torch tensors, ints, problem records) into the C arguments and raises
``GconvError`` on a non-OK status.  If the library has not been built the
first call raises immediately: there is no Python or CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgconv.so")

GCONV_OK = 0
GCONV_ERR_INVALID_ARG = 1
GCONV_ERR_UNSUPPORTED = 2
GCONV_ERR_CUDA = 3
GCONV_ERR_TIMEOUT = 4

GCONV_F32, GCONV_F16, GCONV_BF16 = 0, 1, 2
DTYPE_CODES = {"f32": GCONV_F32, "f16": GCONV_F16, "bf16": GCONV_BF16}

KERNEL_AUTO, KERNEL_DIRECT_DW, KERNEL_DIRECT_GENERIC, KERNEL_IGEMM_TC = 0, 1, 2, 3
KERNEL_BWD_DATA_DIRECT = 4
KERNEL_BWD_WEIGHT = 5
KERNEL_DW_PW = 6
KERNEL_NAMES = {KERNEL_DIRECT_DW: "direct_dw", KERNEL_DIRECT_GENERIC: "direct_generic",
                KERNEL_IGEMM_TC: "igemm_tc", KERNEL_BWD_DATA_DIRECT: "bwd_data_direct",
                KERNEL_BWD_WEIGHT: "bwd_weight", KERNEL_DW_PW: "dw_pw"}


class gconv_problem(ctypes.Structure):
    _fields_ = [("ndim", ctypes.c_int32), ("reserved", ctypes.c_int32), ("N", ctypes.c_int64),
                ("G", ctypes.c_int32), ("C", ctypes.c_int32), ("K", ctypes.c_int32),
                ("in_", ctypes.c_int32 * 3), ("ker", ctypes.c_int32 * 3),
                ("stride", ctypes.c_int32 * 3), ("pad", ctypes.c_int32 * 3),
                ("dil", ctypes.c_int32 * 3)]


class gconv_options(ctypes.Structure):
    _fields_ = [("force_kernel", ctypes.c_int32), ("debug", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("test_flags", ctypes.c_int32),
                ("selected", ctypes.c_int32), ("tile", ctypes.c_int32 * 8),
                ("serial_launch", ctypes.c_int32)]


class GconvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"gconv status {status}: {message}")
        self.status = status


_lib = None
_lock = threading.Lock()


def load_library(path: Optional[str] = None):
    """Load libgconv.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build the CUDA library first "
                               "(python -m depthwise_convolution_forward_gb300.build)")
        lib = ctypes.CDLL(p)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        prob_p = ctypes.POINTER(gconv_problem)
        lib.grouped_conv_fwd.restype = i32
        lib.grouped_conv_fwd.argtypes = [vp, vp, vp, vp, prob_p, i32, vp]
        lib.grouped_conv_fwd_ex.restype = i32
        lib.grouped_conv_fwd_ex.argtypes = [vp, vp, vp, vp, prob_p, i32, vp,
                                            ctypes.POINTER(gconv_options)]
        lib.grouped_conv_bwd_data.restype = i32
        lib.grouped_conv_bwd_data.argtypes = [vp, vp, vp, prob_p, i32, vp, i64, vp]
        lib.grouped_conv_bwd_data_ex.restype = i32
        lib.grouped_conv_bwd_data_ex.argtypes = [vp, vp, vp, prob_p, i32, vp, i64, vp,
                                                 ctypes.POINTER(gconv_options)]
        lib.grouped_conv_bwd_weight.restype = i32
        lib.grouped_conv_bwd_weight.argtypes = [vp, vp, vp, prob_p, i32, vp, i64, vp]
        lib.grouped_conv_bwd_weight_ex.restype = i32
        lib.grouped_conv_bwd_weight_ex.argtypes = [vp, vp, vp, prob_p, i32, vp, i64, vp,
                                                   ctypes.POINTER(gconv_options)]
        lib.grouped_conv_bwd_weight_workspace_size.restype = i32
        lib.grouped_conv_bwd_weight_workspace_size.argtypes = [prob_p, i32, ctypes.POINTER(i64)]
        lib.grouped_conv_bwd_data_route.restype = i32
        lib.grouped_conv_bwd_data_route.argtypes = [prob_p, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.grouped_conv_fwd_dw_pw.restype = i32
        lib.grouped_conv_fwd_dw_pw.argtypes = [vp, vp, vp, vp, vp, vp, prob_p, i32, i32, i32, vp]
        lib.grouped_conv_fwd_dw_pw_ex.restype = i32
        lib.grouped_conv_fwd_dw_pw_ex.argtypes = [vp, vp, vp, vp, vp, vp, prob_p, i32, i32, i32, vp,
                                                  ctypes.POINTER(gconv_options)]
        lib.grouped_conv_fwd_dw_pw_supported.restype = i32
        lib.grouped_conv_fwd_dw_pw_supported.argtypes = [prob_p, i32, i32, i32, ctypes.POINTER(i32)]
        lib.grouped_conv_bwd_data_noalloc.restype = i32
        lib.grouped_conv_bwd_data_noalloc.argtypes = [vp, vp, vp, prob_p, i32, vp]
        lib.grouped_conv_bwd_data_workspace_size.restype = i32
        lib.grouped_conv_bwd_data_workspace_size.argtypes = [prob_p, i32, ctypes.POINTER(i64)]
        lib.grouped_conv_out_shape.restype = i32
        lib.grouped_conv_out_shape.argtypes = [prob_p, ctypes.POINTER(i32)]
        lib.grouped_conv_select.restype = i32
        lib.grouped_conv_select.argtypes = [prob_p, i32, ctypes.POINTER(i32)]
        lib.gconv_epilogue_apply.restype = i32
        lib.gconv_epilogue_apply.argtypes = [vp, vp, vp, i64, i32, i32, vp]
        lib.gconv_device_status.restype = i32
        lib.gconv_device_status.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.gconv_status_string.restype = ctypes.c_char_p
        lib.gconv_status_string.argtypes = [i32]
        lib.gconv_last_error.restype = ctypes.c_char_p
        lib.gconv_last_error.argtypes = []
        _lib = lib
        return lib


def _check(status: int):
    if status != GCONV_OK:
        lib = load_library()
        raise GconvError(status, lib.gconv_last_error().decode())


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_problem(ndim: int, N: int, G: int, C: int, K: int, inp: Sequence[int], ker: Sequence[int],
                 stride: Sequence[int], pad: Sequence[int], dil: Sequence[int]) -> gconv_problem:
    """Problem record; spatial sequences are (D, H, W) / (Z, Y, X)."""
    p = gconv_problem()
    p.ndim, p.reserved, p.N, p.G, p.C, p.K = ndim, 0, N, G, C, K
    for i in range(3):
        p.in_[i], p.ker[i], p.stride[i], p.pad[i], p.dil[i] = inp[i], ker[i], stride[i], pad[i], dil[i]
    return p


def problem_of(wl) -> gconv_problem:
    """Problem record of an ``inputs.Workload``."""
    return make_problem(wl.ndim, wl.N, wl.G, wl.C, wl.K, wl.inp, wl.ker, wl.stride, wl.pad, wl.dil)


def grouped_conv_out_shape(p: gconv_problem) -> tuple:
    lib = load_library()
    out = (ctypes.c_int32 * 3)()
    _check(lib.grouped_conv_out_shape(ctypes.byref(p), out))
    return tuple(out)


def grouped_conv_select(p: gconv_problem, dtype: int) -> int:
    lib = load_library()
    k = ctypes.c_int32(0)
    _check(lib.grouped_conv_select(ctypes.byref(p), dtype, ctypes.byref(k)))
    return k.value


def grouped_conv_fwd(x, w, bias, y, p: gconv_problem, dtype: int, stream=None) -> None:
    lib = load_library()
    _check(lib.grouped_conv_fwd(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), ctypes.byref(p), dtype,
                                _stream(stream)))


def grouped_conv_fwd_ex(x, w, bias, y, p: gconv_problem, dtype: int, stream=None,
                        opt: Optional[gconv_options] = None) -> gconv_options:
    lib = load_library()
    o = opt if opt is not None else gconv_options()
    _check(lib.grouped_conv_fwd_ex(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), ctypes.byref(p), dtype,
                                   _stream(stream), ctypes.byref(o)))
    return o


def gconv_epilogue_apply(acc, bias, y, rows: int, cols: int, dtype: int, stream=None) -> None:
    lib = load_library()
    _check(lib.gconv_epilogue_apply(_ptr(acc), _ptr(bias), _ptr(y), rows, cols, dtype,
                                    _stream(stream)))


def gconv_device_status(stream=None) -> tuple:
    lib = load_library()
    code, where = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.gconv_device_status(_stream(stream), ctypes.byref(code), ctypes.byref(where)))
    return code.value, where.value


def gconv_status_string(status: int) -> str:
    return load_library().gconv_status_string(status).decode()


def gconv_last_error() -> str:
    return load_library().gconv_last_error().decode()


def grouped_conv_bwd_data_workspace_size(p: gconv_problem, dtype: int) -> int:
    """Device workspace bytes grouped_conv_bwd_data needs (0 when none)."""
    lib = load_library()
    n = ctypes.c_int64(0)
    _check(lib.grouped_conv_bwd_data_workspace_size(ctypes.byref(p), dtype, ctypes.byref(n)))
    return n.value


def grouped_conv_bwd_data(dy, w, dx, p: gconv_problem, dtype: int, workspace=None, workspace_bytes: int = 0,
                          stream=None) -> None:
    lib = load_library()
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.grouped_conv_bwd_data(_ptr(dy), _ptr(w), _ptr(dx), ctypes.byref(p), dtype, _ptr(workspace),
                                     workspace_bytes, _stream(stream)))


def grouped_conv_bwd_data_ex(dy, w, dx, p: gconv_problem, dtype: int, workspace=None, workspace_bytes: int = 0,
                             stream=None, opt: Optional[gconv_options] = None) -> gconv_options:
    lib = load_library()
    o = opt if opt is not None else gconv_options()
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.grouped_conv_bwd_data_ex(_ptr(dy), _ptr(w), _ptr(dx), ctypes.byref(p), dtype, _ptr(workspace),
                                        workspace_bytes, _stream(stream), ctypes.byref(o)))
    return o


def grouped_conv_bwd_data_route(p: gconv_problem, dtype: int) -> tuple:
    """(route, launches) of grouped_conv_bwd_data: route 0 direct gather,
    1 stride 1 with transposed flipped weights, 2 stride phases."""
    lib = load_library()
    r, n = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(lib.grouped_conv_bwd_data_route(ctypes.byref(p), dtype, ctypes.byref(r), ctypes.byref(n)))
    return r.value, n.value


def grouped_conv_bwd_weight_workspace_size(p: gconv_problem, dtype: int) -> int:
    """Device workspace bytes grouped_conv_bwd_weight needs (never 0)."""
    lib = load_library()
    n = ctypes.c_int64(0)
    _check(lib.grouped_conv_bwd_weight_workspace_size(ctypes.byref(p), dtype, ctypes.byref(n)))
    return n.value


def grouped_conv_bwd_weight(x, dy, dw, p: gconv_problem, dtype: int, workspace=None, workspace_bytes: int = 0,
                            stream=None) -> None:
    lib = load_library()
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.grouped_conv_bwd_weight(_ptr(x), _ptr(dy), _ptr(dw), ctypes.byref(p), dtype, _ptr(workspace),
                                       workspace_bytes, _stream(stream)))


def grouped_conv_bwd_weight_ex(x, dy, dw, p: gconv_problem, dtype: int, workspace=None, workspace_bytes: int = 0,
                               stream=None, opt: Optional[gconv_options] = None) -> gconv_options:
    lib = load_library()
    o = opt if opt is not None else gconv_options()
    if workspace is not None and not isinstance(workspace, int) and not workspace_bytes:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(lib.grouped_conv_bwd_weight_ex(_ptr(x), _ptr(dy), _ptr(dw), ctypes.byref(p), dtype, _ptr(workspace),
                                          workspace_bytes, _stream(stream), ctypes.byref(o)))
    return o


GCONV_NOALLOC_SCRATCH_BYTES = 1 << 20  # include/gconv.h


def grouped_conv_bwd_data_noalloc(dy, w, dx, p: gconv_problem, dtype: int, stream=None) -> None:
    """Backward data without a caller workspace: the library's fixed scratch
    array (GCONV_NOALLOC_SCRATCH_BYTES) stands in for it; see gconv.h."""
    lib = load_library()
    _check(lib.grouped_conv_bwd_data_noalloc(_ptr(dy), _ptr(w), _ptr(dx), ctypes.byref(p), dtype,
                                             _stream(stream)))


def grouped_conv_fwd_dw_pw(x, w_dw, b_dw, w_pw, b_pw, y, p: gconv_problem, K: int, act: int, dtype: int,
                           stream=None) -> None:
    """Depthwise 3x3 + bias + activation, then the 1x1 projection + bias, in
    one kernel (see gconv.h)."""
    lib = load_library()
    _check(lib.grouped_conv_fwd_dw_pw(_ptr(x), _ptr(w_dw), _ptr(b_dw), _ptr(w_pw), _ptr(b_pw), _ptr(y),
                                      ctypes.byref(p), K, act, dtype, _stream(stream)))


def grouped_conv_fwd_dw_pw_ex(x, w_dw, b_dw, w_pw, b_pw, y, p: gconv_problem, K: int, act: int, dtype: int,
                              stream=None, opt: Optional[gconv_options] = None) -> gconv_options:
    lib = load_library()
    o = opt if opt is not None else gconv_options()
    _check(lib.grouped_conv_fwd_dw_pw_ex(_ptr(x), _ptr(w_dw), _ptr(b_dw), _ptr(w_pw), _ptr(b_pw), _ptr(y),
                                         ctypes.byref(p), K, act, dtype, _stream(stream), ctypes.byref(o)))
    return o


def grouped_conv_fwd_dw_pw_supported(p: gconv_problem, K: int, act: int, dtype: int) -> bool:
    lib = load_library()
    ok = ctypes.c_int32(0)
    _check(lib.grouped_conv_fwd_dw_pw_supported(ctypes.byref(p), K, act, dtype, ctypes.byref(ok)))
    return bool(ok.value)

