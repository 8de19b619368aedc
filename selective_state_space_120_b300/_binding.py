"""ctypes binding of libssscan.so (the C ABI in include/ssscan.h).

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  If the compiled library is missing the calls raise: there is no CPU
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libssscan.so")

SS_OK = 0
SS_ERR_INVALID_ARG = 1
SS_ERR_UNSUPPORTED = 2
SS_ERR_ALIGNMENT = 3
SS_ERR_WORKSPACE = 4
SS_ERR_CUDA = 5
SS_ERR_TIMEOUT = 6
SS_F32 = 0
SS_BF16 = 1
SS_KIND_SCAN, SS_KIND_BIDIR, SS_KIND_CROSS2D, SS_KIND_SCAN_BWD = 0, 1, 2, 3
SS_DEBUG_SKIP_FIRST_COPY = 1
# traversal orders (SS_DIR_*)
(SS_DIR_ROW, SS_DIR_COL, SS_DIR_ROW_REV, SS_DIR_COL_REV, SS_DIR_WIN, SS_DIR_WIN_COL,
 SS_DIR_WIN_REV, SS_DIR_WIN_COL_REV) = range(8)
SS_NOALLOC_SCRATCH_BYTES = 16 << 20
STATUS_NAMES = {0: "SS_OK", 1: "SS_ERR_INVALID_ARG", 2: "SS_ERR_UNSUPPORTED",
                3: "SS_ERR_ALIGNMENT", 4: "SS_ERR_WORKSPACE", 5: "SS_ERR_CUDA",
                6: "SS_ERR_TIMEOUT"}

# Every function the header declares.
EXPORTS = ("ss_selective_scan_fwd", "ss_selective_scan_fwd_opts", "ss_bidir_scan_fwd",
           "ss_cross_scan2d_fwd", "ss_workspace_bytes", "ss_workspace_bytes_opts",
           "ss_get_device_status", "ss_last_error_string", "ss_version",
           "ss_debug_set_wait_budget_ns", "ss_debug_set_flags",
           "ss_selective_scan_fwd_noalloc", "ss_selective_state_update",
           "ss_selective_scan_bwd", "ss_multi_scan_fwd", "ss_multi_scan_workspace_bytes",
           "ss_dwconv3x3_silu_fwd", "ss_multi_scan_bwd", "ss_multi_scan_bwd_workspace_bytes",
           "ss_selective_scan_bwd_opts")


class SSError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class ScanOptions(ctypes.Structure):
    _fields_ = [("chunks", ctypes.c_int), ("flags", ctypes.c_uint), ("h0", ctypes.c_void_p),
                ("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p),
                ("conv_x0", ctypes.c_void_p), ("reserved", ctypes.c_int * 6)]


class BwdExtras(ctypes.Structure):
    _fields_ = [("dh0", ctypes.c_void_p), ("dconv_w", ctypes.c_void_p),
                ("dconv_b", ctypes.c_void_p), ("dconv_x0", ctypes.c_void_p),
                ("reserved", ctypes.c_int * 8)]


SS_SCAN_ZOH = 1
SS_SCAN_CONV_SILU = 2


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads and types the library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libssscan.so not found at {path}; run "
                               "`python -m selective_state_space_120_b300.build`")
        lib = ctypes.CDLL(path)
        i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        scan_args = [i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp,
                     vp, sz]
        lib.ss_selective_scan_fwd.argtypes = scan_args + [vp]
        lib.ss_selective_scan_fwd_opts.argtypes = scan_args + [ctypes.POINTER(ScanOptions), vp]
        lib.ss_bidir_scan_fwd.argtypes = scan_args + [vp]
        lib.ss_selective_state_update.argtypes = [i64, i64, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                                  vp, vp, i32, ctypes.c_uint, vp, vp, vp]
        lib.ss_selective_scan_fwd_noalloc.argtypes = scan_args[:-2] + [
            ctypes.POINTER(ScanOptions), vp]
        lib.ss_cross_scan2d_fwd.argtypes = [i64, i64, i64, i64, i32, i32, i32, vp, vp, vp, vp, vp,
                                            vp, vp, i32, vp, vp, vp, vp, sz, vp]
        # u ... delta_softplus as the forward call, then dout, du, ddelta, dA, dB, dC, dD, dz,
        # ddelta_bias, workspace, workspace_bytes, stream
        lib.ss_selective_scan_bwd.argtypes = scan_args[:15] + [vp] * 9 + [vp, sz, vp]
        # the same, with the forward call's options and the gradients of their tensors
        lib.ss_selective_scan_bwd_opts.argtypes = scan_args[:15] + [vp] * 9 + [
            ctypes.POINTER(ScanOptions), ctypes.POINTER(BwdExtras), vp, sz, vp]
        # batch, dim, H, W, ndirs, orders (host int array), window, dstate, ngroups, io,
        # u, delta, A, B, C, D, delta_bias, delta_softplus, z, out, last_state, workspace,
        # workspace_bytes, stream
        lib.ss_multi_scan_fwd.argtypes = [i64, i64, i64, i64, i32, ctypes.POINTER(i32), i32, i32,
                                          i32, i32] + [vp] * 7 + [i32, vp, vp, vp, vp, sz, vp]
        # batch, dim, H, W, ndirs, orders, window, dstate, ngroups, io, u, delta, A, B, C, D,
        # delta_bias, delta_softplus, z, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias,
        # workspace, workspace_bytes, stream
        lib.ss_multi_scan_bwd.argtypes = ([i64, i64, i64, i64, i32, ctypes.POINTER(i32), i32, i32, i32,
                                           i32] + [vp] * 7 + [i32] + [vp] * 10 + [vp, sz, vp])
        lib.ss_multi_scan_bwd.restype = ctypes.c_int
        lib.ss_multi_scan_bwd_workspace_bytes.argtypes = [i64, i64, i64, i64, i32, i32]
        lib.ss_multi_scan_bwd_workspace_bytes.restype = sz
        lib.ss_dwconv3x3_silu_fwd.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp, vp]
        lib.ss_dwconv3x3_silu_fwd.restype = ctypes.c_int
        lib.ss_multi_scan_workspace_bytes.argtypes = [i64, i64, i64, i64, i32]
        lib.ss_multi_scan_workspace_bytes.restype = sz
        for f in ("ss_selective_scan_fwd", "ss_selective_scan_fwd_opts", "ss_bidir_scan_fwd",
                  "ss_cross_scan2d_fwd", "ss_get_device_status", "ss_debug_set_wait_budget_ns",
                  "ss_debug_set_flags", "ss_selective_scan_fwd_noalloc",
                  "ss_selective_state_update", "ss_selective_scan_bwd", "ss_multi_scan_fwd",
                  "ss_selective_scan_bwd_opts"):
            getattr(lib, f).restype = ctypes.c_int
        lib.ss_workspace_bytes.argtypes = [i32, i64, i64, i64, i32]
        lib.ss_workspace_bytes.restype = sz
        lib.ss_workspace_bytes_opts.argtypes = [i32, i64, i64, i64, i32,
                                                ctypes.POINTER(ScanOptions)]
        lib.ss_workspace_bytes_opts.restype = sz
        lib.ss_get_device_status.argtypes = [vp]
        lib.ss_last_error_string.restype = ctypes.c_char_p
        lib.ss_version.restype = ctypes.c_char_p
        lib.ss_debug_set_wait_budget_ns.argtypes = [ctypes.c_uint64]
        lib.ss_debug_set_flags.argtypes = [ctypes.c_uint32]
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != SS_OK:
        raise SSError(status, load().ss_last_error_string().decode())


def last_error() -> str:
    return load().ss_last_error_string().decode()


def version() -> str:
    return load().ss_version().decode()


def options(chunks: int = 0, flags: int = 0, h0: int | None = None, conv_w: int | None = None,
            conv_b: int | None = None, conv_x0: int | None = None) -> ScanOptions:
    o = ScanOptions()
    o.chunks = int(chunks)
    o.flags = int(flags)
    o.h0 = h0
    o.conv_w = conv_w
    o.conv_b = conv_b
    o.conv_x0 = conv_x0
    return o


def workspace_bytes(kind: int, batch: int, dim: int, seqlen: int, dstate: int,
                    chunks: int = 0) -> int:
    o = options(chunks)
    return int(load().ss_workspace_bytes_opts(kind, batch, dim, seqlen, dstate, ctypes.byref(o)))
