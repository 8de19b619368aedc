"""Float64 CPU oracle for the selective scan -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does, and
this package never imports the product library: the two share no code.

The arithmetic lives in ``ss_oracle.c`` (plain C, float64, sequential over the
scan).  This module compiles it with gcc into ``liboracle.so`` beside the
source and calls it through ctypes with NumPy float64 arrays.

Conventions (see the C file's header for the equations and their sources):
    u [batch, dim, L], delta [batch, K, dim, L], A [K*dim, N],
    B, C [batch, K, G, N, L], D / delta_bias [K*dim], z [batch, dim, L],
    h0 / last_state [batch, K, dim, N]; u, z and the output are indexed by
    position, the per-direction Delta, B, C by that direction's scan step, and a
    direction's order is one of ORDER_*.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

ORDER_FWD = 0       # positions 0..L-1 (row-major for an H x W map)
ORDER_REV = 1       # positions L-1..0
ORDER_COL = 2       # column-major over an H x W map
ORDER_COL_REV = 3   # reverse of column-major
# windowed orders (LocalMamba): w x w windows visited one after another, the
# windows of the last band of rows / last column cut short
ORDER_WIN = 4          # windows row-major, each window row-major
ORDER_WIN_REV = 5      # reverse of ORDER_WIN
ORDER_WIN_COL = 6      # windows column-major, each window column-major
ORDER_WIN_COL_REV = 7  # reverse of ORDER_WIN_COL

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ss_oracle.c into liboracle.so (no fast-math, no vectorisation flags)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.ssor_scan.restype = ctypes.c_int
    lib.ssor_scan.argtypes = [i64, i64, i64, i64, i64, i64, i64,
                              ctypes.POINTER(ctypes.c_int), i64,
                              dp, dp, dp, dp, dp, dp, dp, dp,
                              ctypes.c_int, ctypes.c_int, dp, dp, dp, dp]
    lib.ssor_scan_bwd.restype = ctypes.c_int
    lib.ssor_scan_bwd.argtypes = [i64, i64, i64, i64, i64] + [dp] * 8 + [ctypes.c_int] + [dp] * 10
    lib.ssor_scan_bwd_ext.restype = ctypes.c_int
    lib.ssor_scan_bwd_ext.argtypes = ([i64, i64, i64, i64, i64] + [dp] * 8 + [ctypes.c_int] * 2 +
                                      [dp] * 12)
    lib.ssor_conv_silu.restype = ctypes.c_int
    lib.ssor_conv_silu.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp, dp]
    lib.ssor_conv_silu_bwd.restype = ctypes.c_int
    lib.ssor_conv_silu_bwd.argtypes = [i64, i64, i64, i64] + [dp] * 9
    lib.ssor_softplus_scalar.restype = ctypes.c_double
    lib.ssor_softplus_scalar.argtypes = [ctypes.c_double]
    lib.ssor_position_of.restype = ctypes.c_int64
    lib.ssor_position_of.argtypes = [ctypes.c_int, i64, i64, i64]
    lib.ssor_dwconv3x3_silu.restype = ctypes.c_int
    lib.ssor_dwconv3x3_silu.argtypes = [i64, i64, i64, i64, dp, dp, dp, dp]
    lib.ssor_order_table.restype = ctypes.c_int
    lib.ssor_order_table.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.POINTER(i64)]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _f64(a, shape, name):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if tuple(a.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(a.shape)}")
    return a


def _ptr(a):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
         orders=(ORDER_FWD,), H=None, W=None, zoh=False, h0=None, win=0, _lib_handle=None):
    """Run the oracle.

    ``delta`` is [batch, K, dim, L] and ``B``/``C`` are [batch, K, G, N, L]; for a
    single direction the K axis may be omitted (``delta`` [batch, dim, L],
    ``B``/``C`` [batch, G, N, L]).  ``H``/``W`` default to 1 x L; ``win`` is the
    window size of the windowed orders.
    Returns ``(out [batch, dim, L], last_state [batch, K, dim, N])`` as float64.
    """
    u = np.asarray(u)
    batch, dim, L = u.shape
    K = len(orders)
    delta = np.asarray(delta)
    B = np.asarray(B)
    C = np.asarray(C)
    if delta.ndim == 3:
        delta = delta[:, None]
    if B.ndim == 4:
        B = B[:, None]
    if C.ndim == 4:
        C = C[:, None]
    G, N = B.shape[2], B.shape[3]
    if H is None and W is None:
        H, W = 1, L
    if H * W != L:
        raise ValueError("H*W must equal L")
    u = _f64(u, (batch, dim, L), "u")
    delta = _f64(delta, (batch, K, dim, L), "delta")
    A = _f64(np.asarray(A).reshape(K * dim, N), (K * dim, N), "A")
    B = _f64(B, (batch, K, G, N, L), "B")
    C = _f64(C, (batch, K, G, N, L), "C")
    D = _f64(None if D is None else np.asarray(D).reshape(K * dim), (K * dim,), "D")
    z = _f64(z, (batch, dim, L), "z")
    delta_bias = _f64(None if delta_bias is None else np.asarray(delta_bias).reshape(K * dim),
                      (K * dim,), "delta_bias")
    h0 = _f64(None if h0 is None else np.asarray(h0).reshape(batch, K, dim, N),
              (batch, K, dim, N), "h0")
    out = np.empty((batch, dim, L), dtype=np.float64)
    last = np.empty((batch, K, dim, N), dtype=np.float64)
    work = np.empty((N,), dtype=np.float64)
    ords = (ctypes.c_int * K)(*[int(o) for o in orders])
    lib = _lib_handle if _lib_handle is not None else _load()
    rc = lib.ssor_scan(batch, dim, H, W, N, G, K, ords, int(win),
                           _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
                           _ptr(delta_bias), int(bool(delta_softplus)), int(bool(zoh)),
                           _ptr(h0), _ptr(out), _ptr(last), _ptr(work))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out, last


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                   zoh=False, h0=None):
    """One forward direction: delta [batch, dim, L], B/C [batch, G, N, L], A [dim, N]."""
    out, last = scan(u, delta, A, B, C, D, z, delta_bias, delta_softplus, (ORDER_FWD,),
                     zoh=zoh, h0=h0)
    return out, last[:, 0]


def bidir_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True):
    """Forward + reversed direction, outputs summed: delta [batch, 2, dim, L]."""
    return scan(u, delta, A, B, C, D, z, delta_bias, delta_softplus, (ORDER_FWD, ORDER_REV))


# The SS2D direction set, in the order the key-code listing stacks them:
# row-major, column-major, reversed row-major, reversed column-major.
SS2D_ORDERS = (ORDER_FWD, ORDER_COL, ORDER_REV, ORDER_COL_REV)


def cross_scan2d(u, delta, A, B, C, H, W, D=None, z=None, delta_bias=None, delta_softplus=True):
    """SS2D: u [batch, dim, H, W]; delta [batch, 4, dim, H*W] and B/C
    [batch, 4, G, N, H*W], each direction in its own scan order."""
    u = np.asarray(u)
    batch, dim = u.shape[:2]
    L = H * W
    delta = np.asarray(delta).reshape(batch, 4, dim, L)
    B = np.asarray(B)
    C = np.asarray(C)
    B = B.reshape(B.shape[0], 4, B.shape[2], B.shape[3], L)
    C = C.reshape(C.shape[0], 4, C.shape[2], C.shape[3], L)
    zz = None if z is None else np.asarray(z).reshape(batch, dim, L)
    out, last = scan(u.reshape(batch, dim, L), delta, A, B, C, D, zz, delta_bias, delta_softplus,
                     SS2D_ORDERS, H=H, W=W)
    return out.reshape(batch, dim, H, W), last


def selective_scan_bwd(u, delta, A, B, C, dy, D=None, z=None, delta_bias=None,
                       delta_softplus=True, zoh=False, h0=None):
    """Gradients of one forward direction for the upstream gradient dy
    [batch, dim, L]: Euler input matrix, or the zero-order hold with zoh; zero
    initial state, or h0 [batch, dim, N].  delta [batch, dim, L], B/C
    [batch, G, N, L], A [dim, N].  Returns a dict of float64 arrays: du, ddelta
    [batch, dim, L]; dA [dim, N]; dB, dC [batch, G, N, L]; dD, ddelta_bias
    [dim] (None when D / delta_bias are None); dz [batch, dim, L] (None
    without z); dh0 [batch, dim, N] (None without h0)."""
    u = _f64(u, np.asarray(u).shape, "u")
    batch, dim, L = u.shape
    G, N = np.asarray(B).shape[1], np.asarray(B).shape[2]
    delta = _f64(delta, (batch, dim, L), "delta")
    A = _f64(A, (dim, N), "A")
    B = _f64(B, (batch, G, N, L), "B")
    C = _f64(C, (batch, G, N, L), "C")
    dy = _f64(dy, (batch, dim, L), "dy")
    D = _f64(D, (dim,), "D")
    z = _f64(z, (batch, dim, L), "z")
    bias = _f64(delta_bias, (dim,), "delta_bias")
    out = {k: np.empty(sh) for k, sh in (("du", u.shape), ("ddelta", u.shape), ("dA", A.shape),
                                          ("dB", B.shape), ("dC", C.shape))}
    out["dD"] = np.empty(dim) if D is not None else None
    out["dz"] = np.empty(u.shape) if z is not None else None
    out["ddelta_bias"] = np.empty(dim) if bias is not None else None
    h0 = _f64(h0, (batch, dim, N), "h0")
    out["dh0"] = np.empty((batch, dim, N)) if h0 is not None else None
    work = np.empty(L * N)
    rc = _load().ssor_scan_bwd_ext(batch, dim, L, N, G, _ptr(u), _ptr(delta), _ptr(A), _ptr(B),
                                   _ptr(C), _ptr(D), _ptr(z), _ptr(bias), int(bool(delta_softplus)),
                                   int(bool(zoh)), _ptr(h0), _ptr(dy), _ptr(out["du"]),
                                   _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]),
                                   _ptr(out["dC"]), _ptr(out["dD"]), _ptr(out["dz"]),
                                   _ptr(out["ddelta_bias"]), _ptr(out["dh0"]), _ptr(work))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out


def multi_scan_bwd(u, delta, A, B, C, dy, orders, H=None, W=None, win=0, D=None, z=None,
                   delta_bias=None, delta_softplus=True):
    """Gradients of :func:`scan` with K directions of any orders for the upstream
    gradient ``dy`` [batch, dim, L] of its output.

    Direction k of the forward pass is the single-direction scan of the inputs
    taken in k's order, u_k[s] = u[pos_k(s)] (Delta_k, B_k, C_k already in that
    order), added into the output at pos_k(s); the gate multiplies the sum.  So
    direction k's gradients are those of :func:`selective_scan_bwd` on its
    permuted inputs with the upstream gradient dy_k[s] = dy[pos_k(s)] and gate
    z_k[s] = z[pos_k(s)] -- except dz, which belongs to the sum:
    dz = dy * s * SiLU'(z) with s the pre-gate output of all directions.  du
    adds every direction's du_k back at its positions.  Shapes as :func:`scan`;
    returns a dict like :func:`selective_scan_bwd`, with ddelta [batch, K, dim,
    L], dA [K*dim, N], dB, dC [batch, K, G, N, L], dD and ddelta_bias [K*dim]."""
    u = np.asarray(u, dtype=np.float64)
    batch, dim, L = u.shape
    K = len(orders)
    if H is None and W is None:
        H, W = 1, L
    delta = np.asarray(delta, dtype=np.float64).reshape(batch, K, dim, L)
    B = np.asarray(B, dtype=np.float64)
    C = np.asarray(C, dtype=np.float64)
    G, N = B.shape[2], B.shape[3]
    A = np.asarray(A, dtype=np.float64).reshape(K, dim, N)
    Dk = None if D is None else np.asarray(D, dtype=np.float64).reshape(K, dim)
    bk = None if delta_bias is None else np.asarray(delta_bias, dtype=np.float64).reshape(K, dim)
    dy = np.asarray(dy, dtype=np.float64)
    zz = None if z is None else np.asarray(z, dtype=np.float64)
    out = {"du": np.zeros_like(u), "ddelta": np.empty((batch, K, dim, L)),
           "dA": np.empty((K * dim, N)), "dB": np.empty((batch, K, G, N, L)),
           "dC": np.empty((batch, K, G, N, L)),
           "dD": None if D is None else np.empty(K * dim),
           "ddelta_bias": None if delta_bias is None else np.empty(K * dim), "dz": None}
    for k, order in enumerate(orders):
        pos = order_table(order, H, W, win)
        g = selective_scan_bwd(u[..., pos], delta[:, k], A[k], B[:, k], C[:, k], dy[..., pos],
                               D=None if Dk is None else Dk[k],
                               z=None if zz is None else zz[..., pos],
                               delta_bias=None if bk is None else bk[k],
                               delta_softplus=delta_softplus)
        out["du"][..., pos] += g["du"]
        out["ddelta"][:, k] = g["ddelta"]
        out["dA"][k * dim:(k + 1) * dim] = g["dA"]
        out["dB"][:, k] = g["dB"]
        out["dC"][:, k] = g["dC"]
        if D is not None:
            out["dD"][k * dim:(k + 1) * dim] = g["dD"]
        if delta_bias is not None:
            out["ddelta_bias"][k * dim:(k + 1) * dim] = g["ddelta_bias"]
    if zz is not None:
        s_total, _ = scan(u, delta, A.reshape(K * dim, N), B, C, D, None, delta_bias,
                          delta_softplus, orders, H=H, W=W, win=win)
        sg = 1.0 / (1.0 + np.exp(-zz))
        out["dz"] = dy * s_total * sg * (1.0 + zz * (1.0 - sg))
    return out


def conv_silu(x, w, bias=None, x0=None):
    """The Mamba block's Conv1D -> SiLU before the scan: x [batch, dim, L],
    w [dim, KW], bias [dim], x0 [batch, dim, KW-1] (inputs before the
    sequence, oldest first; default zeros).  Returns u [batch, dim, L] float64."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    batch, dim, L = x.shape
    w = _f64(w, (dim, np.asarray(w).shape[-1]), "w")
    KW = w.shape[1]
    bias = _f64(bias, (dim,), "bias")
    x0 = _f64(x0, (batch, dim, KW - 1), "x0")
    u = np.empty_like(x)
    rc = _load().ssor_conv_silu(batch, dim, L, KW, _ptr(x), _ptr(w), _ptr(bias), _ptr(x0), _ptr(u))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return u


def conv_silu_bwd(x, w, du, bias=None, x0=None):
    """Gradients of :func:`conv_silu` for the upstream gradient du [batch, dim, L]
    of u.  Returns a dict of float64 arrays: dx [batch, dim, L], dw [dim, KW],
    dbias [dim] (None without bias), dx0 [batch, dim, KW-1] (None without x0)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    batch, dim, L = x.shape
    w = _f64(w, (dim, np.asarray(w).shape[-1]), "w")
    KW = w.shape[1]
    du = _f64(du, (batch, dim, L), "du")
    bias = _f64(bias, (dim,), "bias")
    x0 = _f64(x0, (batch, dim, KW - 1), "x0")
    g = {"dx": np.empty_like(x), "dw": np.empty_like(w),
         "dbias": np.empty(dim) if bias is not None else None,
         "dx0": np.empty((batch, dim, KW - 1)) if x0 is not None else None}
    rc = _load().ssor_conv_silu_bwd(batch, dim, L, KW, _ptr(x), _ptr(w), _ptr(bias), _ptr(x0),
                                    _ptr(du), _ptr(g["dx"]), _ptr(g["dw"]), _ptr(g["dbias"]),
                                    _ptr(g["dx0"]))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return g


def dwconv3x3_silu(x, w, bias=None):
    """The SS2D block's input branch: depthwise 3 x 3 cross-correlation with zero
    padding, plus bias, then SiLU.  x [batch, dim, H, W]; w [dim, 3, 3]; bias
    [dim].  Returns u [batch, dim, H, W] float64."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    batch, dim, H, W = x.shape
    w = _f64(w, (dim, 3, 3), "w")
    bias = _f64(bias, (dim,), "bias")
    u = np.empty_like(x)
    rc = _load().ssor_dwconv3x3_silu(batch, dim, H, W, _ptr(x), _ptr(w), _ptr(bias), _ptr(u))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return u


def softplus(x: float) -> float:
    return _load().ssor_softplus_scalar(float(x))


def position(order: int, s: int, H: int, W: int) -> int:
    return _load().ssor_position_of(int(order), int(s), int(H), int(W))


def order_table(order: int, H: int, W: int, win: int = 0) -> np.ndarray:
    """Positions visited by steps 0 .. H*W-1 of a direction with the given order."""
    pos = np.empty(H * W, dtype=np.int64)
    rc = _load().ssor_order_table(int(order), int(H), int(W), int(win),
                                  pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return pos
