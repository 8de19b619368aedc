"""B300-native selective state-space scan (Mamba S6, Vision Mamba bidirectional,
VMamba SS2D) -- torch-facing wrappers over the C ABI of libssscan.so.

The wrappers check shapes and dtypes, allocate outputs and workspace with
PyTorch, and call the library on the current CUDA stream.  All arithmetic runs
in the library's sm_103a kernels; there is no fallback.

    out = selective_scan_fwd(u, delta, A, B, C, D, z, delta_bias, delta_softplus=True)
    out = bidir_scan_fwd(u, delta2, A2, B2, C2, D2, z, bias2)
    out = cross_scan2d_fwd(u_map, delta4, A4, B4, C4, D4, bias4)
    grads = selective_scan_bwd(u, delta, A, B, C, dout, D, z, delta_bias)
    out = multi_scan_fwd(u_map, deltaK, AK, BK, CK, [DIR_WIN, DIR_WIN_COL], window=7)

u, z and out are indexed by position; each direction's delta, B and C are in
that direction's scan order.
"""
from __future__ import annotations

import ctypes

from . import _binding as _b
from ._binding import SSError, load as load_library, version  # noqa: F401

__all__ = ["selective_scan_fwd", "bidir_scan_fwd", "cross_scan2d_fwd", "selective_state_update",
           "device_status",
           "workspace_bytes", "SSError", "load_library", "version"]


def _torch():
    import torch
    return torch


def _io_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return _b.SS_BF16
    if t.dtype == torch.float32:
        return _b.SS_F32
    raise TypeError(f"I/O tensors must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_io(name, t, dtype, device, shape=None):
    torch = _torch()
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def workspace_bytes(kind: int, batch: int, dim: int, seqlen: int, dstate: int, chunks: int = 0):
    return _b.workspace_bytes(kind, batch, dim, seqlen, dstate, chunks)


def selective_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                       return_last_state=False, out=None, chunks=0, workspace=None, stream=None,
                       h0=None, zoh=False, conv_w=None, conv_b=None, conv_x0=None):
    """One-direction selective scan.

    u, delta, z: [batch, dim, L]; A: [dim, N] float32; B, C: [batch, G, N, L];
    D, delta_bias: [dim] float32.  Returns out [batch, dim, L] (and last_state
    [batch, dim, N] float32 if requested).  ``chunks`` forces the sequence split
    (0 automatic, 1 single pass, n >= 2 chunked path); ``workspace`` is an
    optional preallocated uint8 CUDA tensor; ``h0`` [batch, dim, N] float32 is
    the initial state (default zero); ``zoh`` selects the zero-order-hold input
    matrix instead of the Euler one.  With ``conv_w`` [dim, 4] float32 the
    Mamba block's causal Conv1D + SiLU (bias ``conv_b`` [dim], history
    ``conv_x0`` [batch, dim, 3]) is fused in front of the scan and ``u`` is its
    input."""
    torch = _torch()
    lib = _b.load()
    batch, dim, L = u.shape
    G, N = B.shape[1], B.shape[2]
    io, dev = u.dtype, u.device
    _check_io("u", u, io, dev)
    _check_io("delta", delta, io, dev, (batch, dim, L))
    _check_io("B", B, io, dev, (batch, G, N, L))
    _check_io("C", C, io, dev, (batch, G, N, L))
    _check_io("z", z, io, dev, (batch, dim, L))
    _check_io("A", A, torch.float32, dev, (dim, N))
    _check_io("D", D, torch.float32, dev, (dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (dim,))
    _check_io("h0", h0, torch.float32, dev, (batch, dim, N))
    _check_io("conv_w", conv_w, torch.float32, dev, (dim, 4))
    _check_io("conv_b", conv_b, torch.float32, dev, (dim,))
    _check_io("conv_x0", conv_x0, torch.float32, dev, (batch, dim, 3))
    if out is None:
        out = torch.empty_like(u)
    _check_io("out", out, io, dev, (batch, dim, L))
    last = torch.empty(batch, dim, N, dtype=torch.float32, device=dev) if return_last_state else None
    flags = (_b.SS_SCAN_ZOH if zoh else 0) | (_b.SS_SCAN_CONV_SILU if conv_w is not None else 0)
    opts = _b.options(chunks, flags, _ptr(h0), _ptr(conv_w), _ptr(conv_b), _ptr(conv_x0))
    wsb = int(lib.ss_workspace_bytes_opts(_b.SS_KIND_SCAN, batch, dim, L, N, ctypes.byref(opts)))
    if wsb and (workspace is None or workspace.numel() < wsb):
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ws_ptr = _ptr(workspace) if wsb else None
    ws_len = workspace.numel() if wsb else 0
    _b.check(lib.ss_selective_scan_fwd_opts(
        batch, dim, L, N, G, _io_code(u), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(out), _ptr(last),
        ws_ptr, ws_len, ctypes.byref(opts), _stream(stream, dev)))
    return (out, last) if return_last_state else out


def selective_scan_bwd(u, delta, A, B, C, dout, D=None, z=None, delta_bias=None,
                       delta_softplus=True, workspace=None, stream=None, h0=None, zoh=False,
                       conv_w=None, conv_b=None, conv_x0=None):
    """Gradients of :func:`selective_scan_fwd` for the upstream gradient
    ``dout`` [batch, dim, L] of its output, with the forward call's options
    (``h0``, ``zoh``, and the fused Conv1D ``conv_w``, ``conv_b``, ``conv_x0``,
    ``u`` then being the convolution's input).

    Returns a dict: du, ddelta [batch, dim, L] and dz (None without z) in the
    I/O dtype; dA [dim, N], dB, dC [batch, G, N, L], dD (None without D) and
    ddelta_bias (None without delta_bias) in float32; with the options also dh0
    [batch, dim, N] (given h0), dconv_w [dim, 4], dconv_b [dim] and dconv_x0
    [batch, dim, 3] (each given its tensor) in float32.  ``workspace`` is an
    optional preallocated uint8 CUDA tensor (state checkpoints; with the Conv1D
    also the recomputed u and its gradient)."""
    torch = _torch()
    lib = _b.load()
    batch, dim, L = u.shape
    G, N = B.shape[1], B.shape[2]
    io, dev = u.dtype, u.device
    _check_io("u", u, io, dev)
    for name, t in (("delta", delta), ("z", z), ("dout", dout)):
        _check_io(name, t, io, dev, (batch, dim, L))
    _check_io("B", B, io, dev, (batch, G, N, L))
    _check_io("C", C, io, dev, (batch, G, N, L))
    _check_io("A", A, torch.float32, dev, (dim, N))
    _check_io("D", D, torch.float32, dev, (dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (dim,))
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(u),
         "dz": torch.empty_like(u) if z is not None else None,
         "dA": torch.empty(dim, N, **f32), "dB": torch.empty(batch, G, N, L, **f32),
         "dC": torch.empty(batch, G, N, L, **f32),
         "dD": torch.empty(dim, **f32) if D is not None else None,
         "ddelta_bias": torch.empty(dim, **f32) if delta_bias is not None else None}
    _check_io("h0", h0, torch.float32, dev, (batch, dim, N))
    _check_io("conv_w", conv_w, torch.float32, dev, (dim, 4))
    _check_io("conv_b", conv_b, torch.float32, dev, (dim,))
    _check_io("conv_x0", conv_x0, torch.float32, dev, (batch, dim, 3))
    flags = (_b.SS_SCAN_ZOH if zoh else 0) | (_b.SS_SCAN_CONV_SILU if conv_w is not None else 0)
    opts = _b.options(0, flags, _ptr(h0), _ptr(conv_w), _ptr(conv_b), _ptr(conv_x0))
    g["dh0"] = torch.empty(batch, dim, N, **f32) if h0 is not None else None
    g["dconv_w"] = torch.empty(dim, 4, **f32) if conv_w is not None else None
    g["dconv_b"] = torch.empty(dim, **f32) if conv_b is not None else None
    g["dconv_x0"] = torch.empty(batch, dim, 3, **f32) if conv_x0 is not None else None
    ext = _b.BwdExtras()
    ext.dh0, ext.dconv_w = _ptr(g["dh0"]), _ptr(g["dconv_w"])
    ext.dconv_b, ext.dconv_x0 = _ptr(g["dconv_b"]), _ptr(g["dconv_x0"])
    wsb = int(lib.ss_workspace_bytes_opts(_b.SS_KIND_SCAN_BWD, batch, dim, L, N, ctypes.byref(opts)))
    if wsb and (workspace is None or workspace.numel() < wsb):
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    _b.check(lib.ss_selective_scan_bwd_opts(
        batch, dim, L, N, G, _io_code(u), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(dout),
        _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
        _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]), ctypes.byref(opts),
        ctypes.byref(ext), _ptr(workspace) if wsb else None, workspace.numel() if wsb else 0,
        _stream(stream, dev)))
    return g


def multi_scan_fwd(u, delta, A, B, C, orders, window=0, D=None, delta_bias=None,
                   delta_softplus=True, z=None, return_last_state=False, out=None,
                   workspace=None, stream=None):
    """Directions of any traversal over an H x W map, summed by position and gated.

    u, z: [batch, dim, H, W]; delta: [batch, K, dim, H*W] and B, C: [batch, K, G,
    N, H*W], each direction's in its own scan order; A: [K*dim, N]; D,
    delta_bias: [K*dim].  ``orders`` lists K SS_DIR_* codes (DIR_* below);
    ``window`` is the window size of the windowed ones.  Returns out [batch,
    dim, H, W] (and last_state [batch, K, dim, N])."""
    torch = _torch()
    lib = _b.load()
    batch, dim, H, W = u.shape
    K = len(orders)
    G, N = B.shape[2], B.shape[3]
    L = H * W
    io, dev = u.dtype, u.device
    _check_io("u", u, io, dev)
    _check_io("z", z, io, dev, (batch, dim, H, W))
    _check_io("delta", delta, io, dev, (batch, K, dim, L))
    _check_io("B", B, io, dev, (batch, K, G, N, L))
    _check_io("C", C, io, dev, (batch, K, G, N, L))
    _check_io("A", A, torch.float32, dev, (K * dim, N))
    _check_io("D", D, torch.float32, dev, (K * dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (K * dim,))
    if out is None:
        out = torch.empty_like(u)
    _check_io("out", out, io, dev, (batch, dim, H, W))
    last = (torch.empty(batch, K, dim, N, dtype=torch.float32, device=dev)
            if return_last_state else None)
    wsb = int(lib.ss_multi_scan_workspace_bytes(batch, dim, H, W, K))
    if wsb and (workspace is None or workspace.numel() < wsb):
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ords = (ctypes.c_int * K)(*[int(o) for o in orders])
    _b.check(lib.ss_multi_scan_fwd(
        batch, dim, H, W, K, ords, int(window), N, G, _io_code(u), _ptr(u), _ptr(delta), _ptr(A),
        _ptr(B), _ptr(C), _ptr(D), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(z), _ptr(out),
        _ptr(last), _ptr(workspace) if wsb else None, workspace.numel() if wsb else 0,
        _stream(stream, dev)))
    return (out, last) if return_last_state else out


from ._binding import (SS_DIR_COL as DIR_COL, SS_DIR_COL_REV as DIR_COL_REV,  # noqa: E402
                       SS_DIR_ROW as DIR_ROW, SS_DIR_ROW_REV as DIR_ROW_REV,
                       SS_DIR_WIN as DIR_WIN, SS_DIR_WIN_COL as DIR_WIN_COL,
                       SS_DIR_WIN_COL_REV as DIR_WIN_COL_REV, SS_DIR_WIN_REV as DIR_WIN_REV)


def multi_scan_bwd(u, delta, A, B, C, dout, orders, window=0, D=None, delta_bias=None,
                   delta_softplus=True, z=None, workspace=None, stream=None):
    """Gradients of :func:`multi_scan_fwd` for the upstream gradient ``dout``
    [batch, dim, H, W].  Returns a dict: du, dz (None without z) [batch, dim, H,
    W] and ddelta [batch, K, dim, H*W] in the I/O dtype; dA [K*dim, N], dB, dC
    [batch, K, G, N, H*W], dD and ddelta_bias [K*dim] (None when not given) in
    float32."""
    torch = _torch()
    lib = _b.load()
    batch, dim, H, W = u.shape
    K = len(orders)
    G, N = B.shape[2], B.shape[3]
    L = H * W
    io, dev = u.dtype, u.device
    _check_io("u", u, io, dev)
    _check_io("z", z, io, dev, (batch, dim, H, W))
    _check_io("dout", dout, io, dev, (batch, dim, H, W))
    _check_io("delta", delta, io, dev, (batch, K, dim, L))
    _check_io("B", B, io, dev, (batch, K, G, N, L))
    _check_io("C", C, io, dev, (batch, K, G, N, L))
    _check_io("A", A, torch.float32, dev, (K * dim, N))
    _check_io("D", D, torch.float32, dev, (K * dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (K * dim,))
    f32 = dict(dtype=torch.float32, device=dev)
    g = {"du": torch.empty_like(u), "ddelta": torch.empty_like(delta),
         "dz": torch.empty_like(u) if z is not None else None,
         "dA": torch.empty(K * dim, N, **f32), "dB": torch.empty(batch, K, G, N, L, **f32),
         "dC": torch.empty(batch, K, G, N, L, **f32),
         "dD": torch.empty(K * dim, **f32) if D is not None else None,
         "ddelta_bias": torch.empty(K * dim, **f32) if delta_bias is not None else None}
    wsb = int(lib.ss_multi_scan_bwd_workspace_bytes(batch, dim, H, W, N, K))
    if wsb and (workspace is None or workspace.numel() < wsb):
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    ords = (ctypes.c_int * K)(*[int(o) for o in orders])
    _b.check(lib.ss_multi_scan_bwd(
        batch, dim, H, W, K, ords, int(window), N, G, _io_code(u), _ptr(u), _ptr(delta), _ptr(A),
        _ptr(B), _ptr(C), _ptr(D), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(z), _ptr(dout),
        _ptr(g["du"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]), _ptr(g["dD"]),
        _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(workspace) if wsb else None,
        workspace.numel() if wsb else 0, _stream(stream, dev)))
    return g


def dwconv3x3_silu(x, w, bias=None, out=None, stream=None):
    """SS2D's input branch: depthwise 3 x 3 convolution (zero padding) + bias, then
    SiLU.  x [batch, dim, H, W] (bf16 or f32); w [dim, 3, 3] and bias [dim]
    float32.  Returns u like x."""
    torch = _torch()
    lib = _b.load()
    batch, dim, H, W = x.shape
    dev = x.device
    _check_io("x", x, x.dtype, dev)
    _check_io("w", w, torch.float32, dev, (dim, 3, 3))
    _check_io("bias", bias, torch.float32, dev, (dim,))
    if out is None:
        out = torch.empty_like(x)
    _check_io("out", out, x.dtype, dev, tuple(x.shape))
    _b.check(lib.ss_dwconv3x3_silu_fwd(batch, dim, H, W, _io_code(x), _ptr(x), _ptr(w), _ptr(bias),
                                       _ptr(out), _stream(stream, dev)))
    return out


def _multidir_workspace(lib, kind, batch, dim, L, N, dev, workspace):
    torch = _torch()
    wsb = int(lib.ss_workspace_bytes(kind, batch, dim, L, N))
    if wsb and (workspace is None or workspace.numel() < wsb):
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    return (_ptr(workspace), workspace.numel()) if wsb else (None, 0)


def bidir_scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                   return_last_state=False, out=None, workspace=None, stream=None):
    """Bidirectional scan: delta [batch, 2, dim, L] and B, C [batch, 2, G, N, L], the
    reversed direction (index 1) in its own scan order (its step s is token L-1-s);
    A [2*dim, N]; D, delta_bias [2*dim].  Returns out [batch, dim, L] (and
    last_state [batch, 2, dim, N])."""
    torch = _torch()
    lib = _b.load()
    batch, dim, L = u.shape
    G, N = B.shape[2], B.shape[3]
    io, dev = u.dtype, u.device
    _check_io("u", u, io, dev)
    _check_io("delta", delta, io, dev, (batch, 2, dim, L))
    _check_io("B", B, io, dev, (batch, 2, G, N, L))
    _check_io("C", C, io, dev, (batch, 2, G, N, L))
    _check_io("z", z, io, dev, (batch, dim, L))
    _check_io("A", A, torch.float32, dev, (2 * dim, N))
    _check_io("D", D, torch.float32, dev, (2 * dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (2 * dim,))
    if out is None:
        out = torch.empty_like(u)
    _check_io("out", out, io, dev, (batch, dim, L))
    last = torch.empty(batch, 2, dim, N, dtype=torch.float32, device=dev) if return_last_state else None
    ws, wsb = _multidir_workspace(lib, _b.SS_KIND_BIDIR, batch, dim, L, N, dev, workspace)
    _b.check(lib.ss_bidir_scan_fwd(
        batch, dim, L, N, G, _io_code(u), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(out), _ptr(last),
        ws, wsb, _stream(stream, dev)))
    return (out, last) if return_last_state else out


def cross_scan2d_fwd(u, delta, A, B, C, D=None, delta_bias=None, delta_softplus=True, z=None,
                     return_last_state=False, out=None, workspace=None, stream=None):
    """SS2D: u [batch, dim, H, W]; delta [batch, 4, dim, H*W] and B, C
    [batch, 4, G, N, H*W], each direction in its own scan order (row-major,
    column-major, reversed row-major, reversed column-major); A [4*dim, N];
    D, delta_bias [4*dim].  Returns out [batch, dim, H, W] (and last_state
    [batch, 4, dim, N])."""
    torch = _torch()
    lib = _b.load()
    batch, dim, H, W = u.shape
    G, N = B.shape[2], B.shape[3]
    io, dev = u.dtype, u.device
    _check_io("u", u, io, dev)
    _check_io("delta", delta, io, dev, (batch, 4, dim, H * W))
    _check_io("B", B, io, dev, (batch, 4, G, N, H * W))
    _check_io("C", C, io, dev, (batch, 4, G, N, H * W))
    _check_io("z", z, io, dev, (batch, dim, H, W))
    _check_io("A", A, torch.float32, dev, (4 * dim, N))
    _check_io("D", D, torch.float32, dev, (4 * dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (4 * dim,))
    if out is None:
        out = torch.empty_like(u)
    _check_io("out", out, io, dev, (batch, dim, H, W))
    last = torch.empty(batch, 4, dim, N, dtype=torch.float32, device=dev) if return_last_state else None
    ws, wsb = _multidir_workspace(lib, _b.SS_KIND_CROSS2D, batch, dim, H * W, N, dev, workspace)
    _b.check(lib.ss_cross_scan2d_fwd(
        batch, dim, H, W, N, G, _io_code(u), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
        _ptr(D), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(z), _ptr(out), _ptr(last),
        ws, wsb, _stream(stream, dev)))
    return (out, last) if return_last_state else out


def selective_state_update(x, delta, A, B, C, state, D=None, z=None, delta_bias=None,
                           delta_softplus=True, zoh=False, out=None, stream=None):
    """One recurrence step for token-by-token inference, updating ``state`` in place.

    x, delta, z: [batch, dim]; A: [dim, N] float32; B, C: [batch, G, N];
    D, delta_bias: [dim] float32; state: [batch, dim, N] float32.  Returns out
    [batch, dim]."""
    torch = _torch()
    lib = _b.load()
    batch, dim = x.shape
    G, N = B.shape[1], B.shape[2]
    io, dev = x.dtype, x.device
    _check_io("x", x, io, dev)
    _check_io("delta", delta, io, dev, (batch, dim))
    _check_io("B", B, io, dev, (batch, G, N))
    _check_io("C", C, io, dev, (batch, G, N))
    _check_io("z", z, io, dev, (batch, dim))
    _check_io("A", A, torch.float32, dev, (dim, N))
    _check_io("D", D, torch.float32, dev, (dim,))
    _check_io("delta_bias", delta_bias, torch.float32, dev, (dim,))
    _check_io("state", state, torch.float32, dev, (batch, dim, N))
    if out is None:
        out = torch.empty_like(x)
    _check_io("out", out, io, dev, (batch, dim))
    _b.check(lib.ss_selective_state_update(
        batch, dim, N, G, _io_code(x), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
        _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _b.SS_SCAN_ZOH if zoh else 0,
        _ptr(state), _ptr(out), _stream(stream, dev)))
    return out


def device_status(stream=None) -> None:
    """Synchronises the stream and raises SSError if a kernel abandoned a bounded wait."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    _b.check(_b.load().ss_get_device_status(_stream(stream, dev)))
