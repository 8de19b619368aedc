"""Shared helpers of the GPU parity tests: build seeded inputs, run the library
and the oracle on the same bits, and compare with the tolerance of the I/O
dtype.  Tolerances: max |y - y_ref| / (1 + |y_ref|) <= 1e-4 for float32 I/O and
<= 2e-2 for bfloat16 I/O; last_state (always float32) to the same bound."""
from __future__ import annotations

import numpy as np

from selective_state_space_120_b300 import workloads as wk

TOL = {"f32": 1e-4, "bf16": 2e-2}


def to_torch(a, device="cuda"):
    import torch
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def from_torch(t):
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def rel_err(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if got.size == 0:
        return 0.0
    assert np.all(np.isfinite(got)), "non-finite output"
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def assert_close(got, ref, io, what="out"):
    e = rel_err(got, ref)
    assert e <= TOL[io], f"{what}: max relative error {e:.3e} > {TOL[io]:.0e}"
    return e


def workload(name, batch, dim, L, N=16, G=1, K=1, io="bf16", with_z=True, with_D=True,
             H=1, W=0):
    return wk.Workload(name, batch, dim, L, N=N, G=G, K=K, io=io, with_z=with_z, with_D=with_D,
                       last_state=True, H=H, W=W)


def oracle_run(oracle, inp, rows=None, h0=None, zoh=False, softplus=True, with_bias=True):
    """Oracle output for the whole workload, or for a list of (b, d) rows.
    Returns (out [batch | len(rows), dim | -, L], last [.., K, .., N]).
    ``softplus`` is the delta_softplus flag; ``with_bias=False`` passes no
    delta_bias (zero)."""
    wl = inp.wl
    K = wl.K
    u, dl, A, B, C = (inp.as_f64(n) for n in ("u", "delta", "A", "B", "C"))
    D, z = inp.as_f64("D"), inp.as_f64("z")
    bias = inp.as_f64("delta_bias") if with_bias else None
    orders = {1: (oracle.ORDER_FWD,), 2: (oracle.ORDER_FWD, oracle.ORDER_REV),
              4: oracle.SS2D_ORDERS}[K]
    H, W = (wl.H, wl.W) if K == 4 else (1, wl.L)
    if rows is None:
        return oracle.scan(u, dl, A, B, C, D, z, bias, softplus, orders, H=H, W=W, zoh=zoh,
                           h0=None if h0 is None else np.asarray(h0, np.float64)[:, None])
    outs, lasts = [], []
    dpg = wl.dim // wl.G
    for (b, d) in rows:
        g = d // dpg
        sel = [k * wl.dim + d for k in range(K)]
        o, l = oracle.scan(u[b:b + 1, d:d + 1], dl[b:b + 1, :, d:d + 1], A[sel],
                           B[b:b + 1, :, g:g + 1], C[b:b + 1, :, g:g + 1],
                           None if D is None else D[sel],
                           None if z is None else z[b:b + 1, d:d + 1],
                           None if bias is None else bias[sel], softplus, orders, H=H, W=W)
        outs.append(o[0, 0])
        lasts.append(l[0, :, 0])
    return np.stack(outs), np.stack(lasts)


def device_inputs(inp):
    return {n: to_torch(getattr(inp, n)) for n in ("u", "delta", "A", "B", "C", "D", "z",
                                                   "delta_bias")}


def gpu_run(inp, chunks=0, t=None, h0=None, zoh=False, softplus=True, with_bias=True):
    """Runs the library on the workload; returns (out, last_state) as torch tensors.
    ``softplus`` is the delta_softplus flag; ``with_bias=False`` passes no
    delta_bias (NULL)."""
    import selective_state_space_120_b300 as ss
    wl = inp.wl
    t = t or device_inputs(inp)
    bias = t["delta_bias"] if with_bias else None
    if wl.K == 1:
        return ss.selective_scan_fwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                                     t["D"], t["z"], bias, softplus,
                                     return_last_state=True, chunks=chunks,
                                     h0=None if h0 is None else to_torch(h0), zoh=zoh)
    if wl.K == 2:
        return ss.bidir_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                 bias, softplus, return_last_state=True)
    H, W = wl.H, wl.W
    bsz, dim, L = t["u"].shape
    G, N = t["B"].shape[2], t["B"].shape[3]
    out, last = ss.cross_scan2d_fwd(t["u"].view(bsz, dim, H, W), t["delta"],
                                    t["A"], t["B"], t["C"], t["D"], bias, softplus,
                                    z=None if t["z"] is None else t["z"].view(bsz, dim, H, W),
                                    return_last_state=True)
    return out.view(bsz, dim, L), last
