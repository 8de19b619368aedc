"""GPU parity at the edges of the Delta preparation, on every forward entry point.

The step size is Delta' = softplus(Delta + b_Delta), or Delta + b_Delta when the
flag is off ("Mamba Series from Selective State Spaces to Visual State Space
Models", mathematical form of the selective SSM: Delta = softplus(W_Delta x +
b_Delta); key code: delta_bias, delta_softplus).  The seeded workloads keep the
softplus argument in about [-7, -2], so these cases move it elsewhere:

  softplus_off   flag off, Delta > 0 and b_Delta = dt0 > 0 (Delta' = Delta + b_Delta)
  no_bias        flag on, delta_bias NULL (Delta' = softplus(Delta))
  no_bias_off    flag off, delta_bias NULL, Delta > 0 (Delta' = Delta)
  large          flag on, b_Delta from 12 to 22 across channels: the softplus
                 argument crosses the kernels' x > 15 cut-off, and
                 exp(Delta' A) is about 0, the memoryless limit of the formulas
                 (the state is reset at every step; same page, core insight 1)
  zero           flag off, Delta = 0, b_Delta = 0: Abar = 1 and Bbar = 0, so the
                 state stays 0 and out = D*u*SiLU(z) exactly

Each case runs through the direct and the chunked single-direction scan, the
unaligned-row path, the no-allocation entry point, both bidirectional paths
(aligned L = 256, unaligned L = 197), both SS2D paths (aligned 8 x 16, unaligned
6 x 10), the any-order scan (windowed orders) and the one-step decode, and is
compared element by element with the float64 oracle on the same inputs:
max |y - y_ref| / (1 + |y_ref|) <= 1e-4 (float32 I/O) or 2e-2 (bf16 I/O), and
last_state to the same bound (exactly 0 in the zero case).
"""
import ctypes

import numpy as np
import pytest

from selective_state_space_120_b300 import workloads as wk
from tests import scan_cases as sc

pytestmark = pytest.mark.gpu

MODES = ["softplus_off", "no_bias", "no_bias_off", "large", "zero"]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_120_b300 as ss
    ss.load_library()


def _set_delta(inp, fn):
    """Applies fn to the raw Delta values (float64) and stores them back in the
    workload's I/O representation."""
    v = fn(inp.as_f64("delta"))
    if inp.delta.dtype == np.uint16:
        inp.delta[...] = wk.round_bf16_bits(v.astype(np.float32))
    else:
        inp.delta[...] = v.astype(np.float32)


def apply_mode(inp, mode):
    """Edits the inputs for one edge case; returns (softplus flag, with_bias)."""
    if mode == "softplus_off":
        _set_delta(inp, np.abs)
        inp.delta_bias[...] = np.log1p(np.exp(inp.delta_bias.astype(np.float64))).astype(np.float32)
        return False, True
    if mode == "no_bias":
        return True, False
    if mode == "no_bias_off":
        _set_delta(inp, np.abs)
        return False, False
    if mode == "large":
        n = inp.delta_bias.size
        inp.delta_bias[...] = np.linspace(12.0, 22.0, n, dtype=np.float32)
        return True, True
    if mode == "zero":
        _set_delta(inp, np.zeros_like)
        inp.delta_bias[...] = 0.0
        return False, True
    raise ValueError(mode)


def _compare(mode, io, out, last, ref, ref_last):
    sc.assert_close(out, ref, io)
    got_last = np.asarray(last, dtype=np.float64)
    sc.assert_close(got_last, ref_last, io, "last_state")
    if mode == "zero":
        assert np.all(got_last == 0.0), "the state must stay exactly zero"


def _case(oracle, wl, mode, chunks=0):
    inp = wk.make_inputs(wl, seed=2)
    softplus, with_bias = apply_mode(inp, mode)
    out, last = sc.gpu_run(inp, chunks=chunks, softplus=softplus, with_bias=with_bias)
    ref, ref_last = sc.oracle_run(oracle, inp, softplus=softplus, with_bias=with_bias)
    if wl.K == 1:
        ref_last = ref_last[:, 0]
    _compare(mode, wl.io, sc.from_torch(out), last.cpu().numpy(), ref, ref_last)
    if mode == "zero":
        u, z, D = inp.as_f64("u"), inp.as_f64("z"), inp.as_f64("D")
        dsum = D.reshape(wl.K, wl.dim).sum(axis=0)[None, :, None]
        want = dsum * u * (z / (1.0 + np.exp(-z)) if z is not None else 1.0)
        sc.assert_close(sc.from_torch(out), want, wl.io, "D*u*SiLU(z)")


# ---------------------------------------------------------------- single direction
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_direct(oracle, mode, io):
    _case(oracle, sc.workload("edge_direct", 2, 40, 256, io=io), mode, chunks=1)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_chunked(oracle, mode, io):
    _case(oracle, sc.workload("edge_chunked", 1, 24, 1200, io=io), mode, chunks=3)


@pytest.mark.parametrize("mode", MODES)
def test_scan_unaligned_rows(oracle, mode):
    _case(oracle, sc.workload("edge_unaligned", 2, 20, 197), mode)


@pytest.mark.parametrize("mode", MODES)
def test_scan_noalloc(oracle, mode):
    import torch
    from selective_state_space_120_b300 import _binding as b
    lib = b.load()
    wl = sc.workload("edge_noalloc", 1, 24, 1200)
    inp = wk.make_inputs(wl, seed=2)
    softplus, with_bias = apply_mode(inp, mode)
    t = sc.device_inputs(inp)
    out = torch.empty_like(t["u"])
    last = torch.empty(wl.batch, wl.dim, wl.N, dtype=torch.float32, device="cuda")
    opts = b.options(3)
    bias = t["delta_bias"] if with_bias else None
    b.check(lib.ss_selective_scan_fwd_noalloc(
        wl.batch, wl.dim, wl.L, wl.N, wl.G, b.SS_BF16, t["u"].data_ptr(),
        t["delta"][:, 0].contiguous().data_ptr(), t["A"].data_ptr(),
        t["B"][:, 0].contiguous().data_ptr(), t["C"][:, 0].contiguous().data_ptr(),
        t["D"].data_ptr(), t["z"].data_ptr(), None if bias is None else bias.data_ptr(),
        int(softplus), out.data_ptr(), last.data_ptr(), ctypes.byref(opts),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp, softplus=softplus, with_bias=with_bias)
    _compare(mode, wl.io, sc.from_torch(out), last.cpu().numpy(), ref, ref_last[:, 0])


@pytest.mark.parametrize("mode", MODES)
def test_scan_zero_order_hold(oracle, mode):
    """The zero-order-hold input matrix under the same edges (Delta' = 0 gives
    Bbar = 0 there too)."""
    wl = sc.workload("edge_zoh", 2, 24, 512, io="f32")
    inp = wk.make_inputs(wl, seed=2)
    softplus, with_bias = apply_mode(inp, mode)
    out, last = sc.gpu_run(inp, softplus=softplus, with_bias=with_bias, zoh=True)
    ref, ref_last = sc.oracle_run(oracle, inp, softplus=softplus, with_bias=with_bias, zoh=True)
    _compare(mode, wl.io, sc.from_torch(out), last.cpu().numpy(), ref, ref_last[:, 0])


# ---------------------------------------------------------------- multi-direction
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("L", [256, 197])
def test_bidirectional(oracle, mode, L):
    _case(oracle, sc.workload("edge_bidir", 2, 24, L, K=2), mode)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("H,W,io", [(8, 16, "f32"), (8, 16, "bf16"), (6, 10, "bf16")])
def test_cross_scan2d(oracle, mode, H, W, io):
    """8 x 16 rows are 16-byte aligned (the TMA path); 6 x 10 bf16 rows are not
    (the on-chip merge path)."""
    _case(oracle, sc.workload("edge_ss2d", 2, 12, H * W, K=4, io=io, with_z=False, H=H, W=W), mode)


@pytest.mark.parametrize("mode", MODES)
def test_any_order_windowed(oracle, mode):
    import selective_state_space_120_b300 as ss
    H, W, win, batch, dim = 8, 12, 3, 2, 24
    orders = [ss.DIR_WIN, ss.DIR_WIN_COL, ss.DIR_WIN_REV, ss.DIR_WIN_COL_REV]
    wl = sc.workload("edge_win", batch, dim, H * W, K=4, H=H, W=W)
    inp = wk.make_inputs(wl, seed=2)
    softplus, with_bias = apply_mode(inp, mode)
    t = sc.device_inputs(inp)
    out, last = ss.multi_scan_fwd(t["u"].view(batch, dim, H, W), t["delta"], t["A"], t["B"],
                                  t["C"], orders, win, t["D"],
                                  t["delta_bias"] if with_bias else None, softplus,
                                  z=t["z"].view(batch, dim, H, W), return_last_state=True)
    ref, ref_last = oracle.scan(inp.as_f64("u"), inp.as_f64("delta"), inp.as_f64("A"),
                                inp.as_f64("B"), inp.as_f64("C"), inp.as_f64("D"), inp.as_f64("z"),
                                inp.as_f64("delta_bias") if with_bias else None, softplus,
                                [oracle.ORDER_WIN, oracle.ORDER_WIN_COL, oracle.ORDER_WIN_REV,
                                 oracle.ORDER_WIN_COL_REV], H=H, W=W, win=win)
    _compare(mode, wl.io, sc.from_torch(out).reshape(batch, dim, H * W), last.cpu().numpy(),
             ref, ref_last)


# ---------------------------------------------------------------- one-step decode
@pytest.mark.parametrize("mode", MODES)
def test_state_update(oracle, mode):
    """One decode step from a random state (the zero case then keeps the state
    unchanged instead of zero)."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("edge_step", 3, 40, 1, io="f32")
    inp = wk.make_inputs(wl, seed=2)
    softplus, with_bias = apply_mode(inp, mode)
    h0 = (np.random.default_rng(5).standard_normal((wl.batch, wl.dim, wl.N)) * 0.5).astype(np.float32)
    t = sc.device_inputs(inp)
    state = sc.to_torch(h0).clone()
    out = ss.selective_state_update(t["u"][:, :, 0].contiguous(), t["delta"][:, 0, :, 0].contiguous(),
                                    t["A"], t["B"][:, 0, :, :, 0].contiguous(),
                                    t["C"][:, 0, :, :, 0].contiguous(), state, t["D"],
                                    t["z"][:, :, 0].contiguous(),
                                    t["delta_bias"] if with_bias else None, softplus)
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp, h0=h0, softplus=softplus, with_bias=with_bias)
    sc.assert_close(sc.from_torch(out), ref[:, :, 0], wl.io)
    got = state.cpu().numpy().astype(np.float64)
    sc.assert_close(got, ref_last[:, 0], wl.io, "state")
    if mode == "zero":
        assert np.array_equal(got, h0.astype(np.float64)), "Abar = 1, Bbar = 0: state unchanged"
