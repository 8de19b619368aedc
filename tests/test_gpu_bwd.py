"""GPU parity of the backward pass: ss_selective_scan_bwd against the float64
oracle's gradients (oracle.selective_scan_bwd), on the same seeded inputs and
upstream gradient (B300 only).

Tolerance.  Each gradient tensor g with float64 reference r must satisfy
    max |g - r| / (rms(r) + |r|) <= 1e-3 (float32 I/O) or 1e-2 (bf16 I/O).
The float32 arithmetic follows chains of up to 1/(Delta' |A|) ~ 1000 steps
(Delta' >= 1e-3 in the workload recipe, |A| >= 1), along which the relative
error of the hardware exponential (about 2^-22) compounds to ~2.4e-4; the
bf16 outputs (du, ddelta, dz) add their rounding of 2^-9.  dA, dB, dC, dD and
ddelta_bias are sums with cancellation over batch, time or channels, so the
scale is the tensor's rms rather than 1.
"""
import numpy as np
import pytest

from selective_state_space_120_b300 import workloads as wk
from tests import scan_cases as sc

pytestmark = pytest.mark.gpu

TOL_BWD = {"f32": 1e-3, "bf16": 1e-2}
NAMES = ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_120_b300 as ss
    ss.load_library()


def _dout_f64(wl, dout):
    return (wk.bf16_bits_to_f32(dout) if wl.io == "bf16" else dout).astype(np.float64)


def gpu_bwd(inp, dout, use_D=True, use_z=True, use_bias=True, softplus=True, workspace=None):
    import selective_state_space_120_b300 as ss
    t = sc.device_inputs(inp)
    g = ss.selective_scan_bwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                              sc.to_torch(dout), t["D"] if use_D else None,
                              t["z"] if use_z else None,
                              t["delta_bias"] if use_bias else None, softplus,
                              workspace=workspace)
    return {k: (None if v is None else sc.from_torch(v)) for k, v in g.items()}


def oracle_bwd(oracle, inp, dout, use_D=True, use_z=True, use_bias=True, softplus=True):
    return oracle.selective_scan_bwd(
        inp.as_f64("u"), inp.as_f64("delta")[:, 0], inp.as_f64("A"), inp.as_f64("B")[:, 0],
        inp.as_f64("C")[:, 0], _dout_f64(inp.wl, dout),
        D=inp.as_f64("D") if use_D else None, z=inp.as_f64("z") if use_z else None,
        delta_bias=inp.as_f64("delta_bias") if use_bias else None, delta_softplus=softplus)


def grad_err(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite gradient"
    scale = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    den = scale + np.abs(ref)
    diff = np.abs(got - ref)
    if not np.any(den > 0):
        return float(np.max(diff)) if diff.size else 0.0
    return float(np.max(np.where(den > 0, diff / np.where(den > 0, den, 1.0), diff)))


def assert_grads(got, ref, io, names=NAMES):
    errs = {}
    for k in names:
        if ref[k] is None:
            assert got[k] is None, k
            continue
        e = grad_err(got[k], ref[k])
        errs[k] = e
        assert e <= TOL_BWD[io], f"{k}: error {e:.3e} > {TOL_BWD[io]:.0e} (errors so far {errs})"
    return errs


def _check(oracle, wl, **kw):
    inp = wk.make_inputs(wl, seed=0)
    dout = wk.make_dout(wl, seed=0)
    return assert_grads(gpu_bwd(inp, dout, **kw), oracle_bwd(oracle, inp, dout, **kw), wl.io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 32, 64])
def test_bwd_all_dstates(oracle, io, N):
    """Several channel blocks (the last one partly empty) and a ragged last
    tile and checkpoint block (200 = 6 * 32 + 8 = 12 * 16 + 8 steps)."""
    _check(oracle, sc.workload(f"bn{N}", 2, 40, 200, N=N, io=io))


@pytest.mark.parametrize("L", [8, 16, 32, 48, 520])
def test_bwd_lengths(oracle, L):
    """Shorter than one tile, exactly one checkpoint block, one tile, and a
    tail past the last checkpoint; groups of 18 channels sharing B and C."""
    _check(oracle, sc.workload(f"bl{L}", 2, 36, L, G=2))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_without_gate_skip_bias(oracle, io):
    wl = sc.workload(f"bopt_{io}", 2, 24, 136, io=io)
    _check(oracle, wl, use_z=False)
    _check(oracle, wl, use_D=False)
    _check(oracle, wl, use_bias=False)


def test_bwd_softplus_off(oracle):
    """Without the softplus (and without a bias) Delta' is delta itself, and
    ddelta = dDelta'."""
    wl = sc.workload("bsp", 1, 20, 96, io="f32")
    inp = wk.make_inputs(wl, seed=3)
    # without softplus and bias Delta' is delta itself: keep it positive, so
    # that Abar = exp(Delta' A) stays below 1
    inp.delta = np.abs(inp.delta).astype(np.float32) + 0.01
    dout = wk.make_dout(wl, seed=3)
    got = gpu_bwd(inp, dout, softplus=False, use_bias=False)
    ref = oracle_bwd(oracle, inp, dout, softplus=False, use_bias=False)
    assert_grads(got, ref, wl.io)


def test_bwd_long_row(oracle):
    """4096 steps: 128 tiles and 256 checkpoints per row."""
    _check(oracle, sc.workload("blong", 1, 48, 4096))


def test_bwd_many_groups(oracle):
    _check(oracle, sc.workload("bg4", 3, 64, 104, G=4, io="f32"))


def test_bwd_repeatable(oracle):
    """The summed outputs use atomic adds: two calls agree to float32 rounding,
    and the per-element outputs are identical."""
    wl = sc.workload("brep", 2, 96, 256)
    inp = wk.make_inputs(wl, seed=1)
    dout = wk.make_dout(wl, seed=1)
    a = gpu_bwd(inp, dout)
    b = gpu_bwd(inp, dout)
    for k in ("du", "ddelta", "dz"):
        assert np.array_equal(a[k], b[k]), k
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        scale = np.max(np.abs(a[k])) + 1e-30
        assert np.max(np.abs(a[k] - b[k])) <= 1e-5 * scale, k


def test_bwd_empty_zeroes_sums():
    import torch

    import selective_state_space_120_b300 as ss
    dev = torch.device("cuda")
    u = torch.zeros(2, 8, 0, dtype=torch.bfloat16, device=dev)
    B = torch.zeros(2, 1, 16, 0, dtype=torch.bfloat16, device=dev)
    A = -torch.ones(8, 16, device=dev)
    g = ss.selective_scan_bwd(u, u.clone(), A, B, B.clone(), u.clone(),
                              D=torch.ones(8, device=dev), delta_bias=torch.zeros(8, device=dev))
    torch.cuda.synchronize()
    for k in ("dA", "dD", "ddelta_bias"):
        assert torch.count_nonzero(g[k]).item() == 0, k


def test_bwd_timeout_path_reports_and_recovers(oracle):
    """With SS_DEBUG_SKIP_FIRST_COPY the first thread block never issues its
    first tile's copies: its bounded wait runs out after the 2 ms budget, the
    call reports SS_ERR_TIMEOUT through the device status, and the next call is
    exact."""
    import selective_state_space_120_b300 as ss
    from selective_state_space_120_b300 import _binding as b
    lib = b.load()
    wl = sc.workload("bto", 2, 64, 512)
    inp = wk.make_inputs(wl)
    dout = wk.make_dout(wl)
    ss.device_status()
    b.check(lib.ss_debug_set_wait_budget_ns(2_000_000))
    b.check(lib.ss_debug_set_flags(b.SS_DEBUG_SKIP_FIRST_COPY))
    try:
        t = sc.device_inputs(inp)
        # the abandoned thread block leaves its part of the outputs unwritten
        ss.selective_scan_bwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                              sc.to_torch(dout), t["D"], t["z"], t["delta_bias"], True)
        with pytest.raises(ss.SSError) as ei:
            ss.device_status()
        assert ei.value.status == b.SS_ERR_TIMEOUT
    finally:
        b.check(lib.ss_debug_set_flags(0))
        b.check(lib.ss_debug_set_wait_budget_ns(0))
    ss.device_status()
    assert_grads(gpu_bwd(inp, dout), oracle_bwd(oracle, inp, dout), wl.io)
    ss.device_status()


@pytest.mark.slow
def test_bwd_full_size_sampled(oracle):
    """The Mamba-130M layer shape (8 x 1536 x 2048, N = 16, bf16) in the launch
    configuration the benchmark times.  Against the oracle: every per-element
    gradient of batch 0 and dB, dC of batch 0 (one full group: all 1536
    channels), and dA, dD, ddelta_bias of eight channels summed over all eight
    batches."""
    wl = wk.MAMBA_LAYER
    inp = wk.make_inputs(wl, seed=0)
    dout = wk.make_dout(wl, seed=0)
    got = gpu_bwd(inp, dout)
    f = {n: inp.as_f64(n) for n in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")}
    g64 = _dout_f64(wl, dout)
    r0 = oracle.selective_scan_bwd(f["u"][:1], f["delta"][:1, 0], f["A"], f["B"][:1, 0],
                                   f["C"][:1, 0], g64[:1], D=f["D"], z=f["z"][:1],
                                   delta_bias=f["delta_bias"])
    sub = {k: (got[k][:1] if got[k] is not None else None) for k in ("du", "ddelta", "dz", "dB", "dC")}
    assert_grads(sub, r0, wl.io, names=("du", "ddelta", "dz", "dB", "dC"))
    ch = np.array([0, 1, 31, 32, 700, 1024, 1534, 1535])
    rc = oracle.selective_scan_bwd(f["u"][:, ch], f["delta"][:, 0][:, ch], f["A"][ch], f["B"][:, 0],
                                   f["C"][:, 0], g64[:, ch], D=f["D"][ch], z=f["z"][:, ch],
                                   delta_bias=f["delta_bias"][ch])
    sums = {"dA": got["dA"][ch], "dD": got["dD"][ch], "ddelta_bias": got["ddelta_bias"][ch]}
    assert_grads(sums, rc, wl.io, names=("dA", "dD", "ddelta_bias"))


# ---------------------------------------------------------------- multi-direction backward
def _oracle_order(oracle, code):
    import selective_state_space_120_b300 as ss
    return {ss.DIR_ROW: oracle.ORDER_FWD, ss.DIR_COL: oracle.ORDER_COL,
            ss.DIR_ROW_REV: oracle.ORDER_REV, ss.DIR_COL_REV: oracle.ORDER_COL_REV,
            ss.DIR_WIN: oracle.ORDER_WIN, ss.DIR_WIN_COL: oracle.ORDER_WIN_COL,
            ss.DIR_WIN_REV: oracle.ORDER_WIN_REV, ss.DIR_WIN_COL_REV: oracle.ORDER_WIN_COL_REV}[code]


def _multi_check(oracle, H, W, orders, window, batch=2, dim=24, N=16, G=1, io="bf16",
                 with_z=True, with_D=True, use_bias=True):
    import selective_state_space_120_b300 as ss
    K, L = len(orders), H * W
    wl = sc.workload(f"mb{H}x{W}k{K}", batch, dim, L, N=N, G=G, K=K, io=io, with_z=with_z,
                     with_D=with_D, H=H, W=W)
    inp = wk.make_inputs(wl, seed=9)
    dout = wk.make_dout(wl, seed=9)
    t = sc.device_inputs(inp)
    m4 = lambda x: None if x is None else x.view(batch, dim, H, W)  # noqa: E731
    g = ss.multi_scan_bwd(m4(t["u"]), t["delta"], t["A"], t["B"], t["C"], m4(sc.to_torch(dout)),
                          orders, window, t["D"], t["delta_bias"] if use_bias else None, True,
                          z=m4(t["z"]))
    ref = oracle.multi_scan_bwd(inp.as_f64("u"), inp.as_f64("delta"), inp.as_f64("A"),
                                inp.as_f64("B"), inp.as_f64("C"), _dout_f64(wl, dout),
                                [_oracle_order(oracle, o) for o in orders], H=H, W=W, win=window,
                                D=inp.as_f64("D"), z=inp.as_f64("z"),
                                delta_bias=inp.as_f64("delta_bias") if use_bias else None)
    got = {k: (None if v is None else sc.from_torch(v)) for k, v in g.items()}
    for k in ("du", "dz"):
        if got[k] is not None:
            got[k] = got[k].reshape(batch, dim, L)
    return assert_grads(got, ref, io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_multi_bwd_bidirectional(oracle, io):
    import selective_state_space_120_b300 as ss
    _multi_check(oracle, 1, 200, [ss.DIR_ROW, ss.DIR_ROW_REV], 0, io=io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_multi_bwd_ss2d(oracle, io):
    import selective_state_space_120_b300 as ss
    _multi_check(oracle, 8, 12, [ss.DIR_ROW, ss.DIR_COL, ss.DIR_ROW_REV, ss.DIR_COL_REV], 0, io=io)


def test_multi_bwd_windowed_cut_short(oracle):
    import selective_state_space_120_b300 as ss
    _multi_check(oracle, 7, 8, [ss.DIR_WIN, ss.DIR_WIN_COL, ss.DIR_WIN_REV, ss.DIR_WIN_COL_REV], 3)


def test_multi_bwd_video_orders(oracle):
    import selective_state_space_120_b300 as ss
    _multi_check(oracle, 4, 36, [ss.DIR_ROW, ss.DIR_ROW_REV, ss.DIR_COL, ss.DIR_COL_REV], 0)


def test_multi_bwd_all_orders_groups(oracle):
    _multi_check(oracle, 8, 8, list(range(8)), 3, dim=32, N=4, G=2, io="f32")


def test_multi_bwd_without_gate_skip_bias(oracle):
    import selective_state_space_120_b300 as ss
    _multi_check(oracle, 6, 16, [ss.DIR_COL_REV, ss.DIR_WIN], 4, with_z=False)
    _multi_check(oracle, 6, 16, [ss.DIR_ROW_REV, ss.DIR_COL], 0, with_D=False, use_bias=False)


def test_multi_bwd_larger_map(oracle):
    """Several tiles and checkpoint blocks per direction on a 32 x 40 map."""
    import selective_state_space_120_b300 as ss
    _multi_check(oracle, 32, 40, [ss.DIR_ROW, ss.DIR_COL, ss.DIR_ROW_REV, ss.DIR_COL_REV], 0,
                 batch=1, dim=40)


# ---------------------------------------------------------------- options: ZOH, h0, Conv1D
def _h0(wl, seed=11):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((wl.batch, wl.dim, wl.N)) * 0.5).astype(np.float32)


def _conv(wl, seed=31, bias=True, history=True):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((wl.dim, 4)) * 0.5).astype(np.float32)
    b = (rng.standard_normal(wl.dim) * 0.1).astype(np.float32) if bias else None
    x0 = rng.standard_normal((wl.batch, wl.dim, 3)).astype(np.float32) if history else None
    return w, b, x0


def _opts_case(oracle, wl, zoh=False, with_h0=False, conv=None, seed=0):
    """The backward pass with the forward call's options against the oracle:
    its scan gradients (zero-order hold, initial state) and, with the Conv1D,
    its convolution followed by the scan, differentiated through both."""
    import torch
    import selective_state_space_120_b300 as ss
    inp = wk.make_inputs(wl, seed=seed)
    dout = wk.make_dout(wl, seed=seed)
    h0 = _h0(wl) if with_h0 else None
    t = sc.device_inputs(inp)
    kw = {}
    if conv is not None:
        w, b, x0 = conv
        kw = dict(conv_w=sc.to_torch(w), conv_b=sc.to_torch(b), conv_x0=sc.to_torch(x0))
    g = ss.selective_scan_bwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                              sc.to_torch(dout), t["D"], t["z"], t["delta_bias"], True,
                              h0=None if h0 is None else sc.to_torch(h0), zoh=zoh, **kw)
    torch.cuda.synchronize()
    got = {k: (None if v is None else sc.from_torch(v)) for k, v in g.items()}
    u = inp.as_f64("u")
    if conv is not None:
        w, b, x0 = conv
        f64 = lambda a: None if a is None else a.astype(np.float64)  # noqa: E731
        u = oracle.conv_silu(u, f64(w), f64(b), f64(x0))
    ref = oracle.selective_scan_bwd(u, inp.as_f64("delta")[:, 0], inp.as_f64("A"),
                                    inp.as_f64("B")[:, 0], inp.as_f64("C")[:, 0],
                                    _dout_f64(wl, dout), D=inp.as_f64("D"), z=inp.as_f64("z"),
                                    delta_bias=inp.as_f64("delta_bias"), delta_softplus=True,
                                    zoh=zoh, h0=None if h0 is None else h0.astype(np.float64))
    names = list(NAMES)
    if with_h0:
        names.append("dh0")
    if conv is not None:
        w, b, x0 = conv
        cg = oracle.conv_silu_bwd(inp.as_f64("u"), w.astype(np.float64), ref["du"],
                                  None if b is None else b.astype(np.float64),
                                  None if x0 is None else x0.astype(np.float64))
        ref = dict(ref)
        ref["du"] = cg["dx"]
        ref["dconv_w"], ref["dconv_b"], ref["dconv_x0"] = cg["dw"], cg["dbias"], cg["dx0"]
        names += ["dconv_w", "dconv_b", "dconv_x0"]
    return assert_grads(got, ref, wl.io, names)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [48, 200])
def test_bwd_zero_order_hold(oracle, io, L):
    """The zero-order-hold input matrix: every gradient, including dA's term
    from the derivative of (exp(Delta'A) - 1)/A, on a ragged tail."""
    _opts_case(oracle, sc.workload(f"bzoh{L}", 2, 40, L, io=io), zoh=True)


def test_bwd_zero_order_hold_large_steps(oracle):
    """|Delta' A| well above the series threshold for every state."""
    wl = sc.workload("bzohl", 1, 24, 96, io="f32")
    inp = wk.make_inputs(wl, seed=0)
    inp.delta_bias[:] = 1.5
    dout = wk.make_dout(wl, seed=0)
    import torch
    import selective_state_space_120_b300 as ss
    t = sc.device_inputs(inp)
    g = ss.selective_scan_bwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                              sc.to_torch(dout), t["D"], t["z"], t["delta_bias"], True, zoh=True)
    torch.cuda.synchronize()
    got = {k: (None if v is None else sc.from_torch(v)) for k, v in g.items()}
    ref = oracle.selective_scan_bwd(inp.as_f64("u"), inp.as_f64("delta")[:, 0], inp.as_f64("A"),
                                    inp.as_f64("B")[:, 0], inp.as_f64("C")[:, 0],
                                    _dout_f64(wl, dout), D=inp.as_f64("D"), z=inp.as_f64("z"),
                                    delta_bias=inp.as_f64("delta_bias"), zoh=True)
    assert_grads(got, ref, "f32")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("L", [8, 200, 520])
def test_bwd_initial_state(oracle, io, L):
    """A given initial state and its gradient dh0 = Abar_0 (.) dh_0: one
    checkpoint block, a ragged tail, and several tiles."""
    _opts_case(oracle, sc.workload(f"bh0{L}", 2, 40, L, io=io), with_h0=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_zero_order_hold_and_initial_state(oracle, io):
    _opts_case(oracle, sc.workload("bzh", 2, 36, 136, G=2, io=io), zoh=True, with_h0=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("bias,history", [(True, True), (False, False), (True, False)])
def test_bwd_fused_conv_silu(oracle, io, bias, history):
    """The Conv1D + SiLU fused in front: gradients of its input x, weights,
    bias and history, and every scan gradient, against the oracle's
    convolution followed by its scan, differentiated through both; the
    sequence spans two convolution tiles and a ragged tail."""
    wl = sc.workload("bconv", 2, 40, 264, io=io)
    _opts_case(oracle, wl, conv=_conv(wl, bias=bias, history=history))


def test_bwd_fused_conv_with_every_option(oracle):
    wl = sc.workload("bconvall", 2, 24, 520, io="f32")
    _opts_case(oracle, wl, zoh=True, with_h0=True, conv=_conv(wl))
