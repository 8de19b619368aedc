"""GPU parity: the CUDA library against the float64 oracle, element by element,
on the same seeded inputs (B300 only).

Small cases span several channel blocks and time tiles and end on ragged
tails; full-size workloads are checked on sampled channels, which the oracle
computes independently (each channel's scan depends only on its own row).
"""
import numpy as np
import pytest

from selective_state_space_120_b300 import workloads as wk
from tests import scan_cases as sc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_120_b300 as ss
    ss.load_library()


def _check(oracle, wl, chunks=0):
    inp = wk.make_inputs(wl, seed=0)
    out, last = sc.gpu_run(inp, chunks=chunks)
    ref, ref_last = sc.oracle_run(oracle, inp)
    e = sc.assert_close(sc.from_torch(out), ref, wl.io)
    got_last = last.cpu().numpy().astype(np.float64)
    if wl.K == 1:
        ref_last = ref_last[:, 0]
    sc.assert_close(got_last, ref_last, wl.io, "last_state")
    return e


# ---------------------------------------------------------------- single direction
def test_tiny_f32_config(oracle):
    """1 x 16 x 64, N = 16, float32 I/O (the tiny S6 workload), whole output."""
    _check(oracle, wk.TINY_F32)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 32, 64])
def test_scan_all_dstates(oracle, io, N):
    _check(oracle, sc.workload(f"n{N}", 2, 40, 208, N=N, io=io))


@pytest.mark.parametrize("L", [8, 16, 200, 264, 1000])
def test_scan_ragged_lengths_tma_path(oracle, L):
    _check(oracle, sc.workload(f"l{L}", 2, 36, L, G=2))


@pytest.mark.parametrize("L", [1, 7, 31, 33, 197, 257])
def test_scan_unaligned_lengths(oracle, L):
    """Rows that are not 16-byte multiples, 20 channels (which P = 8 rows to a
    view row does not divide): the on-chip gather path."""
    _check(oracle, sc.workload(f"u{L}", 2, 20, L))


@pytest.mark.parametrize("L", [1, 7, 33, 197, 1001])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_view_rows(oracle, L, io):
    """Rows that are not 16-byte multiples, read in place through view tiles
    (P = 8 rows to a view row in bf16, 4 in fp32), several channel blocks and a
    partial last one, the gate and last_state."""
    _check(oracle, sc.workload(f"sv{L}", 2, 72, L, io=io))


@pytest.mark.parametrize("L,N,G,io", [(198, 2, 1, "bf16"), (196, 4, 2, "bf16"), (197, 8, 2, "f32"),
                                      (197, 32, 1, "bf16"), (99, 64, 1, "f32")])
def test_scan_view_rows_dstates_groups(oracle, L, N, G, io):
    """View tiles with two, four and eight rows to a view row, every state
    count's configuration, groups, no gate."""
    _check(oracle, sc.workload(f"svn{N}_{L}", 2, 48, L, N=N, G=G, io=io, with_z=False))


@pytest.mark.parametrize("chunks", [0, 3])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_view_rows_chunked(oracle, chunks, io):
    """Few rows of an unaligned length: the chunked path over view tiles
    (automatic chunking, and three chunks)."""
    _check(oracle, sc.workload("svc", 1, 16, 3001, io=io), chunks=chunks)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_view_rows_isolate_channels(oracle, io):
    """A view tile holds the neighbouring rows' values past each row's ends: a
    NaN in one channel's u and z and an infinite Delta in another's must not
    reach any other channel."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("sv_iso", 2, 16, 197, io=io)
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    t["u"][0, 5] = float("nan")
    t["z"][0, 5] = float("nan")
    t["delta"][0, 0, 10] = float("inf")
    out, last = ss.selective_scan_fwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                                      t["D"], t["z"], t["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp)
    keep = [d for d in range(wl.dim) if d not in (5, 10)]
    got = sc.from_torch(out)
    sc.assert_close(got[0, keep], ref[0, keep], io)
    sc.assert_close(got[1], ref[1], io)
    got_last = last.cpu().numpy().astype(np.float64)
    sc.assert_close(got_last[0, keep], ref_last[0, 0, keep], io, "last_state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_scan_without_gate_or_skip(oracle, io):
    _check(oracle, sc.workload("nozd", 1, 33, 96, io=io, with_z=False, with_D=False))


@pytest.mark.parametrize("chunks", [2, 3, 5])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_chunked_long_sequence_path(oracle, chunks, io):
    """The chunk-local pass, carry and fix-up reproduce the sequential scan."""
    _check(oracle, sc.workload("chunked", 1, 24, 1200, io=io), chunks=chunks)


def test_chunked_equals_direct_to_fp32_rounding():
    wl = sc.workload("cmp", 2, 64, 2048, io="f32")
    inp = wk.make_inputs(wl)
    o1, l1 = sc.gpu_run(inp, chunks=1)
    o4, l4 = sc.gpu_run(inp, chunks=4)
    assert sc.rel_err(sc.from_torch(o4), sc.from_torch(o1)) < 2e-5
    assert sc.rel_err(l4.cpu().numpy(), l1.cpu().numpy()) < 2e-5


def test_chunked_long_edge_chunks_equal_direct():
    """Few rows (160 CTAs of 32 channels, a quarter of the GPU's slots): the
    automatic split makes the first and last L-chunks several times longer
    than the middle ones; every row still equals the single pass to fp32
    rounding."""
    wl = sc.workload("edges", 1, 5120, 4096, io="f32")
    inp = wk.make_inputs(wl)
    o1, l1 = sc.gpu_run(inp, chunks=1)
    oa, la = sc.gpu_run(inp, chunks=0)
    assert sc.rel_err(sc.from_torch(oa), sc.from_torch(o1)) < 2e-5
    assert sc.rel_err(la.cpu().numpy(), l1.cpu().numpy()) < 2e-5


@pytest.mark.parametrize("io,L", [("f32", 8192), ("bf16", 16384)])
def test_chunked_long_edge_chunks_against_oracle(oracle, io, L):
    """The long-sequence shape's rows with fewer steps, automatic split (long
    first and last L-chunks, middle ones between): sampled channels over the
    whole sequence and their last states against the oracle."""
    _sampled(oracle, sc.workload("edges_" + io, 1, 5120, L, io=io), nrows=6)


def test_deterministic_and_guarded():
    """Two runs give identical bits; nothing is written outside `out`."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("det", 2, 40, 136)
    inp = wk.make_inputs(wl)
    t = sc.device_inputs(inp)
    n = t["u"].numel()
    pad = 4096
    guard = torch.full((n + 2 * pad,), float("nan"), dtype=torch.bfloat16, device="cuda")
    out = guard[pad:pad + n].view_as(t["u"])
    outs = []
    for _ in range(2):
        ss.selective_scan_fwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0], t["D"],
                              t["z"], t["delta_bias"], True, out=out)
        outs.append(out.clone())
    torch.cuda.synchronize()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    assert torch.isnan(guard[:pad]).all() and torch.isnan(guard[pad + n:]).all()


def test_multidir_deterministic():
    import torch
    for wl in (sc.workload("bi_det", 2, 24, 197, K=2),
               sc.workload("ss_det", 2, 12, 64, K=4, with_z=False, H=8, W=8)):
        inp = wk.make_inputs(wl)
        t = sc.device_inputs(inp)
        a, _ = sc.gpu_run(inp, t=t)
        b, _ = sc.gpu_run(inp, t=t)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), wl.name


def test_empty_inputs_are_noops():
    import torch
    import selective_state_space_120_b300 as ss
    u = torch.empty(0, 8, 32, dtype=torch.bfloat16, device="cuda")
    B = torch.empty(0, 1, 16, 32, dtype=torch.bfloat16, device="cuda")
    A = -torch.ones(8, 16, device="cuda")
    out = ss.selective_scan_fwd(u, u, A, B, B)
    assert out.shape == u.shape


def test_timeout_path_reports_and_recovers(oracle):
    """A wait that nothing will satisfy: with SS_DEBUG_SKIP_FIRST_COPY the first
    thread block never issues its first tile's copies, so its bounded wait runs
    out after the (2 ms) budget.  The call reports SS_ERR_TIMEOUT through the
    device status, the context stays usable, and the next call is exact."""
    import selective_state_space_120_b300 as ss
    from selective_state_space_120_b300 import _binding as b
    lib = b.load()
    wl = sc.workload("to", 2, 64, 2048)
    inp = wk.make_inputs(wl)
    ss.device_status()
    b.check(lib.ss_debug_set_wait_budget_ns(2_000_000))
    b.check(lib.ss_debug_set_flags(b.SS_DEBUG_SKIP_FIRST_COPY))
    try:
        sc.gpu_run(inp, chunks=1)
        with pytest.raises(ss.SSError) as ei:
            ss.device_status()
        assert ei.value.status == b.SS_ERR_TIMEOUT
    finally:
        b.check(lib.ss_debug_set_flags(0))
        b.check(lib.ss_debug_set_wait_budget_ns(0))
    ss.device_status()  # cleared
    out, last = sc.gpu_run(inp, chunks=1)
    ref, ref_last = sc.oracle_run(oracle, inp)
    sc.assert_close(sc.from_torch(out), ref, "bf16")
    sc.assert_close(last.cpu().numpy(), ref_last[:, 0], "bf16", "last_state")
    ss.device_status()


# ---------------------------------------------------------------- options: h0, ZOH
def _h0(wl, seed=11):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((wl.batch, wl.dim, wl.N)) * 0.5).astype(np.float32)


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_initial_state(oracle, chunks, io):
    """A given initial state, on the direct and the chunked path (TMA rows)."""
    wl = sc.workload("h0", 2, 40, 1024, io=io)
    inp = wk.make_inputs(wl)
    h0 = _h0(wl)
    out, last = sc.gpu_run(inp, chunks=chunks, h0=h0)
    ref, ref_last = sc.oracle_run(oracle, inp, h0=h0)
    sc.assert_close(sc.from_torch(out), ref, io)
    sc.assert_close(last.cpu().numpy(), ref_last[:, 0], io, "last_state")


def test_initial_state_unaligned_rows(oracle):
    wl = sc.workload("h0u", 2, 24, 77)
    inp = wk.make_inputs(wl)
    h0 = _h0(wl)
    out, last = sc.gpu_run(inp, h0=h0)
    ref, ref_last = sc.oracle_run(oracle, inp, h0=h0)
    sc.assert_close(sc.from_torch(out), ref, "bf16")
    sc.assert_close(last.cpu().numpy(), ref_last[:, 0], "bf16", "last_state")


def test_continuing_a_sequence_across_calls():
    """Scanning L1 steps, then L2 steps from the first call's last_state, gives
    the output and final state of one scan over L1 + L2 steps (fp32 I/O)."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("split", 2, 32, 1024, io="f32")
    inp = wk.make_inputs(wl)
    t = sc.device_inputs(inp)
    full, last_full = sc.gpu_run(inp, t=t)
    cut = 512
    parts = {k: (None if v is None else v) for k, v in t.items()}
    def piece(a, lo, hi):
        return None if a is None else a[..., lo:hi].contiguous()
    o1, l1 = ss.selective_scan_fwd(piece(parts["u"], 0, cut), piece(parts["delta"][:, 0], 0, cut),
                                   parts["A"], piece(parts["B"][:, 0], 0, cut),
                                   piece(parts["C"][:, 0], 0, cut), parts["D"],
                                   piece(parts["z"], 0, cut), parts["delta_bias"], True,
                                   return_last_state=True)
    o2, l2 = ss.selective_scan_fwd(piece(parts["u"], cut, None), piece(parts["delta"][:, 0], cut, None),
                                   parts["A"], piece(parts["B"][:, 0], cut, None),
                                   piece(parts["C"][:, 0], cut, None), parts["D"],
                                   piece(parts["z"], cut, None), parts["delta_bias"], True,
                                   return_last_state=True, h0=l1)
    torch.cuda.synchronize()
    got = torch.cat([o1, o2], dim=-1)
    assert sc.rel_err(got.cpu().numpy(), full.cpu().numpy()) < 2e-5
    assert sc.rel_err(l2.cpu().numpy(), last_full.cpu().numpy()) < 2e-5


@pytest.mark.parametrize("chunks", [1, 4])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zero_order_hold(oracle, chunks, io):
    """SS_SCAN_ZOH: Bbar = (exp(Delta A) - 1)/A * B, against the oracle's ZOH."""
    wl = sc.workload("zoh", 2, 36, 1024, io=io)
    inp = wk.make_inputs(wl)
    out, last = sc.gpu_run(inp, chunks=chunks, zoh=True)
    ref, ref_last = sc.oracle_run(oracle, inp, zoh=True)
    sc.assert_close(sc.from_torch(out), ref, io)
    sc.assert_close(last.cpu().numpy(), ref_last[:, 0], io, "last_state")


def test_zero_order_hold_large_steps_and_unaligned_rows(oracle):
    """Large Delta (|Delta A| well above the series threshold) and rows the TMA
    path does not take."""
    wl = sc.workload("zohu", 1, 24, 61, io="f32")
    inp = wk.make_inputs(wl)
    inp.delta_bias[:] = 1.5  # Delta' ~ 1.7: exp(Delta A) far from 1 for every state
    out, last = sc.gpu_run(inp, zoh=True)
    ref, ref_last = sc.oracle_run(oracle, inp, zoh=True)
    sc.assert_close(sc.from_torch(out), ref, "f32")
    sc.assert_close(last.cpu().numpy(), ref_last[:, 0], "f32", "last_state")


# ---------------------------------------------------------------- fused Conv1D + SiLU
def _conv_params(dim, seed=31):
    rng = np.random.default_rng(seed)
    return ((rng.standard_normal((dim, 4)) * 0.5).astype(np.float32),
            (rng.standard_normal(dim) * 0.1).astype(np.float32))


def _conv_case(oracle, wl, chunks, with_history):
    import torch
    import selective_state_space_120_b300 as ss
    inp = wk.make_inputs(wl)
    w, cb = _conv_params(wl.dim)
    rng = np.random.default_rng(32)
    x0 = rng.standard_normal((wl.batch, wl.dim, 3)).astype(np.float32) if with_history else None
    h0 = _h0(wl) if with_history else None
    t = sc.device_inputs(inp)
    out, last = ss.selective_scan_fwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0], t["C"][:, 0],
                                      t["D"], t["z"], t["delta_bias"], True, return_last_state=True,
                                      chunks=chunks, h0=None if h0 is None else sc.to_torch(h0),
                                      conv_w=sc.to_torch(w), conv_b=sc.to_torch(cb),
                                      conv_x0=None if x0 is None else sc.to_torch(x0))
    torch.cuda.synchronize()
    u = oracle.conv_silu(inp.as_f64("u"), w.astype(np.float64), cb.astype(np.float64),
                         None if x0 is None else x0.astype(np.float64))
    ref, ref_last = oracle.scan(u, inp.as_f64("delta"), inp.as_f64("A"), inp.as_f64("B"),
                                inp.as_f64("C"), inp.as_f64("D"), inp.as_f64("z"),
                                inp.as_f64("delta_bias"), True,
                                h0=None if h0 is None else h0.astype(np.float64)[:, None])
    sc.assert_close(sc.from_torch(out), ref, wl.io)
    sc.assert_close(last.cpu().numpy(), ref_last[:, 0], wl.io, "last_state")


@pytest.mark.parametrize("chunks", [1, 3])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_fused_conv_silu(oracle, chunks, io):
    """The Conv1D(k=4) + SiLU input branch fused in front of the scan, on the
    direct and the chunked path, against the oracle's conv followed by its scan."""
    _conv_case(oracle, sc.workload("conv", 2, 40, 1024, io=io), chunks, False)


@pytest.mark.parametrize("chunks", [1, 4])
def test_fused_conv_silu_continuing(oracle, chunks):
    """Conv history and initial state given: the call continues a sequence."""
    _conv_case(oracle, sc.workload("convh", 2, 24, 520), chunks, True)


# ---------------------------------------------------------------- single-step decode
@pytest.mark.parametrize("N", [1, 4, 16, 64])
@pytest.mark.parametrize("io,zoh", [("f32", False), ("bf16", False), ("f32", True)])
def test_state_update_one_step(oracle, N, io, zoh):
    """One decode step from a random state equals the oracle over one step with
    h0 = state; the state is updated in place."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("step", 3, 40, 1, N=N, G=2, io=io)
    inp = wk.make_inputs(wl)
    h0 = _h0(wl)
    t = sc.device_inputs(inp)
    state = sc.to_torch(h0).clone()
    out = ss.selective_state_update(t["u"][:, :, 0].contiguous(), t["delta"][:, 0, :, 0].contiguous(),
                                    t["A"], t["B"][:, 0, :, :, 0].contiguous(),
                                    t["C"][:, 0, :, :, 0].contiguous(), state, t["D"],
                                    t["z"][:, :, 0].contiguous(), t["delta_bias"], True, zoh=zoh)
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp, h0=h0, zoh=zoh)
    sc.assert_close(sc.from_torch(out), ref[:, :, 0], io)
    sc.assert_close(state.cpu().numpy(), ref_last[:, 0], io, "state")


def test_state_update_chain_equals_scan():
    """T decode steps from a zero state reproduce the scan over T steps (fp32)."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("chain", 2, 24, 40, io="f32")
    inp = wk.make_inputs(wl)
    t = sc.device_inputs(inp)
    full, last = sc.gpu_run(inp, t=t)
    state = torch.zeros(wl.batch, wl.dim, wl.N, device="cuda")
    outs = []
    for k in range(wl.L):
        outs.append(ss.selective_state_update(
            t["u"][:, :, k].contiguous(), t["delta"][:, 0, :, k].contiguous(), t["A"],
            t["B"][:, 0, :, :, k].contiguous(), t["C"][:, 0, :, :, k].contiguous(), state, t["D"],
            t["z"][:, :, k].contiguous(), t["delta_bias"], True))
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=-1)
    assert sc.rel_err(got.cpu().numpy(), full.cpu().numpy()) < 2e-5
    assert sc.rel_err(state.cpu().numpy(), last.cpu().numpy()) < 2e-5


# ---------------------------------------------------------------- bidirectional
@pytest.mark.parametrize("L", [1, 7, 33, 197, 256])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bidirectional(oracle, L, io):
    _check(oracle, sc.workload(f"bi{L}", 2, 24, L, K=2, io=io))


def test_bidirectional_groups_dstate(oracle):
    _check(oracle, sc.workload("bi_g", 2, 32, 50, N=8, G=2, K=2))


@pytest.mark.parametrize("L", [7, 197])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bidirectional_unaligned_rows_without_workspace(oracle, L, io):
    """Rows that are not 16-byte aligned with no workspace given: the call
    merges on chip instead of re-pitching its inputs (same results)."""
    import ctypes
    import torch
    from selective_state_space_120_b300 import _binding as b
    lib = b.load()
    wl = sc.workload(f"bi_nows{L}", 2, 24, L, K=2, io=io)
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    out = torch.empty_like(t["u"])
    last = torch.empty(wl.batch, 2, wl.dim, wl.N, dtype=torch.float32, device="cuda")
    p = lambda x: None if x is None else x.data_ptr()  # noqa: E731
    b.check(lib.ss_bidir_scan_fwd(wl.batch, wl.dim, L, wl.N, wl.G, b.SS_BF16 if io == "bf16" else b.SS_F32,
                                  p(t["u"]), p(t["delta"]), p(t["A"]), p(t["B"]), p(t["C"]), p(t["D"]),
                                  p(t["z"]), p(t["delta_bias"]), 1, p(out), p(last), None, 0,
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp)
    sc.assert_close(sc.from_torch(out), ref, io)
    sc.assert_close(last.cpu().numpy().astype(np.float64), ref_last, io, "last_state")


@pytest.mark.parametrize("L", [1, 5, 9, 197, 1001])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bidirectional_view_rows(oracle, L, io):
    """Rows that are not 16-byte aligned, with the workspace: both directions
    run as TMA scans that read the rows in place through a view of P rows to a
    view row (P = 8 in bf16, 4 in fp32; several channel blocks and a partial
    last one, N = 8)."""
    _check(oracle, sc.workload(f"bi_v{L}", 3, 72, L, N=8, K=2, io=io))


@pytest.mark.parametrize("L,io", [(198, "bf16"), (196, "bf16"), (198, "f32"), (102, "f32")])
@pytest.mark.parametrize("N", [4, 16])
def test_bidirectional_view_rows_fold(oracle, L, io, N):
    """Two or four rows to a view row (L = 198 and 196 in bf16, 198 and 102 in
    fp32), with N = 4 (one B row to a box) and N = 16."""
    _check(oracle, sc.workload(f"bi_vf{L}", 2, 40, L, N=N, K=2, io=io))


@pytest.mark.parametrize("L,N", [(197, 32), (197, 64), (196, 2), (197, 8)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bidirectional_view_rows_dstates(oracle, L, N, io):
    """View tiles of the other state counts' configurations: N = 32 and 64
    (8 warps of 32 channels a CTA), N = 2 with two rows to a view row in bf16,
    N = 8 with eight (bf16) or four (fp32) rows to a view row."""
    _check(oracle, sc.workload(f"bi_vn{N}_{L}", 2, 40, L, N=N, K=2, io=io))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bidirectional_view_rows_isolate_channels(oracle, io):
    """A view tile holds the neighbouring rows' values past each row's ends: a
    NaN in one channel's u and an infinite Delta in another's must not reach
    any other channel (the rest match the oracle on the clean inputs)."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload("bi_viso", 2, 16, 197, N=8, K=2, io=io)
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    t["u"][0, 5] = float("nan")
    t["delta"][0, :, 10] = float("inf")
    out, last = ss.bidir_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                  t["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp)
    keep = [d for d in range(wl.dim) if d not in (5, 10)]
    got = sc.from_torch(out)
    sc.assert_close(got[0, keep], ref[0, keep], io)
    sc.assert_close(got[1], ref[1], io)
    got_last = last.cpu().numpy().astype(np.float64)
    sc.assert_close(got_last[0][:, keep], ref_last[0][:, keep], io, "last_state")


@pytest.mark.parametrize("L", [5, 197])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bidirectional_repitched_rows(oracle, L, io):
    """Channels per group that P does not divide (18): the inputs are copied
    into rows of a 16-byte pitch, and both directions run as TMA scans."""
    _check(oracle, sc.workload(f"bi_rp{L}", 3, 18, L, N=8, K=2, io=io))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("dim", [48, 36])
def test_bidirectional_repitched_rows_groups(oracle, io, dim):
    """Two groups, given the workspace the size query reports (sized for one
    group) and given more.  24 channels a group: read in place through the view
    either way (its two slices do not grow with the groups).  18 channels a
    group: the re-pitched B and C grow with the groups, so the reported size is
    too small and the call merges on chip; with room it re-pitches.  All agree
    with the oracle."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = sc.workload(f"bi_rpg{dim}", 2, dim, 197, N=8, G=2, K=2, io=io)
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    ref, ref_last = sc.oracle_run(oracle, inp)
    for extra in (0, 1 << 20):
        need = ss.workspace_bytes(1, wl.batch, wl.dim, wl.L, wl.N) + extra
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        out, last = ss.bidir_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                                      t["delta_bias"], True, return_last_state=True, workspace=ws)
        torch.cuda.synchronize()
        sc.assert_close(sc.from_torch(out), ref, io)
        sc.assert_close(last.cpu().numpy().astype(np.float64), ref_last, io, "last_state")


# ---------------------------------------------------------------- SS2D
@pytest.mark.parametrize("H,W", [(1, 1), (3, 5), (5, 3), (8, 8), (7, 16), (56, 56)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_cross_scan2d(oracle, H, W, io):
    _check(oracle, sc.workload(f"ss2d{H}x{W}", 2, 12, H * W, K=4, io=io, with_z=False, H=H, W=W))


def test_cross_scan2d_gated_groups(oracle):
    """Unaligned rows (60 bf16 = 120 bytes) with 8 channels a group and N = 4,
    which the view's P = 2 divides: view tiles, with a gate and two groups."""
    _check(oracle, sc.workload("ss2d_gz", 1, 16, 6 * 10, N=4, G=2, K=4, H=6, W=10))


@pytest.mark.parametrize("H,W", [(1, 1), (3, 5), (5, 3), (7, 7), (14, 14), (6, 10)])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_cross_scan2d_view_maps(oracle, H, W, io):
    """Maps whose rows are not 16-byte aligned (VMamba's 14 x 14 and 7 x 7
    stages among them), 24 channels: the four directions over view tiles (the
    column pair over the transposed copy), merged by step."""
    _check(oracle, sc.workload(f"ss2dv{H}x{W}", 2, 24, H * W, K=4, io=io, with_z=False, H=H, W=W))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_cross_scan2d_unaligned_on_chip(oracle, io):
    """Unaligned rows with 12 channels, which P = 8 (bf16) or 4 (fp32) rows to a
    view row does not divide: the on-chip merge path."""
    _check(oracle, sc.workload("ss2d_oc", 2, 12, 7 * 7, K=4, io=io, H=7, W=7))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_cross_scan2d_view_isolate_channels(oracle, io):
    """A view tile holds the neighbouring rows' values past each row's ends: a
    NaN in one channel's map must not reach any other channel."""
    import torch
    import selective_state_space_120_b300 as ss
    H, W = 7, 7
    wl = sc.workload("ss2dv_iso", 2, 16, H * W, K=4, io=io, with_z=False, H=H, W=W)
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    t["u"][0, 5] = float("nan")
    bsz, dim, L = t["u"].shape
    out, last = ss.cross_scan2d_fwd(t["u"].view(bsz, dim, H, W), t["delta"], t["A"], t["B"], t["C"],
                                    t["D"], t["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    ref, ref_last = sc.oracle_run(oracle, inp)
    keep = [d for d in range(wl.dim) if d != 5]
    got = sc.from_torch(out.view(bsz, dim, L))
    sc.assert_close(got[0, keep], ref[0, keep], io)
    sc.assert_close(got[1], ref[1], io)


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_cross_scan2d_gated_groups_workspace_path(oracle, io):
    """Aligned rows: four TMA-staged direction scans merged through the fp32
    workspace, with a z gate, two groups, N = 8 and a channel count that leaves
    a partial channel block."""
    _check(oracle, sc.workload("ss2d_gzw", 2, 40, 4 * 8, N=8, G=2, K=4, io=io, H=4, W=8))


@pytest.mark.parametrize("L", [64, 200])
def test_bidirectional_workspace_path_groups(oracle, L):
    _check(oracle, sc.workload(f"bi_w{L}", 2, 48, L, N=16, G=2, K=2))


# ---------------------------------------------------------------- full-size workloads
def _sampled(oracle, wl, nrows=12, seed=1):
    import torch
    inp = wk.make_inputs(wl, seed=0)
    out, last = sc.gpu_run(inp)
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    rows = [(int(rng.integers(wl.batch)), int(rng.integers(wl.dim))) for _ in range(nrows)]
    rows += [(0, 0), (wl.batch - 1, wl.dim - 1)]
    ref, ref_last = sc.oracle_run(oracle, inp, rows)
    got = np.stack([sc.from_torch(out[b, d]) for b, d in rows])
    sc.assert_close(got, ref, wl.io)
    if wl.K == 1:
        got_l = np.stack([last[b, d].cpu().numpy() for b, d in rows])
        sc.assert_close(got_l, ref_last[:, 0], wl.io, "last_state")
    else:
        got_l = np.stack([last[b, :, d].cpu().numpy() for b, d in rows])
        sc.assert_close(got_l, ref_last, wl.io, "last_state")
    assert torch.isfinite(out.float()).all()


@pytest.mark.slow
@pytest.mark.parametrize("wl", [wk.MAMBA_LAYER, wk.LONG_SEQ, wk.VIM_BIDIR, wk.VMAMBA_SS2D,
                                wk.MAMBA_LAYER_UNALIGNED, wk.VMAMBA_SS2D_14], ids=lambda w: w.name)
def test_full_size_sampled(oracle, wl):
    _sampled(oracle, wl)
