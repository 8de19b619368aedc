"""ss_selective_scan_fwd_noalloc: the scan for callers that cannot allocate.

Some callers may not allocate device memory while they run: a plug-in driven
by another engine that owns every device buffer, or a latency-critical loop in
which cudaMalloc/cudaFree could synchronise the device.  They cannot hand the
long-sequence chunked path a workspace, so this entry point runs that path on
a fixed scratch array that the library keeps in static device memory.

These tests call it through the C ABI and compare it with the existing entry
point (ss_selective_scan_fwd_opts with a caller-provided workspace) on the same
inputs, bit for bit (same kernels, same L-chunks), for two calls in a row: the
shared scratch keeps the first call's contents, and the second call must not
be affected by them.  The file is named so that pytest collects it last.
"""
import ctypes

import pytest

from selective_state_space_120_b300 import workloads as wk
from tests import scan_cases as sc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_120_b300 as ss
    from selective_state_space_120_b300 import _binding as b
    ss.load_library()
    return b.load()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call_args(t, wl, out, last):
    io = 1 if wl.io == "bf16" else 0
    return (wl.batch, wl.dim, wl.L, wl.N, wl.G, io, _ptr(t["u"]), _ptr(t["delta"]),
            _ptr(t["A"]), _ptr(t["B"]), _ptr(t["C"]), _ptr(t["D"]), _ptr(t["z"]),
            _ptr(t["delta_bias"]), 1, _ptr(out), _ptr(last))


def _device(inp):
    t = sc.device_inputs(inp)
    t["delta"] = t["delta"][:, 0].contiguous()
    t["B"] = t["B"][:, 0].contiguous()
    t["C"] = t["C"][:, 0].contiguous()
    return t


def _run_both(lib, wl, seed, chunks):
    """(noalloc out, last), (workspace out, last) on the same inputs."""
    import torch
    from selective_state_space_120_b300 import _binding as b
    inp = wk.make_inputs(wl, seed=seed)
    t = _device(inp)
    opts = b.options(chunks)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    out_na = torch.empty_like(t["u"])
    last_na = torch.empty(wl.batch, wl.dim, wl.N, dtype=torch.float32, device="cuda")
    b.check(lib.ss_selective_scan_fwd_noalloc(*_call_args(t, wl, out_na, last_na),
                                              ctypes.byref(opts), stream))

    need = int(lib.ss_workspace_bytes_opts(b.SS_KIND_SCAN, wl.batch, wl.dim, wl.L, wl.N,
                                           ctypes.byref(opts)))
    assert 0 < need <= b.SS_NOALLOC_SCRATCH_BYTES, need  # the chunked path, with scratch
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    out_ws = torch.empty_like(t["u"])
    last_ws = torch.empty_like(last_na)
    b.check(lib.ss_selective_scan_fwd_opts(*_call_args(t, wl, out_ws, last_ws), _ptr(ws), need,
                                           ctypes.byref(opts), stream))
    torch.cuda.synchronize()
    return (out_na, last_na), (out_ws, last_ws)


def _compare(wl, got, want):
    """Both entry points run the same kernels with the same L-chunks on the same
    inputs, so their results must be identical bit for bit; a stale word of the
    shared scratch would show up here even where it stays within the tolerance."""
    import torch
    (o1, l1), (o2, l2) = got, want
    assert torch.equal(o1.view(torch.int16) if o1.dtype == torch.bfloat16 else o1.view(torch.int32),
                       o2.view(torch.int16) if o2.dtype == torch.bfloat16 else o2.view(torch.int32)), \
        f"out differs: max relative difference {sc.rel_err(sc.from_torch(o1), sc.from_torch(o2)):.3e}"
    assert torch.equal(l1.view(torch.int32), l2.view(torch.int32)), "last_state differs"


@pytest.mark.parametrize("chunks", [4, 0])
def test_noalloc_matches_workspace_entry_point_two_calls(lib, chunks):
    """Forced four L-chunks, and the automatic choice on a long sequence with
    few rows (which also takes the chunked path); two calls in a row with
    different inputs, each checked against the workspace entry point."""
    wl = sc.workload("noalloc", 1, 96, 16384, io="bf16")
    for seed in (0, 1):
        na, ws = _run_both(lib, wl, seed, chunks)
        _compare(wl, na, ws)


def test_noalloc_float32_two_calls(lib):
    wl = sc.workload("noalloc_f32", 2, 40, 4096, io="f32")
    for seed in (3, 4):
        na, ws = _run_both(lib, wl, seed, 3)
        _compare(wl, na, ws)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    """A split that would need more scratch than the fixed array is refused on
    the host with SS_ERR_UNSUPPORTED, before anything is launched."""
    import torch
    from selective_state_space_120_b300 import _binding as b
    wl = sc.workload("too_big", 8, 1536, 2048, io="bf16")
    opts = b.options(64)
    need = int(lib.ss_workspace_bytes_opts(b.SS_KIND_SCAN, wl.batch, wl.dim, wl.L, wl.N,
                                           ctypes.byref(opts)))
    assert need > b.SS_NOALLOC_SCRATCH_BYTES
    t = _device(wk.make_inputs(wl))
    out = torch.empty_like(t["u"])
    st = lib.ss_selective_scan_fwd_noalloc(*_call_args(t, wl, out, None), ctypes.byref(opts),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == b.SS_ERR_UNSUPPORTED
    assert "scratch" in b.last_error()
