"""Host-side checks of the C ABI (no kernel is launched).

The library loads and exports every function include/ssscan.h declares; bad
arguments are rejected with the documented status before anything is
enqueued; workspace sizing is a host computation.  The calls with fake
addresses all fail validation; they run only where no GPU is present, so that
a validation bug could never hand a fake address to a kernel.
"""
import ctypes
import os
import re

import pytest

from selective_state_space_120_b300 import _binding as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssscan.h")


def _gpu_present():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # noqa: BLE001
        return False


fake_ptrs = pytest.mark.skipif(_gpu_present(), reason="fake-address checks run on CPU hosts only")


@pytest.fixture(scope="module")
def lib():
    from selective_state_space_120_b300 import build
    build.build()
    return b.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:ss_status|size_t|const char \*)\s*(ss_\w+)\s*\(", text,
                                 re.M)))


def test_header_declarations_match_binding():
    assert _declared() == sorted(b.EXPORTS)


def test_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
    assert b.version().startswith("ssscan")


A16 = 0x10000  # a 16-byte aligned fake address


def _scan(lib, batch=1, dim=8, L=32, N=16, G=1, io=b.SS_BF16, u=A16, delta=A16 + 0x100000,
          A=A16 + 0x200000, B=A16 + 0x300000, C=A16 + 0x400000, D=None, z=None, bias=None,
          out=A16 + 0x500000, last=None, ws=None, wsb=0):
    return lib.ss_selective_scan_fwd(batch, dim, L, N, G, io, u, delta, A, B, C, D, z, bias, 1,
                                     out, last, ws, wsb, None)


@fake_ptrs
def test_rejects_null_required_pointers(lib):
    assert _scan(lib, u=None) == b.SS_ERR_INVALID_ARG
    assert _scan(lib, B=None) == b.SS_ERR_INVALID_ARG
    assert _scan(lib, out=None) == b.SS_ERR_INVALID_ARG
    assert "required" in b.last_error()


@fake_ptrs
def test_rejects_bad_sizes(lib):
    assert _scan(lib, batch=-1, out=None) == b.SS_ERR_INVALID_ARG
    assert _scan(lib, dim=6, G=4, out=None) == b.SS_ERR_INVALID_ARG      # 6 % 4 != 0
    assert _scan(lib, G=0, out=None) == b.SS_ERR_INVALID_ARG


@fake_ptrs
@pytest.mark.parametrize("N", [0, 3, 5, 12, 128])
def test_rejects_unsupported_dstate(lib, N):
    assert _scan(lib, N=N, out=None) == b.SS_ERR_UNSUPPORTED


@fake_ptrs
def test_rejects_unknown_dtype(lib):
    assert _scan(lib, io=7, out=None) == b.SS_ERR_UNSUPPORTED


@fake_ptrs
def test_rejects_misaligned_pointers(lib):
    assert _scan(lib, u=A16 + 2) == b.SS_ERR_ALIGNMENT
    assert _scan(lib, z=A16 + 0x600008) == b.SS_ERR_ALIGNMENT
    assert _scan(lib, out=A16 + 0x500004) == b.SS_ERR_ALIGNMENT


@fake_ptrs
def test_rejects_out_aliasing_inputs(lib):
    assert _scan(lib, out=A16) == b.SS_ERR_INVALID_ARG                  # out == u
    assert _scan(lib, out=A16 + 0x100000 + 64) == b.SS_ERR_INVALID_ARG  # inside delta
    assert "overlap" in b.last_error()


@fake_ptrs
def test_rejects_missing_workspace_on_chunked_path(lib):
    opts = b.options(chunks=4)
    need = b.workspace_bytes(b.SS_KIND_SCAN, 1, 8, 4096, 16, chunks=4)
    assert need > 0
    args = (1, 8, 4096, 16, 1, b.SS_BF16, A16, A16 + 0x100000, A16 + 0x200000, A16 + 0x300000,
            A16 + 0x400000, None, None, None, 1, A16 + 0x500000, None)
    st = lib.ss_selective_scan_fwd_opts(*args, None, 0, ctypes.byref(opts), None)
    assert st == b.SS_ERR_WORKSPACE
    st = lib.ss_selective_scan_fwd_opts(*args, A16 + 0x700000, need - 1, ctypes.byref(opts), None)
    assert st == b.SS_ERR_WORKSPACE
    st = lib.ss_selective_scan_fwd_opts(*args, A16 + 0x700008, need, ctypes.byref(opts), None)
    assert st == b.SS_ERR_ALIGNMENT


@fake_ptrs
def test_rejects_nonzero_reserved_options(lib):
    opts = b.options()
    opts.reserved[3] = 1
    st = lib.ss_selective_scan_fwd_opts(1, 8, 32, 16, 1, b.SS_BF16, A16, A16 + 0x100000,
                                        A16 + 0x200000, A16 + 0x300000, A16 + 0x400000, None, None,
                                        None, 1, A16 + 0x500000, None, None, 0, ctypes.byref(opts),
                                        None)
    assert st == b.SS_ERR_INVALID_ARG


@fake_ptrs
def test_empty_inputs_return_ok_without_pointers(lib):
    assert _scan(lib, batch=0, u=None, delta=None, A=None, B=None, C=None, out=None) == b.SS_OK
    assert _scan(lib, L=0, u=None, delta=None, A=None, B=None, C=None, out=None) == b.SS_OK
    st = lib.ss_cross_scan2d_fwd(2, 4, 0, 5, 16, 1, b.SS_BF16, None, None, None, None, None, None,
                                 None, 1, None, None, None, None, 0, None)
    assert st == b.SS_OK


@fake_ptrs
def test_bidir_and_cross2d_validate(lib):
    st = lib.ss_bidir_scan_fwd(1, 8, 32, 16, 1, b.SS_BF16, A16, None, A16, A16, A16, None, None,
                               None, 1, A16 + 0x500000, None, None, 0, None)
    assert st == b.SS_ERR_INVALID_ARG
    st = lib.ss_cross_scan2d_fwd(1, 8, -3, 4, 16, 1, b.SS_BF16, A16, A16, A16, A16, A16, None,
                                 None, 1, None, A16 + 0x500000, None, None, 0, None)
    assert st == b.SS_ERR_INVALID_ARG
    st = lib.ss_cross_scan2d_fwd(1, 8, 3, 4, 12, 1, b.SS_BF16, A16, A16, A16, A16, A16, None,
                                 None, 1, None, A16 + 0x500000, None, None, 0, None)
    assert st == b.SS_ERR_UNSUPPORTED


@fake_ptrs
def test_scan_options_are_validated(lib):
    base = (1, 8, 32, 16, 1, b.SS_BF16, A16, A16 + 0x100000, A16 + 0x200000, A16 + 0x300000,
            A16 + 0x400000, None, None, None, 1, A16 + 0x500000, None, None, 0)
    bad_flag = b.options(flags=4)
    assert lib.ss_selective_scan_fwd_opts(*base, ctypes.byref(bad_flag), None) == b.SS_ERR_INVALID_ARG
    assert "flags" in b.last_error()
    bad_h0 = b.options(h0=A16 + 0x600004)
    assert lib.ss_selective_scan_fwd_opts(*base, ctypes.byref(bad_h0), None) == b.SS_ERR_ALIGNMENT
    h0_on_out = b.options(h0=A16 + 0x500000)
    assert lib.ss_selective_scan_fwd_opts(*base, ctypes.byref(h0_on_out), None) == b.SS_ERR_INVALID_ARG
    no_w = b.options(flags=b.SS_SCAN_CONV_SILU)
    assert lib.ss_selective_scan_fwd_opts(*base, ctypes.byref(no_w), None) == b.SS_ERR_INVALID_ARG
    w_no_flag = b.options(conv_w=A16 + 0x700000)
    assert lib.ss_selective_scan_fwd_opts(*base, ctypes.byref(w_no_flag), None) == b.SS_ERR_INVALID_ARG
    unaligned_rows = list(base)
    unaligned_rows[2] = 33                  # 66-byte rows: no fused conv
    conv = b.options(flags=b.SS_SCAN_CONV_SILU, conv_w=A16 + 0x700000)
    assert lib.ss_selective_scan_fwd_opts(*unaligned_rows, ctypes.byref(conv), None) == b.SS_ERR_UNSUPPORTED
    assert ctypes.sizeof(b.ScanOptions) == 64


@fake_ptrs
def test_state_update_validates(lib):
    args = [2, 8, 16, 1, b.SS_BF16, A16, A16 + 0x1000, A16 + 0x2000, A16 + 0x3000, A16 + 0x4000,
            None, None, None, 1, 0, A16 + 0x5000, A16 + 0x6000, None]
    bad = list(args); bad[15] = None           # no state
    assert lib.ss_selective_state_update(*bad) == b.SS_ERR_INVALID_ARG
    bad = list(args); bad[15] = A16 + 0x5004   # misaligned state
    assert lib.ss_selective_state_update(*bad) == b.SS_ERR_ALIGNMENT
    bad = list(args); bad[14] = 2              # unknown flag
    assert lib.ss_selective_state_update(*bad) == b.SS_ERR_INVALID_ARG
    bad = list(args); bad[2] = 12              # unsupported dstate
    assert lib.ss_selective_state_update(*bad) == b.SS_ERR_UNSUPPORTED


@fake_ptrs
def test_debug_flags_reject_unknown_bits(lib):
    assert lib.ss_debug_set_flags(2) == b.SS_ERR_INVALID_ARG
    assert "unknown flag" in b.last_error()


def test_workspace_sizing_is_host_only(lib):
    # multi-direction calls: unaligned bidirectional rows are read through view tiles (both
    # directions' terms, fp32 [2, rows, Lp]) or re-pitched; the size covers the re-pitched path
    # (with ngroups = 1: the terms, u forward and reversed, Delta of both directions [rows, Lp]
    # each in the I/O type, B and C [batch*2*N, Lp]; Lp = L rounded up to 16 bytes, the larger of
    # the two dtypes: float32);
    # aligned rows merge through an fp32 [batch, dim, L] accumulator
    rows, Lp = 128 * 768, 200
    a256 = lambda n: (n + 255) // 256 * 256  # noqa: E731
    want = (a256(2 * rows * Lp * 4) + 2 * a256(rows * Lp * 4) + a256(2 * rows * Lp * 4) +
            2 * a256(128 * 2 * 16 * Lp * 4))
    assert b.workspace_bytes(b.SS_KIND_BIDIR, 128, 768, 197, 16) == want
    # (SS2D: four fp32 slices, one per direction, and a transposed copy of u for
    # the column directions)
    assert b.workspace_bytes(b.SS_KIND_CROSS2D, 32, 192, 3136, 16) == 5 * 32 * 192 * 3136 * 4
    assert b.workspace_bytes(b.SS_KIND_BIDIR, 2, 24, 256, 16) == 2 * 24 * 256 * 4
    # plenty of batch*dim parallelism: single pass, no workspace
    assert b.workspace_bytes(b.SS_KIND_SCAN, 8, 1536, 2048, 16) == 0
    # forced chunks: hend + carry (N floats each) + one float per row and chunk
    need = b.workspace_bytes(b.SS_KIND_SCAN, 2, 8, 4096, 16, chunks=4)
    assert need == 2 * 8 * 4 * (2 * 16 + 1) * 4
    assert b.workspace_bytes(b.SS_KIND_SCAN, 0, 8, 4096, 16) == 0
    # long sequence with few rows: the automatic choice splits it
    assert b.workspace_bytes(b.SS_KIND_SCAN, 1, 5120, 131072, 16) > 0


def _bwd_args(batch=1, dim=8, L=32, N=16, G=1, io=b.SS_BF16, **kw):
    """Arguments of ss_selective_scan_bwd with fake aligned addresses, each
    tensor in its own 1 MiB window; keyword overrides by name."""
    names = ("u", "delta", "A", "B", "C", "D", "z", "bias", "dout", "du", "ddelta", "dA", "dB",
             "dC", "dD", "dz", "dbias", "ws")
    ptr = {n: A16 + i * 0x100000 for i, n in enumerate(names)}
    for n in ("D", "z", "bias", "dD", "dz", "dbias"):
        ptr[n] = None
    wsb = kw.pop("wsb", b.workspace_bytes(b.SS_KIND_SCAN_BWD, batch, dim, L, N))
    ptr.update(kw)
    return (batch, dim, L, N, G, io, ptr["u"], ptr["delta"], ptr["A"], ptr["B"], ptr["C"],
            ptr["D"], ptr["z"], ptr["bias"], 1, ptr["dout"], ptr["du"], ptr["ddelta"], ptr["dA"],
            ptr["dB"], ptr["dC"], ptr["dD"], ptr["dz"], ptr["dbias"], ptr["ws"], wsb, None)


@fake_ptrs
def test_backward_validates(lib):
    bwd = lib.ss_selective_scan_bwd
    assert bwd(*_bwd_args(dout=None)) == b.SS_ERR_INVALID_ARG
    assert bwd(*_bwd_args(dC=None)) == b.SS_ERR_INVALID_ARG
    # dz exactly when z is given
    assert bwd(*_bwd_args(z=A16 + 0x6_000000)) == b.SS_ERR_INVALID_ARG
    assert "dz is required" in b.last_error()
    assert bwd(*_bwd_args(dz=A16 + 0x6_000000)) == b.SS_ERR_INVALID_ARG
    assert bwd(*_bwd_args(dB=A16 + 0x4_000008)) == b.SS_ERR_ALIGNMENT
    # rows of 20 bf16 values are not 16-byte aligned
    assert bwd(*_bwd_args(L=20)) == b.SS_ERR_UNSUPPORTED
    assert bwd(*_bwd_args(N=12)) == b.SS_ERR_UNSUPPORTED
    # a gradient output on top of an input, or two outputs on top of each other
    assert bwd(*_bwd_args(du=A16 + 0x100000)) == b.SS_ERR_INVALID_ARG
    assert bwd(*_bwd_args(dA=A16 + 0xa00000)) == b.SS_ERR_INVALID_ARG
    assert bwd(*_bwd_args(ws=A16 + 0x900000)) == b.SS_ERR_INVALID_ARG
    # workspace missing or short
    assert bwd(*_bwd_args(ws=None)) == b.SS_ERR_WORKSPACE
    assert bwd(*_bwd_args(wsb=b.workspace_bytes(b.SS_KIND_SCAN_BWD, 1, 8, 32, 16) - 1)) == \
        b.SS_ERR_WORKSPACE


@fake_ptrs
def test_backward_with_options_validates(lib):
    """ss_selective_scan_bwd_opts: the options as the forward call validates
    them, plus the gradients of their tensors."""
    def call(chunks=0, flags=0, h0=None, conv_w=None, conv_b=None, conv_x0=None, dh0=None,
             dconv_w=None, dconv_b=None, dconv_x0=None, wsb=None, reserved=0):
        o = b.options(chunks, flags, h0, conv_w, conv_b, conv_x0)
        ex = b.BwdExtras()
        ex.dh0, ex.dconv_w, ex.dconv_b, ex.dconv_x0 = dh0, dconv_w, dconv_b, dconv_x0
        ex.reserved[0] = reserved
        args = list(_bwd_args())
        if wsb is not None:
            args[-2] = wsb
        return lib.ss_selective_scan_bwd_opts(*args[:-3], ctypes.byref(o), ctypes.byref(ex),
                                              *args[-3:])
    F = A16 + 0x2000000  # a free window
    assert call(chunks=2) == b.SS_ERR_INVALID_ARG                       # no sequence split here
    assert call(dh0=F) == b.SS_ERR_INVALID_ARG                          # dh0 without h0
    assert "h0" in b.last_error()
    assert call(flags=b.SS_SCAN_CONV_SILU, conv_w=F) == b.SS_ERR_INVALID_ARG  # dconv_w missing
    assert call(dconv_w=F + 0x100000) == b.SS_ERR_INVALID_ARG           # conv gradient, no conv
    assert call(flags=b.SS_SCAN_CONV_SILU, conv_w=F, dconv_w=F + 0x100000,
                dconv_b=F + 0x200000) == b.SS_ERR_INVALID_ARG           # dconv_b without conv_b
    assert call(h0=F, dh0=F + 0x100008) == b.SS_ERR_ALIGNMENT
    assert call(reserved=1) == b.SS_ERR_INVALID_ARG
    assert call(flags=4) == b.SS_ERR_INVALID_ARG                        # unknown flag
    # the Conv1D path needs room for the recomputed u and its gradient too
    o = b.options(0, b.SS_SCAN_CONV_SILU, None, F)
    need = int(lib.ss_workspace_bytes_opts(b.SS_KIND_SCAN_BWD, 1, 8, 32, 16, ctypes.byref(o)))
    assert need == 8 * 4 * 16 * 4 + 2 * 8 * 32 * 4  # checkpoints + u + du, fp32 (256-aligned)
    assert call(flags=b.SS_SCAN_CONV_SILU, conv_w=F, dconv_w=F + 0x100000,
                wsb=need - 1) == b.SS_ERR_WORKSPACE


def test_backward_workspace_holds_a_checkpoint_per_8_steps(lib):
    # [batch*dim, ceil(L/8), N] float32
    assert b.workspace_bytes(b.SS_KIND_SCAN_BWD, 8, 1536, 2048, 16) == 8 * 1536 * 256 * 16 * 4
    assert b.workspace_bytes(b.SS_KIND_SCAN_BWD, 2, 3, 17, 4) == 2 * 3 * 3 * 4 * 4
    assert b.workspace_bytes(b.SS_KIND_SCAN_BWD, 2, 3, 0, 4) == 0
    assert b.workspace_bytes(b.SS_KIND_SCAN_BWD, 2, 3, 64, 12) == 0


@fake_ptrs
def test_multi_scan_validates(lib):
    def call(ndirs=2, orders=(b.SS_DIR_WIN, b.SS_DIR_ROW), window=2, H=4, W=8, wsb=None, ws=A16 + 0x900000):
        ords = (ctypes.c_int * max(1, len(orders)))(*orders)
        if wsb is None:
            wsb = b.load().ss_multi_scan_workspace_bytes(1, 8, H, W, ndirs)
        return lib.ss_multi_scan_fwd(1, 8, H, W, ndirs, ords, window, 16, 1, b.SS_BF16, A16,
                                     A16 + 0x100000, A16 + 0x200000, A16 + 0x300000, A16 + 0x400000,
                                     None, None, 1, None, A16 + 0x500000, None, ws, wsb, None)
    assert call(ndirs=0) == b.SS_ERR_INVALID_ARG
    assert call(ndirs=9, orders=(0,) * 9) == b.SS_ERR_INVALID_ARG
    assert call(orders=(b.SS_DIR_WIN, 8)) == b.SS_ERR_INVALID_ARG
    assert "SS_DIR_" in b.last_error()
    assert call(window=0) == b.SS_ERR_INVALID_ARG          # a windowed order needs a window
    assert call(H=3, W=5) == b.SS_ERR_UNSUPPORTED          # rows of 15 bf16 values
    assert call(ws=None) == b.SS_ERR_WORKSPACE
    # (WIN, ROW) needs the two accumulators and one bf16 copy of u in window order
    need = 2 * 8 * 32 * 4 + 8 * 32 * 2
    assert call(wsb=need - 4) == b.SS_ERR_WORKSPACE
    assert call(ws=A16 + 0x100000) == b.SS_ERR_INVALID_ARG  # workspace on top of delta
    # the bound: three accumulators and three fp32-sized copies
    assert b.load().ss_multi_scan_workspace_bytes(2, 8, 4, 8, 3) == 3 * 2 * 8 * 32 * 4 + 3 * 2 * 8 * 32 * 4
    assert b.load().ss_multi_scan_workspace_bytes(2, 8, 4, 8, 8) == 8 * 2 * 8 * 32 * 4 + 3 * 2 * 8 * 32 * 4


@fake_ptrs
def test_dwconv_validates(lib):
    args = [1, 4, 8, 8, b.SS_BF16, A16, A16 + 0x100000, None, A16 + 0x200000, None]
    bad = list(args); bad[5] = None
    assert lib.ss_dwconv3x3_silu_fwd(*bad) == b.SS_ERR_INVALID_ARG
    bad = list(args); bad[8] = A16 + 0x40
    assert lib.ss_dwconv3x3_silu_fwd(*bad) == b.SS_ERR_INVALID_ARG     # u on top of x
    bad = list(args); bad[7] = A16 + 0x300004
    assert lib.ss_dwconv3x3_silu_fwd(*bad) == b.SS_ERR_ALIGNMENT
    bad = list(args); bad[4] = 7
    assert lib.ss_dwconv3x3_silu_fwd(*bad) == b.SS_ERR_UNSUPPORTED
    bad = list(args); bad[2] = 0
    assert lib.ss_dwconv3x3_silu_fwd(*bad) == b.SS_OK                  # empty: nothing to do


@fake_ptrs
def test_multi_scan_bwd_validates(lib):
    def call(ndirs=2, orders=(b.SS_DIR_ROW, b.SS_DIR_COL), window=0, H=4, W=8, dz=None, z=None,
             wsb=None, ws=A16 + 0x2000000, du=A16 + 0x900000):
        ords = (ctypes.c_int * max(1, len(orders)))(*orders)
        if wsb is None:
            wsb = b.load().ss_multi_scan_bwd_workspace_bytes(1, 8, H, W, 16, ndirs)
        return lib.ss_multi_scan_bwd(1, 8, H, W, ndirs, ords, window, 16, 1, b.SS_BF16, A16,
                                     A16 + 0x100000, A16 + 0x200000, A16 + 0x300000,
                                     A16 + 0x400000, None, None, 1, z, A16 + 0x500000, du,
                                     A16 + 0xa00000, A16 + 0xb00000, A16 + 0xc00000,
                                     A16 + 0xd00000, None, dz, None, ws, wsb, None)
    assert call(orders=(b.SS_DIR_WIN, 1), window=0) == b.SS_ERR_INVALID_ARG
    assert call(z=A16 + 0x600000) == b.SS_ERR_INVALID_ARG           # dz missing
    assert call(dz=A16 + 0x700000) == b.SS_ERR_INVALID_ARG          # dz without z
    assert call(H=3, W=5) == b.SS_ERR_UNSUPPORTED
    assert call(ws=None) == b.SS_ERR_WORKSPACE
    assert call(du=A16 + 0x100000) == b.SS_ERR_INVALID_ARG          # du on top of delta
    assert b.load().ss_multi_scan_bwd_workspace_bytes(1, 8, 4, 8, 16, 2) > 0
