"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one slip in a private copy of the oracle's C source (a dropped
term, a flipped sign, a swapped operand, a wrong index map), builds it, and
runs every pin of ``test_oracle_pins`` against it: at least one pin must fail.
The product library is not involved.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle as _oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(_oracle.__file__), "ss_oracle.c")

MUTANTS = {
    "drop_skip_D": ("o_row[p] += y + Dd * up;", "o_row[p] += y;"),
    "flip_sign_of_A": ("const double abar = exp(dt * a);", "const double abar = exp(-dt * a);"),
    "no_state_decay": ("h[n] = abar * h[n] + bbar * up;", "h[n] = h[n] + bbar * up;"),
    "swap_B_for_C_in_input": ("bbar = dt * B_grp[n * L + s];", "bbar = dt * C_grp[n * L + s];"),
    "swap_C_for_B_in_readout": ("y += C_grp[n * L + s] * h[n];", "y += B_grp[n * L + s] * h[n];"),
    "drop_delta_bias": ("double dt = dl_row[s] + bd;", "double dt = dl_row[s];"),
    "softplus_without_log1p": ("log1p(exp(-fabs(x)))", "exp(-fabs(x))"),
    "sigmoid_instead_of_silu": ("out[i] *= zi / (1.0 + exp(-zi));", "out[i] *= 1.0 / (1.0 + exp(-zi));"),
    "reverse_off_by_one": ("case SSOR_ORDER_REV: return L - 1 - s;",
                           "case SSOR_ORDER_REV: return (L - s) % L;"),
    "column_map_transposed": ("case SSOR_ORDER_COL: return (s % H) * W + s / H;",
                              "case SSOR_ORDER_COL: return (s % W) * H + s / W;"),
    "zoh_divides_wrong_way": ("bbar = (abar - 1.0) / a * B_grp[n * L + s];",
                              "bbar = (abar - 1.0) * a * B_grp[n * L + s];"),
    "delta_by_position": ("double dt = dl_row[s] + bd;", "double dt = dl_row[p] + bd;"),
    "B_by_position": ("bbar = dt * B_grp[n * L + s];", "bbar = dt * B_grp[n * L + p];"),
    "conv_kernel_reversed": ("v += w[d * KW + j] * xv;", "v += w[d * KW + (KW - 1 - j)] * xv;"),
    "bwd_no_decay_of_dh": ("carry[n] = abar * dh;", "carry[n] = dh;"),
    "bwd_dA_missing_dt": ("dA[d * N + n] += dabar * abar * dt;", "dA[d * N + n] += dabar * abar;"),
    "bwd_dB_uses_C": ("dBg[n * L + t] += dh * dt * u[row + t];",
                      "dBg[n * L + t] += ds * dt * u[row + t];"),
    "bwd_softplus_derivative": ("1.0 / (1.0 + exp(-r)) : 1.0;", "1.0 / (1.0 + exp(r)) : 1.0;"),
    "conv_history_off_by_one": ("else xv = x0r ? x0r[(KW - 1) + s] : 0.0;",
                                "else xv = x0r ? x0r[(KW - 2) + s] : 0.0;"),
    "window_cells_transposed": ("for (int64_t c = c0; c < c0 + w && c < W; ++c) pos[s++] = r * W + c;",
                                "for (int64_t c = c0; c < c0 + w && c < W; ++c) pos[s++] = c * H + r;"),
    "window_reverse_missing": ("const int64_t t = pos[i];", "const int64_t t = pos[j];"),
    "dwconv_kernel_transposed": ("v += w[d * 9 + (i + 1) * 3 + (j + 1)] * xp[rr * W + cc];",
                                 "v += w[d * 9 + (j + 1) * 3 + (i + 1)] * xp[rr * W + cc];"),
    "group_map_interleaved": ("const int64_t g = d / dpg;", "const int64_t g = d % ngroups;"),
    "ignores_initial_state": ("h[n] = h0 ? h0[((b * K + k) * dim + d) * N + n] : 0.0;",
                              "h[n] = 0.0;"),
    "last_state_not_final": ("last_state[((b * K + k) * dim + d) * N + n] = h[n];",
                             "last_state[((b * K + k) * dim + d) * N + n] = h[n] * 0.5;"),
    "bwd_zoh_delta_uses_euler_input": ("ddt += dabar * abar * a + dh * abar * bu;",
                                       "ddt += dabar * abar * a + dh * bu;"),
    "bwd_h0_ignored_in_decay": (
        "const double prev = t ? h_work[(t - 1) * N + n] : (h0r ? h0r[n] : 0.0);\n"
        "                    const double dh = ds",
        "const double prev = t ? h_work[(t - 1) * N + n] : 0.0;\n"
        "                    const double dh = ds"),
    "conv_bwd_dw_missing_input": ("dw[d * KW + j] += xr[s] * dv;", "dw[d * KW + j] += dv;"),
    "conv_bwd_silu_derivative": ("sg * (1.0 + v * (1.0 - sg));", "sg;"),
}


class _Variant:
    """The oracle's Python API, bound to another build of the C source."""
    ORDER_FWD, ORDER_REV = _oracle.ORDER_FWD, _oracle.ORDER_REV
    ORDER_COL, ORDER_COL_REV = _oracle.ORDER_COL, _oracle.ORDER_COL_REV
    SS2D_ORDERS = _oracle.SS2D_ORDERS
    ORDER_WIN, ORDER_WIN_REV = _oracle.ORDER_WIN, _oracle.ORDER_WIN_REV
    ORDER_WIN_COL, ORDER_WIN_COL_REV = _oracle.ORDER_WIN_COL, _oracle.ORDER_WIN_COL_REV

    def __init__(self, path):
        self.lib = _oracle._bind(path)

    def scan(self, *a, **k):
        return _oracle.scan(*a, _lib_handle=self.lib, **k)

    def selective_scan(self, u, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=True, zoh=False, h0=None):
        out, last = self.scan(u, delta, A, B, C, D, z, delta_bias, delta_softplus,
                              (self.ORDER_FWD,), zoh=zoh, h0=h0)
        return out, last[:, 0]

    def bidir_scan(self, u, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True):
        return self.scan(u, delta, A, B, C, D, z, delta_bias, delta_softplus,
                         (self.ORDER_FWD, self.ORDER_REV))

    def selective_scan_bwd(self, *a, **k):
        real = _oracle._load
        _oracle._load = lambda: self.lib
        try:
            return _oracle.selective_scan_bwd(*a, **k)
        finally:
            _oracle._load = real

    def multi_scan_bwd(self, *a, **k):
        real = _oracle._load
        _oracle._load = lambda: self.lib
        try:
            return _oracle.multi_scan_bwd(*a, **k)
        finally:
            _oracle._load = real

    def conv_silu_bwd(self, *a, **k):
        real = _oracle._load
        _oracle._load = lambda: self.lib
        try:
            return _oracle.conv_silu_bwd(*a, **k)
        finally:
            _oracle._load = real

    def conv_silu(self, x, w, bias=None, x0=None):
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        batch, dim, L = x.shape
        w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        KW = w.shape[1]
        bias = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
        x0 = None if x0 is None else np.ascontiguousarray(np.asarray(x0, dtype=np.float64))
        u = np.empty_like(x)
        rc = self.lib.ssor_conv_silu(batch, dim, L, KW, _oracle._ptr(x), _oracle._ptr(w),
                                     _oracle._ptr(bias), _oracle._ptr(x0), _oracle._ptr(u))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return u

    def dwconv3x3_silu(self, x, w, bias=None):
        x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
        batch, dim, H, W = x.shape
        w = np.ascontiguousarray(np.asarray(w, dtype=np.float64))
        bias = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float64))
        u = np.empty_like(x)
        rc = self.lib.ssor_dwconv3x3_silu(batch, dim, H, W, _oracle._ptr(x), _oracle._ptr(w),
                                          _oracle._ptr(bias), _oracle._ptr(u))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return u

    def softplus(self, x):
        return self.lib.ssor_softplus_scalar(float(x))

    def position(self, order, s, H, W):
        return self.lib.ssor_position_of(int(order), int(s), int(H), int(W))

    def order_table(self, order, H, W, win=0):
        pos = np.empty(H * W, dtype=np.int64)
        rc = self.lib.ssor_order_table(int(order), int(H), int(W), int(win),
                                       pos.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return pos


def _pin_calls():
    calls = []
    for name in dir(pins):
        if not name.startswith("test_"):
            continue
        fn = getattr(pins, name)
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if params:
            argnames = [a.strip() for a in params[0].args[0].split(",")]
            for vals in params[0].args[1]:
                calls.append((f"{name}{vals}", fn, dict(zip(argnames, vals))))
        else:
            calls.append((name, fn, {}))
    return calls


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_mutant(mutant, tmp_path):
    old, new = MUTANTS[mutant]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor not found once: {old!r}"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", str(so), str(mpath), "-lm"])
    variant = _Variant(str(so))
    failed = []
    for label, fn, kwargs in _pin_calls():
        try:
            with np.errstate(all="ignore"):
                fn(variant, **kwargs)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(label)
    assert failed, f"no pin caught the mutant {mutant}"
