"""GPU parity of the any-order multi-direction scan (ss_multi_scan_fwd) against
the float64 oracle: LocalMamba's windowed traversals, VideoMamba's
spatio-temporal scans of a clip taken as a frames x pixels map, and mixed
order lists (B300 only).  Tolerances as for the other scans:
max |y - y_ref| / (1 + |y_ref|) <= 1e-4 (float32 I/O), 2e-2 (bf16 I/O)."""
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


def _oracle_order(oracle, code):
    import selective_state_space_120_b300 as ss
    return {ss.DIR_ROW: oracle.ORDER_FWD, ss.DIR_COL: oracle.ORDER_COL,
            ss.DIR_ROW_REV: oracle.ORDER_REV, ss.DIR_COL_REV: oracle.ORDER_COL_REV,
            ss.DIR_WIN: oracle.ORDER_WIN, ss.DIR_WIN_COL: oracle.ORDER_WIN_COL,
            ss.DIR_WIN_REV: oracle.ORDER_WIN_REV, ss.DIR_WIN_COL_REV: oracle.ORDER_WIN_COL_REV}[code]


def _check(oracle, H, W, orders, window, batch=2, dim=24, N=16, G=1, io="bf16", with_z=True):
    import selective_state_space_120_b300 as ss
    K = len(orders)
    wl = sc.workload(f"ord{H}x{W}k{K}", batch, dim, H * W, N=N, G=G, K=K, io=io, with_z=with_z,
                     H=H, W=W)
    inp = wk.make_inputs(wl, seed=5)
    t = sc.device_inputs(inp)
    z = None if t["z"] is None else t["z"].view(batch, dim, H, W)
    out, last = ss.multi_scan_fwd(t["u"].view(batch, dim, H, W), t["delta"], t["A"], t["B"], t["C"],
                                  orders, window, t["D"], t["delta_bias"], True, z=z,
                                  return_last_state=True)
    ref, ref_last = oracle.scan(inp.as_f64("u"), inp.as_f64("delta"), inp.as_f64("A"),
                                inp.as_f64("B"), inp.as_f64("C"), inp.as_f64("D"), inp.as_f64("z"),
                                inp.as_f64("delta_bias"), True,
                                [_oracle_order(oracle, o) for o in orders], H=H, W=W, win=window)
    sc.assert_close(sc.from_torch(out).reshape(batch, dim, H * W), ref, io)
    sc.assert_close(last.cpu().numpy().astype(np.float64), ref_last, io, "last_state")


def _windowed():
    import selective_state_space_120_b300 as ss
    return [ss.DIR_WIN, ss.DIR_WIN_COL, ss.DIR_WIN_REV, ss.DIR_WIN_COL_REV]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("H,W,w", [(8, 12, 2), (7, 8, 3), (16, 16, 4)])
def test_windowed_directions(oracle, io, H, W, w):
    """Four windowed directions; 7 x 8 with 3 x 3 windows cuts the last band of
    rows and the last column short."""
    _check(oracle, H, W, _windowed(), w, io=io)


def test_windowed_56x56_w7(oracle):
    """The VMamba-T stage-1 map with 7 x 7 windows, several channel blocks and tiles."""
    _check(oracle, 56, 56, _windowed(), 7, batch=1, dim=40)


def test_video_spatiotemporal_orders(oracle):
    """A clip of 4 frames of 6 x 6 pixels as a 4 x 36 map: spatial-first
    (frame by frame) and temporal-first (pixel by pixel through the frames)
    scans, both ways."""
    import selective_state_space_120_b300 as ss
    _check(oracle, 4, 36, [ss.DIR_ROW, ss.DIR_ROW_REV, ss.DIR_COL, ss.DIR_COL_REV], 0)


@pytest.mark.parametrize("N", [4, 32])
def test_all_eight_orders_and_groups(oracle, N):
    import selective_state_space_120_b300 as ss
    _check(oracle, 8, 8, list(range(8)), 3, dim=32, N=N, G=2, io="f32")


@pytest.mark.parametrize("orders", [[4], [7], [0, 5, 6]])
def test_fewer_directions_and_no_gate(oracle, orders):
    _check(oracle, 6, 12, orders, 4, with_z=False)
