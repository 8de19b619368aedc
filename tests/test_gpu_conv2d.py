"""GPU parity of the SS2D block's input branch (ss_dwconv3x3_silu_fwd: depthwise
3 x 3 convolution with zero padding, bias, SiLU) against the float64 oracle,
alone and chained into the four-direction scan (B300 only).  Tolerances as for
the scans: max |y - y_ref| / (1 + |y_ref|) <= 1e-4 (float32 I/O), 2e-2 (bf16)."""
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


def _inputs(batch, dim, H, W, io, seed=7):
    wl = wk.Workload(f"dw{H}x{W}", batch, dim, H * W, K=4, io=io, H=H, W=W, conv2d=True)
    return wl, wk.make_inputs(wl, seed=seed)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(2, 24, 7, 9), (1, 8, 56, 56), (1, 4, 130, 70), (1, 3, 1, 1),
                                   (2, 5, 1, 33), (1, 2, 17, 1), (1, 3, 200, 24), (1, 2, 9, 300),
                                   (1, 2, 40, 260)])
def test_dwconv3x3_silu(oracle, io, shape):
    """Band kernel: whole planes, several bands (200 x 24), rows of 16-byte
    multiples or not, 1-wide maps; tile kernel (maps wider than 256): tiles cut
    short on both axes."""
    import selective_state_space_120_b300 as ss
    batch, dim, H, W = shape
    wl, inp = _inputs(batch, dim, H, W, io)
    x = sc.to_torch(inp.u).view(batch, dim, H, W)
    u = ss.dwconv3x3_silu(x, sc.to_torch(inp.conv2d_w), sc.to_torch(inp.conv2d_b))
    ref = oracle.dwconv3x3_silu(inp.as_f64("u").reshape(batch, dim, H, W),
                                inp.conv2d_w.astype(np.float64), inp.conv2d_b.astype(np.float64))
    sc.assert_close(sc.from_torch(u), ref, io)


def test_dwconv_without_bias(oracle):
    import selective_state_space_120_b300 as ss
    wl, inp = _inputs(2, 6, 12, 20, "f32")
    x = sc.to_torch(inp.u).view(2, 6, 12, 20)
    u = ss.dwconv3x3_silu(x, sc.to_torch(inp.conv2d_w))
    ref = oracle.dwconv3x3_silu(inp.as_f64("u").reshape(2, 6, 12, 20), inp.conv2d_w.astype(np.float64))
    sc.assert_close(sc.from_torch(u), ref, "f32")


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_ss2d_block_input_branch(oracle, io):
    """DWConv 3x3 -> SiLU -> SS2D on the GPU against the oracle's convolution
    followed by its four-direction scan (the bf16 case also rounds u to bf16
    between the two calls, inside the tolerance)."""
    import selective_state_space_120_b300 as ss
    batch, dim, H, W = 2, 16, 12, 16
    wl, inp = _inputs(batch, dim, H, W, io)
    t = sc.device_inputs(inp)
    x = t["u"].view(batch, dim, H, W)
    u = ss.dwconv3x3_silu(x, sc.to_torch(inp.conv2d_w), sc.to_torch(inp.conv2d_b))
    out = ss.cross_scan2d_fwd(u, t["delta"], t["A"], t["B"], t["C"], t["D"], t["delta_bias"], True,
                              z=t["z"].view(batch, dim, H, W))
    u_ref = oracle.dwconv3x3_silu(inp.as_f64("u").reshape(batch, dim, H, W),
                                  inp.conv2d_w.astype(np.float64), inp.conv2d_b.astype(np.float64))
    ref, _ = oracle.scan(u_ref.reshape(batch, dim, H * W), inp.as_f64("delta"), inp.as_f64("A"),
                         inp.as_f64("B"), inp.as_f64("C"), inp.as_f64("D"), inp.as_f64("z"),
                         inp.as_f64("delta_bias"), True, oracle.SS2D_ORDERS, H=H, W=W)
    sc.assert_close(sc.from_torch(out).reshape(batch, dim, H * W), ref, io)
