"""GPU parity at the benchmark's full sizes, in the launch configurations the
benchmark times, for the paths the other full-size cases do not cover: the
windowed four-direction scan, the Mamba layer with its fused Conv1D + SiLU,
the SS2D block's DWConv 3x3 + SiLU, the backward pass of the SS2D and
windowed scans, and token-by-token decoding (B300 only).

The oracle computes sampled channels one by one (every scan channel depends on
its own inputs and on B, C of its group only); the backward pass is checked on
every gradient of batch 0 and on the batch sums of eight channels.  Tolerances
are those of the smaller cases: max |y - y_ref| / (1 + |y_ref|) <= 2e-2 for
bf16 outputs, and max |g - r| / (rms(r) + |r|) <= 1e-2 for bf16 gradients."""
import numpy as np
import pytest

from selective_state_space_120_b300 import workloads as wk
from tests import scan_cases as sc
from tests.test_gpu_bwd import _dout_f64, _oracle_order, assert_grads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import selective_state_space_120_b300 as ss
    ss.load_library()


def _rows(wl, n=10, seed=3):
    rng = np.random.default_rng(seed)
    rows = [(int(rng.integers(wl.batch)), int(rng.integers(wl.dim))) for _ in range(n)]
    return rows + [(0, 0), (wl.batch - 1, wl.dim - 1)]


def _row_inputs(f, wl, b, d):
    """The inputs of channel d of batch b alone, as a one-channel problem."""
    K, dpg = wl.K, wl.dim // wl.G
    g = d // dpg
    sel = [k * wl.dim + d for k in range(K)]
    return dict(u=f["u"][b:b + 1, d:d + 1], delta=f["delta"][b:b + 1, :, d:d + 1], A=f["A"][sel],
                B=f["B"][b:b + 1, :, g:g + 1], C=f["C"][b:b + 1, :, g:g + 1],
                D=None if f["D"] is None else f["D"][sel],
                z=None if f["z"] is None else f["z"][b:b + 1, d:d + 1],
                delta_bias=f["delta_bias"][sel])


def _f64(inp):
    return {n: inp.as_f64(n) for n in ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")}


def test_windowed_full_size_sampled(oracle):
    """LocalMamba's four windowed directions (7 x 7 windows) on 32 x 192 x 56 x 56."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = wk.LOCAL_WIN
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    out, last = ss.multi_scan_fwd(t["u"].view(wl.batch, wl.dim, wl.H, wl.W), t["delta"], t["A"],
                                  t["B"], t["C"], list(wl.orders), wl.win, t["D"],
                                  t["delta_bias"], True, return_last_state=True)
    torch.cuda.synchronize()
    f = _f64(inp)
    orders = [_oracle_order(oracle, o) for o in wl.orders]
    rows = _rows(wl)
    refs, ref_lasts = [], []
    for b, d in rows:
        r = _row_inputs(f, wl, b, d)
        o, l = oracle.scan(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"], r["z"],
                           r["delta_bias"], True, orders, H=wl.H, W=wl.W, win=wl.win)
        refs.append(o[0, 0])
        ref_lasts.append(l[0, :, 0])
    o2 = out.view(wl.batch, wl.dim, wl.L)
    got = np.stack([sc.from_torch(o2[b, d]) for b, d in rows])
    sc.assert_close(got, np.stack(refs), wl.io)
    got_l = np.stack([last[b, :, d].cpu().numpy() for b, d in rows])
    sc.assert_close(got_l, np.stack(ref_lasts), wl.io, "last_state")
    assert torch.isfinite(out.float()).all()


def test_conv_full_size_sampled(oracle):
    """The Mamba-130M layer (8 x 1536 x 2048) with Conv1D(k=4) + SiLU fused in
    front of the scan, weights from the workload recipe."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = wk.MAMBA_LAYER_CONV
    inp = wk.make_inputs(wl, seed=0)
    t = sc.device_inputs(inp)
    out, last = ss.selective_scan_fwd(t["u"], t["delta"][:, 0], t["A"], t["B"][:, 0],
                                      t["C"][:, 0], t["D"], t["z"], t["delta_bias"], True,
                                      return_last_state=True, conv_w=sc.to_torch(inp.conv_w),
                                      conv_b=sc.to_torch(inp.conv_b))
    torch.cuda.synchronize()
    f = _f64(inp)
    cw, cb = inp.conv_w.astype(np.float64), inp.conv_b.astype(np.float64)
    rows = _rows(wl)
    refs, ref_lasts = [], []
    for b, d in rows:
        r = _row_inputs(f, wl, b, d)
        u = oracle.conv_silu(r["u"], cw[d:d + 1], cb[d:d + 1])
        o, l = oracle.scan(u, r["delta"], r["A"], r["B"], r["C"], r["D"], r["z"],
                           r["delta_bias"], True)
        refs.append(o[0, 0])
        ref_lasts.append(l[0, 0, 0])
    got = np.stack([sc.from_torch(out[b, d]) for b, d in rows])
    sc.assert_close(got, np.stack(refs), wl.io)
    got_l = np.stack([last[b, d].cpu().numpy() for b, d in rows])
    sc.assert_close(got_l, np.stack(ref_lasts), wl.io, "last_state")
    assert torch.isfinite(out.float()).all()


def test_dwconv_full_size_sampled(oracle):
    """DWConv 3x3 + SiLU on the VMamba-T stage-1 map, 32 x 192 x 56 x 56, bf16."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = wk.Workload("dwconv_full", 32, 192, 56 * 56, K=4, with_z=False, H=56, W=56, conv2d=True)
    inp = wk.make_inputs(wl, seed=0)
    x = sc.to_torch(inp.u).view(wl.batch, wl.dim, wl.H, wl.W)
    u = ss.dwconv3x3_silu(x, sc.to_torch(inp.conv2d_w), sc.to_torch(inp.conv2d_b))
    torch.cuda.synchronize()
    xf = inp.as_f64("u").reshape(wl.batch, wl.dim, wl.H, wl.W)
    w, cb = inp.conv2d_w.astype(np.float64), inp.conv2d_b.astype(np.float64)
    rows = _rows(wl, n=30)
    ref = np.stack([oracle.dwconv3x3_silu(xf[b:b + 1, d:d + 1], w[d:d + 1], cb[d:d + 1])[0, 0]
                    for b, d in rows])
    got = np.stack([sc.from_torch(u[b, d]) for b, d in rows])
    sc.assert_close(got, ref, wl.io)
    assert torch.isfinite(u.float()).all()


@pytest.mark.parametrize("wl", [wk.VMAMBA_SS2D, wk.LOCAL_WIN], ids=lambda w: w.name)
def test_multi_bwd_full_size_sampled(oracle, wl):
    """Backward pass of the four-direction map workloads (32 x 192 x 56 x 56, no
    gate): SS2D's row/column orders, and LocalMamba's 7 x 7 windowed orders.
    Against the oracle: du, ddelta, dB, dC of batch 0 (all 192 channels, so dB
    and dC are complete sums), and dA, dD, ddelta_bias of eight channels summed
    over all 32 batches."""
    import selective_state_space_120_b300 as ss
    inp = wk.make_inputs(wl, seed=0)
    dout = wk.make_dout(wl, seed=0)
    t = sc.device_inputs(inp)
    bsz, dim, H, W, K = wl.batch, wl.dim, wl.H, wl.W, wl.K
    orders = list(wl.orders) or [ss.DIR_ROW, ss.DIR_COL, ss.DIR_ROW_REV, ss.DIR_COL_REV]
    g = ss.multi_scan_bwd(t["u"].view(bsz, dim, H, W), t["delta"], t["A"], t["B"], t["C"],
                          sc.to_torch(dout).view(bsz, dim, H, W), orders, wl.win, t["D"],
                          t["delta_bias"], True)
    got = {k: (None if v is None else sc.from_torch(v)) for k, v in g.items()}
    got["du"] = got["du"].reshape(bsz, dim, wl.L)
    f = _f64(inp)
    dy = _dout_f64(wl, dout)
    ords = [_oracle_order(oracle, o) for o in orders]
    r0 = oracle.multi_scan_bwd(f["u"][:1], f["delta"][:1], f["A"], f["B"][:1], f["C"][:1], dy[:1],
                               ords, H=H, W=W, win=wl.win, D=f["D"], delta_bias=f["delta_bias"])
    sub = {k: got[k][:1] for k in ("du", "ddelta", "dB", "dC")}
    assert_grads(sub, r0, wl.io, names=("du", "ddelta", "dB", "dC"))
    ch = np.array([0, 1, 31, 32, 95, 128, 190, 191])
    sel = np.concatenate([k * dim + ch for k in range(K)])
    rc = oracle.multi_scan_bwd(f["u"][:, ch], f["delta"][:, :, ch], f["A"][sel], f["B"], f["C"],
                               dy[:, ch], ords, H=H, W=W, win=wl.win, D=f["D"][sel],
                               delta_bias=f["delta_bias"][sel])
    sums = {"dA": got["dA"][sel], "dD": got["dD"][sel], "ddelta_bias": got["ddelta_bias"][sel]}
    assert_grads(sums, rc, wl.io, names=("dA", "dD", "ddelta_bias"))


def test_decode_full_size_sampled(oracle):
    """Token-by-token decoding on the Mamba-130M layer shape (batch 8, dim 1536,
    N = 16, bf16), the launch configuration the benchmark times: eight steps
    from a random state against the oracle's eight-step scan from that state,
    on sampled channels (outputs and the final state)."""
    import torch
    import selective_state_space_120_b300 as ss
    wl = wk.scaled(wk.MAMBA_LAYER, "decode_full", L=8, last_state=True)
    inp = wk.make_inputs(wl, seed=0)
    h0 = np.random.default_rng(7).standard_normal((wl.batch, wl.dim, wl.N)).astype(np.float32)
    t = sc.device_inputs(inp)
    state = torch.from_numpy(h0).cuda()
    outs = []
    for k in range(wl.L):
        outs.append(ss.selective_state_update(
            t["u"][:, :, k].contiguous(), t["delta"][:, 0, :, k].contiguous(), t["A"],
            t["B"][:, 0, :, :, k].contiguous(), t["C"][:, 0, :, :, k].contiguous(), state, t["D"],
            t["z"][:, :, k].contiguous(), t["delta_bias"], True))
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=-1)
    f = _f64(inp)
    rows = _rows(wl, n=20)
    refs, ref_last = [], []
    for b, d in rows:
        r = _row_inputs(f, wl, b, d)
        o, l = oracle.scan(r["u"], r["delta"], r["A"], r["B"], r["C"], r["D"], r["z"],
                           r["delta_bias"], True, h0=h0[b:b + 1, None, d:d + 1].astype(np.float64))
        refs.append(o[0, 0])
        ref_last.append(l[0, 0, 0])
    sc.assert_close(np.stack([sc.from_torch(got[b, d]) for b, d in rows]), np.stack(refs), wl.io)
    sc.assert_close(np.stack([state[b, d].cpu().numpy() for b, d in rows]), np.stack(ref_last),
                    wl.io, "state")
