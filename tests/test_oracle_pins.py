"""Pins for the float64 oracle (CPU only).

Each test checks the oracle against something other than itself: a worked
example evaluated by hand, a closed form, an independent formulation (the
semiseparable-matrix form, the LTI convolution), an explicit permutation with
NumPy, or an invariant of the recurrence.  Together they are chosen so that a
plausible slip in the oracle (a dropped term, a sign, an index, a swapped B/C,
a wrong direction order) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softplus(x):
    return np.logaddexp(0.0, x)


def _silu(z):
    return z / (1.0 + np.exp(-z))


def _rand_case(rng, batch=2, dim=3, L=17, N=4, G=1, K=1, with_z=True):
    u = rng.standard_normal((batch, dim, L))
    delta = rng.standard_normal((batch, K, dim, L)) * 0.5
    A = -np.exp(rng.standard_normal((K * dim, N)) * 0.5)
    B = rng.standard_normal((batch, K, G, N, L))
    C = rng.standard_normal((batch, K, G, N, L))
    D = rng.standard_normal(K * dim)
    z = rng.standard_normal((batch, dim, L)) if with_z else None
    bias = rng.standard_normal(K * dim) * 0.5 - 1.0
    return u, delta, A, B, C, D, z, bias


# ---------------------------------------------------------------- worked examples
def test_worked_example_by_hand(oracle):
    """Hand-evaluated recurrence (tests/golden/s6_n1_l4_worked.json)."""
    g = json.load(open(os.path.join(GOLDEN, "s6_n1_l4_worked.json")))
    inp = g["inputs"]
    L = inp["L"]
    u = np.array(inp["u"], float).reshape(1, 1, L)
    B = np.array(inp["B"], float).reshape(1, 1, 1, L)
    C = np.array(inp["C"], float).reshape(1, 1, 1, L)
    A = np.array([[inp["A"]]])
    D = np.array([inp["D"]])
    ln2 = math.log(2.0)
    for case in g["cases"]:
        dval = ln2 if case["delta"].startswith("ln2") else 0.0
        delta = np.full((1, 1, L), dval)
        out, last = oracle.selective_scan(u, delta, A, B, C, D, None,
                                          np.array([case["delta_bias"]]),
                                          case["delta_softplus"], zoh=case["zoh"])
        want = np.array(case["y_ln2_coeff"]) * ln2 + np.array(case["y_const"])
        np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-14, err_msg=case["name"])
        want_last = case["last_state_ln2_coeff"] * ln2 + case["last_state_const"]
        np.testing.assert_allclose(last[0, 0, 0], want_last, rtol=1e-14, err_msg=case["name"])


def test_ss2d_orders_by_hand(oracle):
    """Position maps of the four SS2D directions (tests/golden/ss2d_orders_2x3.json)."""
    g = json.load(open(os.path.join(GOLDEN, "ss2d_orders_2x3.json")))
    H, W = g["H"], g["W"]
    names = {"row": oracle.ORDER_FWD, "col": oracle.ORDER_COL,
             "row_rev": oracle.ORDER_REV, "col_rev": oracle.ORDER_COL_REV}
    for name, want in g["orders"].items():
        got = [oracle.position(names[name], s, H, W) for s in range(H * W)]
        assert got == want, name


# ---------------------------------------------------------------- closed forms
def test_n1_closed_form_time_varying(oracle):
    """N = 1: h_t = sum_{s<=t} exp(A * sum_{r=s+1..t} dt_r) dt_s B_s u_s (exp of a sum, O(L^2))."""
    rng = np.random.default_rng(1)
    L = 200
    u = rng.standard_normal((1, 1, L))
    raw = rng.standard_normal((1, 1, L))
    bias = np.array([-0.7])
    A = np.array([[-0.9]])
    B = rng.standard_normal((1, 1, 1, L))
    C = rng.standard_normal((1, 1, 1, L))
    D = np.array([0.3])
    z = rng.standard_normal((1, 1, L))
    out, last = oracle.selective_scan(u, raw, A, B, C, D, z, bias, True)

    dt = _softplus(raw[0, 0] + bias[0])
    S = np.cumsum(dt)
    h = np.zeros(L)
    for t in range(L):
        s = np.arange(t + 1)
        h[t] = np.sum(np.exp(A[0, 0] * (S[t] - S[s])) * dt[s] * B[0, 0, 0, s] * u[0, 0, s])
    y = (C[0, 0, 0] * h + D[0] * u[0, 0]) * _silu(z[0, 0])
    np.testing.assert_allclose(out[0, 0], y, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(last[0, 0, 0], h[-1], rtol=1e-11)


def test_geometric_series(oracle):
    """Constant abar, bbar, u = 1: h_t = bbar (1 - abar^(t+1)) / (1 - abar)."""
    L = 64
    dt, a = 0.37, -1.3
    u = np.ones((1, 1, L))
    delta = np.full((1, 1, L), dt)
    B = np.full((1, 1, 1, L), 0.8)
    C = np.ones((1, 1, 1, L))
    out, last = oracle.selective_scan(u, delta, np.array([[a]]), B, C, None, None, None, False)
    abar = math.exp(dt * a)
    bbar = dt * 0.8
    t = np.arange(L)
    want = bbar * (1 - abar ** (t + 1)) / (1 - abar)
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-13)
    # Zero-order hold: bbar = (abar - 1) / a * B
    out_z, _ = oracle.selective_scan(u, delta, np.array([[a]]), B, C, None, None, None, False,
                                     zoh=True)
    bz = (abar - 1.0) / a * 0.8
    np.testing.assert_allclose(out_z[0, 0], bz * (1 - abar ** (t + 1)) / (1 - abar), rtol=1e-13)


def test_semiseparable_matrix_form(oracle):
    """General N, groups, D, gate: y = M u with
    M[t, s] = sum_n C[t, n] exp(A_n (S_t - S_s)) dt_s B[s, n]  (s <= t),  S = cumsum(dt)."""
    rng = np.random.default_rng(2)
    batch, dim, L, N, G = 2, 4, 23, 5, 2
    u, delta, A, B, C, D, z, bias = _rand_case(rng, batch, dim, L, N, G)
    out, last = oracle.scan(u, delta, A, B, C, D, z, bias, True)
    dpg = dim // G
    for b in range(batch):
        for d in range(dim):
            g = d // dpg
            dt = _softplus(delta[b, 0, d] + bias[d])
            S = np.cumsum(dt)
            decay = np.exp(A[d][None, None, :] * (S[:, None, None] - S[None, :, None]))  # [t,s,n]
            M = np.einsum("tn,tsn,s,sn->ts", C[b, 0, g].T, decay, dt, B[b, 0, g].T)
            M = np.tril(M)
            y = M @ u[b, d] + D[d] * u[b, d]
            np.testing.assert_allclose(out[b, d], y * _silu(z[b, d]), rtol=1e-10, atol=1e-12)
            h_end = np.array([np.sum(np.exp(A[d, n] * (S[-1] - S)) * dt * B[b, 0, g, n] * u[b, d])
                              for n in range(N)])
            np.testing.assert_allclose(last[b, 0, d], h_end, rtol=1e-10, atol=1e-13)


def test_lti_equals_convolution(oracle):
    """Constant dt, B, C: the scan is the causal convolution y = K * u + D u,
    K_j = sum_n C_n abar_n^j dt B_n (the convolutional view of an LTI SSM)."""
    rng = np.random.default_rng(3)
    L, N = 150, 6
    dt = 0.21
    An = -np.linspace(0.2, 3.0, N)
    Bn = rng.standard_normal(N)
    Cn = rng.standard_normal(N)
    u = rng.standard_normal((1, 1, L))
    delta = np.full((1, 1, L), dt)
    B = np.broadcast_to(Bn[:, None], (N, L)).reshape(1, 1, N, L)
    C = np.broadcast_to(Cn[:, None], (N, L)).reshape(1, 1, N, L)
    out, _ = oracle.selective_scan(u, delta, An[None], B, C, np.array([0.4]), None, None, False)
    j = np.arange(L)
    Kj = np.sum(Cn[None] * np.exp(dt * An[None] * j[:, None]) * dt * Bn[None], axis=1)
    y = np.convolve(u[0, 0], Kj)[:L] + 0.4 * u[0, 0]
    np.testing.assert_allclose(out[0, 0], y, rtol=1e-10, atol=1e-12)


def test_softplus_matches_library(oracle):
    xs = np.concatenate([np.linspace(-50, 50, 401), [-745.0, -30.0, 0.0, 1e-9, 30.0, 700.0]])
    got = np.array([oracle.softplus(x) for x in xs])
    np.testing.assert_allclose(got, np.logaddexp(0.0, xs), rtol=1e-15, atol=1e-300)


# ---------------------------------------------------------------- directions
def test_reverse_is_flipped_forward(oracle):
    """A reversed direction reads u (and writes out) from the last position back
    to the first, with its Delta, B, C already in its own scan order: it equals
    a forward scan of the flipped u (and z) with the same Delta, B, C, flipped
    back."""
    rng = np.random.default_rng(4)
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 2, 3, 31, 4, 1)
    out_r, last_r = oracle.scan(u, delta, A, B, C, D, z, bias, True, (oracle.ORDER_REV,))
    fl = lambda a: np.ascontiguousarray(a[..., ::-1])  # noqa: E731
    out_f, last_f = oracle.scan(fl(u), delta, A, B, C, D, fl(z), bias, True,
                                (oracle.ORDER_FWD,))
    np.testing.assert_allclose(out_r, fl(out_f), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(last_r, last_f, rtol=1e-13)


def test_bidirectional_is_sum_of_two_scans(oracle):
    rng = np.random.default_rng(5)
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 2, 3, 19, 4, 1, K=2)
    out, last = oracle.bidir_scan(u, delta, A, B, C, D, z, bias, True)
    f0, l0 = oracle.scan(u, delta[:, :1], A[:3], B[:, :1], C[:, :1], D[:3], None, bias[:3], True,
                         (oracle.ORDER_FWD,))
    f1, l1 = oracle.scan(u, delta[:, 1:], A[3:], B[:, 1:], C[:, 1:], D[3:], None, bias[3:], True,
                         (oracle.ORDER_REV,))
    np.testing.assert_allclose(out, (f0 + f1) * _silu(z), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(last[:, 0], l0[:, 0], rtol=1e-13)
    np.testing.assert_allclose(last[:, 1], l1[:, 0], rtol=1e-13)


@pytest.mark.parametrize("H,W", [(3, 5), (5, 3), (1, 1), (4, 4), (2, 7)])
def test_ss2d_equals_four_permuted_scans(oracle, H, W):
    """SS2D = four independent 1-D forward scans of explicitly permuted copies of
    the map (row-major, transposed, and both flipped), each with its own Delta,
    B, C in its scan order, mapped back and summed."""
    rng = np.random.default_rng(6 + H * 10 + W)
    batch, dim, N, G = 2, 3, 4, 1
    L = H * W
    u, delta, A, B, C, D, z, bias = _rand_case(rng, batch, dim, L, N, G, K=4)
    out, last = oracle.scan(u, delta, A, B, C, D, z, bias, True, oracle.SS2D_ORDERS, H=H, W=W)

    def to_seq(x, k):          # [..., L] in position order -> scan order of direction k
        m = x.reshape(x.shape[:-1] + (H, W))
        if k in (1, 3):
            m = np.swapaxes(m, -1, -2)
        s = m.reshape(x.shape[:-1] + (L,))
        return np.ascontiguousarray(s[..., ::-1] if k in (2, 3) else s)

    def from_seq(s, k):        # inverse of to_seq
        if k in (2, 3):
            s = s[..., ::-1]
        if k in (1, 3):
            m = s.reshape(s.shape[:-1] + (W, H))
            return np.ascontiguousarray(np.swapaxes(m, -1, -2).reshape(s.shape[:-1] + (L,)))
        return np.ascontiguousarray(s)

    total = np.zeros((batch, dim, L))
    for k in range(4):
        yk, lk = oracle.scan(to_seq(u, k), delta[:, k:k + 1], A[k * dim:(k + 1) * dim],
                             B[:, k:k + 1], C[:, k:k + 1],
                             D[k * dim:(k + 1) * dim], None, bias[k * dim:(k + 1) * dim], True,
                             (oracle.ORDER_FWD,))
        total += from_seq(yk, k)
        np.testing.assert_allclose(last[:, k], lk[:, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(out, total * _silu(z), rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------- limiting cases
def test_delta_to_zero(oracle):
    rng = np.random.default_rng(7)
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 2, 3, 20, 4, 1)
    # softplus off, delta = 0, bias = 0: no input reaches the state.
    out, last = oracle.scan(u, np.zeros_like(delta), A, B, C, D, z, np.zeros_like(bias), False)
    want = D[None, :, None] * u * _silu(z)
    # exact up to the last ulp of exp(): NumPy's exp and libm's may differ by one ulp
    np.testing.assert_allclose(out, want, rtol=4e-16, atol=0)
    np.testing.assert_array_equal(last, np.zeros_like(last))
    # softplus on with a very negative bias: dt ~ 4e-18.
    out2, last2 = oracle.scan(u, np.zeros_like(delta), A, B, C, D, z, np.full_like(bias, -40.0),
                              True)
    np.testing.assert_allclose(out2, want, rtol=0, atol=1e-15)
    assert np.max(np.abs(last2)) < 1e-15


def test_delta_large_is_memoryless(oracle):
    """dt*A below -745: abar is exactly 0 in double, so y_t = dt_t (C_t . B_t) u_t + D u_t."""
    rng = np.random.default_rng(8)
    batch, dim, L, N = 1, 2, 25, 3
    u, _, _, B, C, D, _, _ = _rand_case(rng, batch, dim, L, N, 1)
    dt = rng.uniform(800, 900, size=(batch, 1, dim, L))
    A = -np.ones((dim, N))
    out, last = oracle.scan(u, dt, A, B, C, D, None, None, False)
    cb = np.einsum("nl,nl->l", C[0, 0, 0], B[0, 0, 0])
    want = dt[0, 0] * cb[None] * u[0] + D[:, None] * u[0]
    np.testing.assert_allclose(out[0], want, rtol=1e-13)
    np.testing.assert_allclose(last[0, 0], dt[0, 0, :, -1:] * B[0, 0, 0, :, -1][None] * u[0, :, -1:],
                               rtol=1e-13)


# ---------------------------------------------------------------- invariants
def test_causality(oracle):
    rng = np.random.default_rng(9)
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 1, 2, 40, 4, 1)
    out, _ = oracle.scan(u, delta, A, B, C, D, z, bias, True)
    t0 = 23
    for arr_name in ("u", "delta", "B", "C"):
        args = dict(u=u.copy(), delta=delta.copy(), B=B.copy(), C=C.copy())
        args[arr_name][..., t0] += 1.7
        out2, _ = oracle.scan(args["u"], args["delta"], A, args["B"], args["C"], D, z, bias, True)
        np.testing.assert_array_equal(out2[..., :t0], out[..., :t0])
        assert np.all(out2[..., t0] != out[..., t0]) or arr_name == "C"


def test_linearity_in_u(oracle):
    rng = np.random.default_rng(10)
    u, delta, A, B, C, D, _, bias = _rand_case(rng, 1, 3, 30, 4, 1, with_z=False)
    u2 = rng.standard_normal(u.shape)
    o1, _ = oracle.scan(u, delta, A, B, C, D, None, bias, True)
    o2, _ = oracle.scan(u2, delta, A, B, C, D, None, bias, True)
    o3, _ = oracle.scan(2.5 * u - 0.5 * u2, delta, A, B, C, D, None, bias, True)
    np.testing.assert_allclose(o3, 2.5 * o1 - 0.5 * o2, rtol=1e-11, atol=1e-12)


def test_channel_and_batch_independence(oracle):
    rng = np.random.default_rng(11)
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 3, 4, 15, 4, 2)
    out, last = oracle.scan(u, delta, A, B, C, D, z, bias, True)
    b, d = 2, 3
    g = d // 2
    o1, l1 = oracle.scan(u[b:b + 1, d:d + 1], delta[b:b + 1, :, d:d + 1], A[d:d + 1],
                         B[b:b + 1, :, g:g + 1], C[b:b + 1, :, g:g + 1], D[d:d + 1],
                         z[b:b + 1, d:d + 1], bias[d:d + 1], True)
    np.testing.assert_array_equal(o1[0, 0], out[b, d])
    np.testing.assert_array_equal(l1[0, 0, 0], last[b, 0, d])


def test_split_invariance(oracle):
    """Scanning the first half, then the second half from the carried state,
    equals one scan over the whole sequence."""
    rng = np.random.default_rng(12)
    L, cut = 41, 17
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 2, 3, L, 4, 1)
    full, last = oracle.scan(u, delta, A, B, C, D, z, bias, True)
    a, la = oracle.scan(u[..., :cut], delta[..., :cut], A, B[..., :cut], C[..., :cut], D,
                        z[..., :cut], bias, True)
    b, lb = oracle.scan(u[..., cut:], delta[..., cut:], A, B[..., cut:], C[..., cut:], D,
                        z[..., cut:], bias, True, h0=la)
    np.testing.assert_allclose(np.concatenate([a, b], axis=-1), full, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lb, last, rtol=1e-13)


def test_chunk_carry_rule(oracle):
    """The rule the chunked long-sequence path chains its L-chunks by: a chunk
    scanned from a state h0 ends in exp(A * sum of Delta') * h0 plus the end
    state of the same chunk scanned from zero, and each of its outputs exceeds
    the zero-state one by C_t . (exp(A * S_t) * h0), gated, S_t being the sum
    of Delta' up to and including step t.  Delta' is computed here with NumPy's
    softplus, not the oracle's."""
    rng = np.random.default_rng(21)
    batch, dim, L, N = 2, 3, 23, 4
    u, delta, A, B, C, D, z, bias = _rand_case(rng, batch, dim, L, N, 1)
    delta, B, C = delta[:, 0], B[:, 0], C[:, 0]
    h0 = rng.standard_normal((batch, dim, N))
    y0, l0 = oracle.scan(u, delta, A, B, C, D, z, bias, True)
    y1, l1 = oracle.scan(u, delta, A, B, C, D, z, bias, True, h0=h0)
    dp = _softplus(delta + bias[None, :, None])      # [batch, dim, L]
    S = np.cumsum(dp, axis=-1)
    decay = np.exp(A[None, :, :, None] * S[:, :, None, :])   # [batch, dim, N, L]
    np.testing.assert_allclose(l1[:, 0], decay[..., -1] * h0 + l0[:, 0], rtol=1e-12, atol=1e-13)
    extra = np.einsum("bnl,bdnl,bdn->bdl", C[:, 0], decay, h0) * _silu(z)
    np.testing.assert_allclose(y1 - y0, extra, rtol=1e-10, atol=1e-12)


def test_group_mapping_contiguous_blocks(oracle):
    """Channel d uses group d // (dim / G): changing group 1's B/C leaves channels 0..dim/G-1 alone."""
    rng = np.random.default_rng(13)
    u, delta, A, B, C, D, z, bias = _rand_case(rng, 1, 4, 12, 3, 2)
    out, _ = oracle.scan(u, delta, A, B, C, D, z, bias, True)
    B2 = B.copy()
    B2[:, :, 1] += 1.0
    out2, _ = oracle.scan(u, delta, A, B2, C, D, z, bias, True)
    np.testing.assert_array_equal(out2[:, :2], out[:, :2])
    assert np.all(out2[:, 2:] != out[:, 2:])


# ---------------------------------------------------------------- Conv1D -> SiLU (Mamba block input branch)
def test_conv_silu_identity_kernel_is_silu(oracle):
    """Kernel [0, 0, 0, 1] with no bias passes x through: u = SiLU(x)."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal((2, 3, 17))
    w = np.tile([0.0, 0.0, 0.0, 1.0], (3, 1))
    np.testing.assert_allclose(oracle.conv_silu(x, w), _silu(x), rtol=1e-15, atol=0)


def test_conv_silu_equals_numpy_correlation(oracle):
    """Causal width-4 convolution against np.convolve of the zero-padded row."""
    rng = np.random.default_rng(22)
    batch, dim, L = 2, 3, 29
    x = rng.standard_normal((batch, dim, L))
    w = rng.standard_normal((dim, 4))
    bias = rng.standard_normal(dim)
    got = oracle.conv_silu(x, w, bias)
    for b in range(batch):
        for d in range(dim):
            padded = np.concatenate([np.zeros(3), x[b, d]])
            # out[t] = sum_j w[j] x[t - 3 + j]: a 'valid' correlation, i.e. a
            # convolution with the flipped kernel
            v = np.convolve(padded, w[d][::-1], mode="valid") + bias[d]
            np.testing.assert_allclose(got[b, d], _silu(v), rtol=1e-13, atol=1e-15)


def test_conv_silu_continues_across_a_split(oracle):
    """x0 = the last three inputs of the first part continues the convolution."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((1, 2, 40))
    w = rng.standard_normal((2, 4))
    bias = rng.standard_normal(2)
    full = oracle.conv_silu(x, w, bias)
    second = oracle.conv_silu(x[..., 25:], w, bias, x0=x[..., 22:25])
    np.testing.assert_allclose(second, full[..., 25:], rtol=1e-14, atol=1e-15)
    # and it is causal: changing a later input leaves earlier outputs alone
    x2 = x.copy()
    x2[..., 30] += 1.0
    np.testing.assert_array_equal(oracle.conv_silu(x2, w, bias)[..., :30], full[..., :30])


# ---------------------------------------------------------------- backward pass
def _fd_case(seed, softplus=True, with_z=True, G=2):
    rng = np.random.default_rng(seed)
    batch, dim, L, N = 2, 4, 6, 3
    u = rng.standard_normal((batch, dim, L))
    delta = rng.standard_normal((batch, dim, L)) * 0.5
    A = -np.exp(rng.standard_normal((dim, N)) * 0.5)
    B = rng.standard_normal((batch, G, N, L))
    C = rng.standard_normal((batch, G, N, L))
    D = rng.standard_normal(dim)
    z = rng.standard_normal((batch, dim, L)) if with_z else None
    bias = rng.standard_normal(dim) * 0.5 - 0.5
    dy = rng.standard_normal((batch, dim, L))
    return dict(u=u, delta=delta, A=A, B=B, C=C, D=D, z=z, delta_bias=bias), dy, softplus


@pytest.mark.parametrize("seed,softplus,with_z,G,zoh,with_h0",
                         [(41, True, True, 2, False, False), (42, False, False, 1, False, False),
                          (43, True, True, 1, True, False), (44, True, False, 2, False, True),
                          (45, False, True, 1, True, True)])
def test_backward_matches_finite_differences(oracle, seed, softplus, with_z, G, zoh, with_h0):
    """Every gradient of the oracle's backward pass against central finite
    differences of its forward scan, for the loss sum(dy * out): the Euler and
    the zero-order-hold input matrix, a zero or a given initial state (whose
    gradient is checked too)."""
    args, dy, sp = _fd_case(seed, softplus, with_z, G)
    batch, dim, _ = args["u"].shape
    N = args["A"].shape[1]
    args["h0"] = (np.random.default_rng(seed + 100).standard_normal((batch, dim, N))
                  if with_h0 else None)

    def loss(a):
        h0 = None if a["h0"] is None else a["h0"][:, None]
        out, _ = oracle.selective_scan(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                       a["delta_bias"], sp, zoh=zoh, h0=h0)
        return float(np.sum(dy * out))

    grads = oracle.selective_scan_bwd(args["u"], args["delta"], args["A"], args["B"], args["C"], dy,
                                      args["D"], args["z"], args["delta_bias"], sp, zoh=zoh,
                                      h0=args["h0"])
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}
    eps = 1e-6
    for name, gname in names.items():
        if args[name] is None:
            assert grads[gname] is None
            continue
        x = args[name]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            lp = loss(args)
            x[idx] = keep - eps
            lm = loss(args)
            x[idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grads[gname], fd, rtol=2e-6, atol=2e-7, err_msg=name)


@pytest.mark.parametrize("with_bias,with_x0", [(True, True), (False, False)])
def test_conv_backward_matches_finite_differences(oracle, with_bias, with_x0):
    """Every gradient of the Conv1D + SiLU backward pass against central finite
    differences of its forward, for the loss sum(du * u), with and without the
    bias and the inputs before the sequence."""
    rng = np.random.default_rng(46)
    batch, dim, L, KW = 2, 3, 7, 4
    a = {"x": rng.standard_normal((batch, dim, L)), "w": rng.standard_normal((dim, KW)) * 0.5,
         "bias": rng.standard_normal(dim) * 0.3 if with_bias else None,
         "x0": rng.standard_normal((batch, dim, KW - 1)) if with_x0 else None}
    du = rng.standard_normal((batch, dim, L))

    def loss(a):
        return float(np.sum(du * oracle.conv_silu(a["x"], a["w"], a["bias"], a["x0"])))

    g = oracle.conv_silu_bwd(a["x"], a["w"], du, a["bias"], a["x0"])
    eps = 1e-6
    for name, gname in (("x", "dx"), ("w", "dw"), ("bias", "dbias"), ("x0", "dx0")):
        if a[name] is None:
            assert g[gname] is None
            continue
        x = a[name]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            lp = loss(a)
            x[idx] = keep - eps
            lm = loss(a)
            x[idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g[gname], fd, rtol=2e-6, atol=2e-7, err_msg=name)


def test_backward_single_step_closed_form(oracle):
    """N = 1, L = 1, no gate, no softplus: y = C dt B u + D u, so dy/du = C dt B + D,
    dy/ddelta = C B u, dy/dB = C dt u, dy/dC = dt B u, dy/dD = u, and dA = 0
    (the state starts at zero)."""
    u, dt, B, C, D, A = 0.7, 0.3, -1.2, 0.5, 0.25, -2.0
    g = oracle.selective_scan_bwd(np.full((1, 1, 1), u), np.full((1, 1, 1), dt), np.full((1, 1), A),
                                  np.full((1, 1, 1, 1), B), np.full((1, 1, 1, 1), C),
                                  np.ones((1, 1, 1)), np.array([D]), None, None, False)
    np.testing.assert_allclose(g["du"].ravel(), [C * dt * B + D], rtol=1e-15)
    np.testing.assert_allclose(g["ddelta"].ravel(), [C * B * u], rtol=1e-15)
    np.testing.assert_allclose(g["dB"].ravel(), [C * dt * u], rtol=1e-15)
    np.testing.assert_allclose(g["dC"].ravel(), [dt * B * u], rtol=1e-15)
    np.testing.assert_allclose(g["dD"].ravel(), [u], rtol=1e-15)
    np.testing.assert_array_equal(g["dA"], np.zeros((1, 1)))


# ---------------------------------------------------------------- windowed orders
def test_window_orders_golden(oracle):
    """Windowed orders written out by hand (tests/golden/window_orders.json),
    with a divisible and a cut-short case; the reversed orders are their flips."""
    g = json.load(open(os.path.join(GOLDEN, "window_orders.json")))
    for case in g["cases"]:
        H, W, w = case["H"], case["W"], case["w"]
        for name, order, rev in (("win", oracle.ORDER_WIN, oracle.ORDER_WIN_REV),
                                 ("win_col", oracle.ORDER_WIN_COL, oracle.ORDER_WIN_COL_REV)):
            assert oracle.order_table(order, H, W, w).tolist() == case[name], (H, W, name)
            assert oracle.order_table(rev, H, W, w).tolist() == case[name][::-1], (H, W, name)


@pytest.mark.parametrize("H,W,w", [(4, 6, 2), (14, 14, 7), (8, 12, 4), (6, 6, 3)])
def test_window_orders_equal_numpy_reshape(oracle, H, W, w):
    """When w divides H and W, the windowed order is the map reshaped to
    (H/w, w, W/w, w) with the window axes outermost: (0, 2, 1, 3) for windows
    row-major, (2, 0, 3, 1) for windows and cells column-major."""
    idx = np.arange(H * W).reshape(H // w, w, W // w, w)
    assert np.array_equal(oracle.order_table(oracle.ORDER_WIN, H, W, w),
                          idx.transpose(0, 2, 1, 3).reshape(-1))
    assert np.array_equal(oracle.order_table(oracle.ORDER_WIN_COL, H, W, w),
                          idx.transpose(2, 0, 3, 1).reshape(-1))


@pytest.mark.parametrize("H,W", [(5, 7), (1, 9), (9, 1), (3, 3)])
def test_window_orders_limits(oracle, H, W):
    """w = 1 and w >= max(H, W) leave one cell or one window: row-major and
    column-major traversals; every windowed order is a permutation."""
    row = [oracle.position(oracle.ORDER_FWD, s, H, W) for s in range(H * W)]
    col = [oracle.position(oracle.ORDER_COL, s, H, W) for s in range(H * W)]
    for w in (1, max(H, W), max(H, W) + 3):
        assert oracle.order_table(oracle.ORDER_WIN, H, W, w).tolist() == row
        assert oracle.order_table(oracle.ORDER_WIN_COL, H, W, w).tolist() == col
    for order in (oracle.ORDER_WIN, oracle.ORDER_WIN_REV, oracle.ORDER_WIN_COL,
                  oracle.ORDER_WIN_COL_REV):
        assert sorted(oracle.order_table(order, H, W, 2).tolist()) == list(range(H * W))


@pytest.mark.parametrize("H,W,w", [(6, 8, 2), (5, 7, 3)])
def test_windowed_scan_equals_scan_of_permuted_copy(oracle, H, W, w):
    """A windowed direction equals a 1-D scan of the map's values taken in the
    window order (NumPy fancy indexing), with the outputs put back in place."""
    rng = np.random.default_rng(41)
    batch, dim, N, L = 2, 3, 4, H * W
    u = rng.standard_normal((batch, dim, L))
    z = rng.standard_normal((batch, dim, L))
    dl = rng.standard_normal((batch, dim, L)) * 0.3
    A = -rng.uniform(0.5, 2.0, (dim, N))
    B = rng.standard_normal((batch, 1, N, L))
    C = rng.standard_normal((batch, 1, N, L))
    D = rng.standard_normal(dim)
    bias = rng.standard_normal(dim) * 0.1
    for order in (oracle.ORDER_WIN, oracle.ORDER_WIN_REV, oracle.ORDER_WIN_COL,
                  oracle.ORDER_WIN_COL_REV):
        pos = oracle.order_table(order, H, W, w)
        got, got_last = oracle.scan(u, dl, A, B, C, D, z, bias, True, (order,), H=H, W=W, win=w)
        y, last = oracle.scan(u[..., pos], dl, A, B, C, D, None, bias, True)
        want = np.empty_like(y)
        want[..., pos] = y
        want *= z / (1.0 + np.exp(-z))
        np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(got_last, last, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- DWConv 3x3 + SiLU (SS2D input branch)
def test_dwconv_identity_kernel_is_silu(oracle):
    """Centre tap 1, no bias: u = SiLU(x)."""
    rng = np.random.default_rng(51)
    x = rng.standard_normal((2, 3, 5, 7))
    w = np.zeros((3, 3, 3))
    w[:, 1, 1] = 1.0
    np.testing.assert_allclose(oracle.dwconv3x3_silu(x, w), _silu(x), rtol=1e-15, atol=0)


def test_dwconv_equals_scipy_correlate2d(oracle):
    """Every channel against scipy.signal.correlate2d(mode='same') with zero fill."""
    from scipy.signal import correlate2d
    rng = np.random.default_rng(52)
    batch, dim, H, W = 2, 3, 6, 9
    x = rng.standard_normal((batch, dim, H, W))
    w = rng.standard_normal((dim, 3, 3))
    bias = rng.standard_normal(dim)
    got = oracle.dwconv3x3_silu(x, w, bias)
    for b in range(batch):
        for d in range(dim):
            v = correlate2d(x[b, d], w[d], mode="same", boundary="fill", fillvalue=0.0) + bias[d]
            np.testing.assert_allclose(got[b, d], _silu(v), rtol=1e-13, atol=1e-14)


def test_dwconv_separable_kernel(oracle):
    """A kernel outer(a, c) is a 3-tap correlation along the columns with c, then
    along the rows with a (np.convolve of the reversed taps, zero padded)."""
    rng = np.random.default_rng(53)
    x = rng.standard_normal((1, 1, 5, 8))
    a, c = rng.standard_normal(3), rng.standard_normal(3)
    got = oracle.dwconv3x3_silu(x, np.outer(a, c)[None])
    rows = np.stack([np.convolve(row, c[::-1], mode="same") for row in x[0, 0]])
    both = np.stack([np.convolve(col, a[::-1], mode="same") for col in rows.T]).T
    np.testing.assert_allclose(got[0, 0], _silu(both), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("orders_name,H,W,win", [("bidir", 1, 7, 0), ("ss2d", 3, 4, 0),
                                                 ("windowed", 4, 5, 2)])
def test_multi_direction_backward_matches_finite_differences(oracle, orders_name, H, W, win):
    """Every gradient of the multi-direction backward pass against central finite
    differences of the multi-direction forward scan (loss sum(dy * out)): Vim's
    two directions, SS2D's four, and four windowed ones on a cut-short map."""
    orders = {"bidir": (oracle.ORDER_FWD, oracle.ORDER_REV), "ss2d": oracle.SS2D_ORDERS,
              "windowed": (oracle.ORDER_WIN, oracle.ORDER_WIN_REV, oracle.ORDER_WIN_COL,
                           oracle.ORDER_WIN_COL_REV)}[orders_name]
    K, L = len(orders), H * W
    rng = np.random.default_rng(61 + K)
    batch, dim, N, G = 1, 2, 2, 1
    args = dict(u=rng.standard_normal((batch, dim, L)),
                delta=rng.standard_normal((batch, K, dim, L)) * 0.5,
                A=-np.exp(rng.standard_normal((K * dim, N)) * 0.5),
                B=rng.standard_normal((batch, K, G, N, L)),
                C=rng.standard_normal((batch, K, G, N, L)),
                D=rng.standard_normal(K * dim),
                z=rng.standard_normal((batch, dim, L)),
                delta_bias=rng.standard_normal(K * dim) * 0.5 - 0.5)
    dy = rng.standard_normal((batch, dim, L))

    def loss(a):
        out, _ = oracle.scan(a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                             a["delta_bias"], True, orders, H=H, W=W, win=win)
        return float(np.sum(dy * out))

    grads = oracle.multi_scan_bwd(args["u"], args["delta"], args["A"], args["B"], args["C"], dy,
                                  orders, H=H, W=W, win=win, D=args["D"], z=args["z"],
                                  delta_bias=args["delta_bias"])
    names = {"u": "du", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
             "z": "dz", "delta_bias": "ddelta_bias"}
    eps = 1e-6
    for name, gname in names.items():
        x = args[name]
        fd = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            keep = x[idx]
            x[idx] = keep + eps
            lp = loss(args)
            x[idx] = keep - eps
            lm = loss(args)
            x[idx] = keep
            fd[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grads[gname], fd, rtol=2e-6, atol=2e-7, err_msg=name)
