"""The seeded input recipe shared by the library's tests and the oracle (CPU only)."""
import numpy as np
import torch

from selective_state_space_120_b300 import workloads as wk


def test_recipe_values_and_ranges():
    """u, z ~ N(0,1); raw Delta ~ 0.1 N(0,1); softplus(bias) = dt0 in [1e-3, 1e-1];
    A = -(n+1); D = 1; B, C ~ N(0,1); every I/O tensor rounded to bf16."""
    wl = wk.Workload("recipe", 4, 64, 512, K=2, G=2)
    inp = wk.make_inputs(wl, seed=0)
    assert inp.u.shape == (4, 64, 512) and inp.z.shape == (4, 64, 512)
    assert inp.delta.shape == (4, 2, 64, 512)
    assert inp.B.shape == inp.C.shape == (4, 2, 2, 16, 512)
    np.testing.assert_array_equal(inp.A, np.tile(-(np.arange(16) + 1.0), (2 * 64, 1)))
    np.testing.assert_array_equal(inp.D, np.ones(2 * 64))
    dt0 = np.log1p(np.exp(inp.delta_bias.astype(np.float64)))
    assert dt0.min() >= 1e-3 * (1 - 1e-5) and dt0.max() <= 1e-1 * (1 + 1e-5)
    for name, sd in (("u", 1.0), ("z", 1.0), ("delta", 0.1), ("B", 1.0), ("C", 1.0)):
        v = inp.as_f64(name)
        assert abs(v.mean()) < 0.02 * sd and abs(v.std() - sd) < 0.02 * sd, name
        assert getattr(inp, name).dtype == np.uint16, name   # bf16 bit patterns


def test_recipe_is_reproducible_and_seeded():
    wl = wk.Workload("seeded", 2, 8, 64)
    a, b, c = (wk.make_inputs(wl, seed=s) for s in (0, 0, 1))
    for name in ("u", "delta", "B", "C", "z", "delta_bias"):
        np.testing.assert_array_equal(getattr(a, name), getattr(b, name))
        assert not np.array_equal(getattr(a, name), getattr(c, name))


def test_chunked_draws_continue_one_stream(monkeypatch):
    """Large tensors are drawn in pieces; the pieces are one stream's draws."""
    monkeypatch.setattr(wk, "_CHUNK", 7)
    got = wk._normal(np.random.Generator(np.random.PCG64(3)), (5, 9), 0.5)
    want = (np.random.Generator(np.random.PCG64(3)).standard_normal(45) * 0.5).astype(np.float32)
    np.testing.assert_array_equal(got.ravel(), want)


def test_bf16_rounding_matches_torch():
    """Round-to-nearest-even to bf16, against torch's own conversion, including
    exact ties, values that carry into the exponent, and signed zeros."""
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.0e38, -2.5e-38],
                                 dtype=np.float32),
                        (np.arange(1 << 16, dtype=np.uint32) << 16 | 0x8000).view(np.float32)[:30000:7]])
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(wk.round_bf16_bits(x), want)
    np.testing.assert_array_equal(wk.bf16_bits_to_f32(want), torch.from_numpy(want.view(np.int16))
                                  .view(torch.bfloat16).float().numpy())
