"""Seeded synthetic inputs for the selective scan (shared by tests and the benchmark).

This module only draws random numbers and rounds them; it holds none of the
scan's arithmetic.  Every array is produced on the host from one NumPy PCG64
stream, so the CUDA library and the float64 oracle see the same bits.

Recipe (the workloads of the Mamba / Vim / VMamba pages, with synthetic data):
    draw order: u, z, raw delta, dt0, then for each direction k: B_k, C_k
    u, z            ~ N(0, 1)                           [batch, dim, L]
    raw delta       ~ N(0, 1) * 0.1                     [batch, K, dim, L]
    dt0             = exp(U[ln 1e-3, ln 1e-1])          per (k, d)
    delta_bias      = log(expm1(dt0))  (the inverse of softplus, so that
                      softplus(0 + delta_bias) = dt0)   [K*dim]
    A[k, d, n]      = -(n + 1)                          [K*dim, N]
    B_k, C_k        ~ N(0, 1)                           [batch, K, G, N, L]
    D               = 1                                 [K*dim]
    conv workloads, drawn last: conv_w ~ N(0, 0.5^2) [dim, 4], conv_b ~ N(0, 0.1^2)
    conv2d workloads, drawn last: conv2d_w ~ N(0, 0.3^2) [dim, 3, 3], conv2d_b ~ N(0, 0.1^2)
    backward pass: the upstream gradient dout ~ N(0, 1) [batch, dim, L], from
                   its own PCG64 stream seeded with (seed, 1) (make_dout)
Inputs of a bf16 workload are rounded to bf16 (round-to-nearest-even) on the
host; A, D and delta_bias stay float32.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 24  # values drawn per call, to bound host memory on large workloads


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    dim: int
    L: int
    N: int = 16
    G: int = 1
    K: int = 1            # directions: 1 plain scan, 2 bidirectional, 4 SS2D
    io: str = "bf16"      # "bf16" or "f32"
    with_z: bool = True
    with_D: bool = True
    last_state: bool = False
    H: int = 1
    W: int = 0            # W = L for a plain sequence
    conv: bool = False    # u is the input of a fused Conv1D(k=4) + SiLU
    conv2d: bool = False  # u comes from the SS2D block's DWConv 3x3 + SiLU of an input map x
    orders: tuple = ()    # traversal codes (SS_DIR_*) of an any-order call; () = the kind's own
    win: int = 0          # window size of the windowed orders

    @property
    def elems(self) -> int:
        return self.batch * self.dim * self.L

    @property
    def kind(self) -> str:
        if self.orders:
            return "orders"
        return {1: "scan", 2: "bidir", 4: "ss2d"}[self.K]


# The five workloads, named by what they are.
TINY_F32 = Workload("tiny_s6_f32_b1_d16_l64_n16", 1, 16, 64, io="f32", last_state=True)
MAMBA_LAYER = Workload("mamba130m_layer_b8_d1536_l2048_n16", 8, 1536, 2048)
LONG_SEQ = Workload("long_seq_b1_d5120_l131072_n16", 1, 5120, 131072, last_state=True)
VIM_BIDIR = Workload("vim_s_bidir_b128_d768_l197_n16", 128, 768, 197, K=2)
VMAMBA_SS2D = Workload("vmamba_t_ss2d_b32_d192_56x56_n16", 32, 192, 56 * 56, K=4,
                       with_z=False, H=56, W=56)

ALL = (TINY_F32, MAMBA_LAYER, LONG_SEQ, VIM_BIDIR, VMAMBA_SS2D)

# LocalMamba-style windowed scan on the VMamba-T stage-1 map: four windowed
# directions (7 x 7 windows, row- and column-major, and their reverses; codes
# SS_DIR_WIN, SS_DIR_WIN_COL, SS_DIR_WIN_REV, SS_DIR_WIN_COL_REV), no gate.
LOCAL_WIN = Workload("localmamba_win7_b32_d192_56x56_n16", 32, 192, 56 * 56, K=4, with_z=False,
                     H=56, W=56, orders=(4, 5, 6, 7), win=7)

# The long sequence cut to L = 16384: the same 5120 rows and the same twelve
# L-chunks, with 1/8 of the data, for ncu captures of the chunked path (whose
# full size is beyond a multi-pass capture); not a benchmark line.
LONG_SEQ_PROFILE = Workload("long_seq_b1_d5120_l16384_n16", 1, 5120, 16384, last_state=True)

# The Mamba layer with its Conv1D(k=4) + SiLU input branch fused in front of the
# scan (weights ~ N(0, 0.5^2), bias ~ N(0, 0.1^2)).
MAMBA_LAYER_CONV = Workload("mamba130m_layer_conv_b8_d1536_l2048_n16", 8, 1536, 2048, conv=True)

# VMamba-T's third stage (the deepest): SS2D on a 14 x 14 map of 384 channels,
# whose 196-value rows are not 16-byte multiples in bf16 (views of two rows).
VMAMBA_SS2D_14 = Workload("vmamba_t_ss2d_b32_d384_14x14_n16", 32, 384, 14 * 14, K=4,
                          with_z=False, H=14, W=14)

# The Mamba layer one step shorter: rows of 2047 bf16 values are not 16-byte
# multiples (the scan reads them through views of eight rows to a view row).
MAMBA_LAYER_UNALIGNED = Workload("mamba130m_layer_b8_d1536_l2047_n16", 8, 1536, 2047)


def round_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit patterns (uint16), round-to-nearest-even; finite inputs."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    rounded = (bits + 0x7FFF + ((bits >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _normal(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """N(0,1)*scale as float32, drawn in fixed-size pieces (same stream as one call)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for i in range(0, n, _CHUNK):
        m = min(_CHUNK, n - i)
        v = rng.standard_normal(m)
        if scale != 1.0:
            v *= scale
        out[i:i + m] = v
    return out.reshape(shape)


@dataclass
class Inputs:
    """Host arrays of one workload.  Tensors in the I/O dtype are stored as
    float32 (f32 workloads) or as bf16 bit patterns in uint16 (bf16 workloads)."""
    wl: Workload
    u: np.ndarray
    delta: np.ndarray        # [batch, K, dim, L]
    A: np.ndarray            # [K*dim, N] float32
    B: np.ndarray            # [batch, K, G, N, L]
    C: np.ndarray
    D: np.ndarray | None     # [K*dim] float32
    z: np.ndarray | None
    delta_bias: np.ndarray   # [K*dim] float32
    extra: dict = field(default_factory=dict)
    conv_w: np.ndarray | None = None   # [dim, 4] float32 (conv workloads)
    conv_b: np.ndarray | None = None   # [dim] float32
    conv2d_w: np.ndarray | None = None  # [dim, 3, 3] float32 (conv2d workloads)
    conv2d_b: np.ndarray | None = None  # [dim] float32

    def as_f64(self, name: str) -> np.ndarray | None:
        """The exact values handed to the GPU, widened to float64."""
        a = getattr(self, name)
        if a is None:
            return None
        if a.dtype == np.uint16:
            return bf16_bits_to_f32(a).astype(np.float64)
        return a.astype(np.float64)


def make_inputs(wl: Workload, seed: int = 0) -> Inputs:
    rng = np.random.Generator(np.random.PCG64(seed))
    b, d, L, N, G, K = wl.batch, wl.dim, wl.L, wl.N, wl.G, wl.K
    u = _normal(rng, (b, d, L))
    z = _normal(rng, (b, d, L))
    raw = _normal(rng, (b, K, d, L), 0.1)
    dt0 = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), size=K * d))
    bias = np.log(np.expm1(dt0)).astype(np.float32)
    Bs, Cs = [], []
    for _ in range(K):
        Bs.append(_normal(rng, (b, G, N, L)))
        Cs.append(_normal(rng, (b, G, N, L)))
    Bm = np.stack(Bs, axis=1)
    Cm = np.stack(Cs, axis=1)
    A = np.tile(-(np.arange(N, dtype=np.float32) + 1.0), (K * d, 1))
    D = np.ones(K * d, dtype=np.float32) if wl.with_D else None
    if not wl.with_z:
        z = None
    if wl.io == "bf16":
        cv = round_bf16_bits
    else:
        cv = lambda x: np.ascontiguousarray(x, dtype=np.float32)  # noqa: E731
    inp = Inputs(wl, cv(u), cv(raw), A, cv(Bm), cv(Cm), D,
                 None if z is None else cv(z), bias)
    if wl.conv:
        # drawn after everything else, so the other inputs are those of the
        # same workload without the conv
        inp.conv_w = (rng.standard_normal((d, 4)) * 0.5).astype(np.float32)
        inp.conv_b = (rng.standard_normal(d) * 0.1).astype(np.float32)
    if wl.conv2d:
        # drawn after everything else as well; u is then the map the convolution reads
        inp.conv2d_w = (rng.standard_normal((d, 3, 3)) * 0.3).astype(np.float32)
        inp.conv2d_b = (rng.standard_normal(d) * 0.1).astype(np.float32)
    return inp


def make_dout(wl: Workload, seed: int = 0) -> np.ndarray:
    """Upstream gradient of the scan's output for the backward pass, in the
    workload's I/O representation (float32, or bf16 bits in uint16)."""
    rng = np.random.Generator(np.random.PCG64([seed, 1]))
    g = _normal(rng, (wl.batch, wl.dim, wl.L))
    return round_bf16_bits(g) if wl.io == "bf16" else g


def scaled(wl: Workload, name: str | None = None, **changes) -> Workload:
    """A copy of a workload with some fields changed (for small parity cases)."""
    fields = dict(wl.__dict__)
    fields.update(changes)
    fields["name"] = name or (wl.name + "_small")
    return Workload(**fields)
