"""Host logic of the chunked long-sequence path: the split of a sequence into
L-chunks (csrc/ss_chunks.h), compiled with the host C++ compiler and checked
against the properties the two passes rely on (CPU only)."""
import math
import os
import shutil
import subprocess

import pytest

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "selective_state_space_120_b300", "csrc")

DRIVER = r"""
#include <cstdio>
#include "ss_chunks.h"
int main() {
    long long L, R, S;
    int J, T;
    while (std::scanf("%lld %d %lld %lld %d", &L, &J, &R, &S, &T) == 5) {
        const ssi::ChunkGeom g = ssi::chunk_geom(L, J, R, S, T);
        std::printf("%d %lld %lld\n", g.J, (long long)g.L0, (long long)g.Lm);
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def geom(tmp_path_factory):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    d = tmp_path_factory.mktemp("geom")
    src = d / "geom.cpp"
    src.write_text(DRIVER)
    exe = d / "geom"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)

    def run(cases):
        text = "".join(f"{L} {J} {R} {S} {T}\n" for (L, J, R, S, T) in cases)
        out = subprocess.run([str(exe)], input=text, capture_output=True, text=True, check=True)
        return [tuple(int(x) for x in line.split()) for line in out.stdout.splitlines()]

    return run


def _chunks(L, g):
    """(start, end) of every L-chunk of a geometry (J, L0, Lm)."""
    J, L0, Lm = g
    if J == 1:
        return [(0, L)]
    starts = [0, L0] + [L0 + j * Lm for j in range(1, J - 1)]
    return [(starts[j], starts[j + 1] if j + 1 < J else L) for j in range(J)]


CASES = [(L, J, R, S, T)
         for L in (1, 31, 32, 33, 200, 1200, 2047, 4096, 16384, 131072, 131071, 1 << 20)
         for J in (1, 2, 3, 5, 12, 19, 64)
         for (R, S) in ((2, 592), (16, 592), (160, 592), (300, 592), (384, 444), (160, 740))
         for T in (16, 32)]


def test_chunks_tile_the_sequence(geom):
    """Every split covers [0, L) with J <= the request non-empty chunks, each
    starting on a multiple of the step tile T (the copies' 16-byte rule)."""
    for c, g in zip(CASES, geom(CASES)):
        L, J, R, S, T = c
        assert 1 <= g[0] <= max(1, J), (c, g)
        ch = _chunks(L, g)
        assert ch[0][0] == 0 and ch[-1][1] == L, (c, g)
        for (a, b), (a2, _) in zip(ch, ch[1:]):
            assert b == a2, (c, g)
        for a, b in ch:
            assert b > a and a % T == 0, (c, g)


def test_equal_split_when_one_chunk_fills_half_the_gpu(geom):
    """R CTAs a chunk filling more than half of the S slots, or two chunks:
    equal chunks of ceil(L / J) steps rounded up to T, the last one shorter."""
    cases = [c for c in CASES if c[1] >= 2 and (2 * c[2] > c[3] or c[1] == 2)]
    for c, g in zip(cases, geom(cases)):
        L, J, R, S, T = c
        lc = (math.ceil(L / J) + T - 1) // T * T
        if lc >= L:
            assert g == (1, L, L), (c, g)
            continue
        assert g == (math.ceil(L / lc), lc, lc), (c, g)


def test_long_edge_chunks_balance_both_passes(geom):
    """With a quarter of the slots per chunk (the 1 x 5120 x 131072 scan: 160
    CTAs a chunk on 592 slots), the last chunk is about (J-2)*R/(S-R) middle
    chunks long and the first about 0.67 of that, so each pass's long chunk
    lasts as long as the other slots take over the middle chunks."""
    g = geom([(131072, 19, 160, 592, 32)])[0]
    assert g == (19, 20096, 4768)
    J, L0, Lm = g
    last = 131072 - L0 - (J - 2) * Lm
    want_last = (J - 2) * 160 / (592 - 160)
    assert abs(last / Lm - want_last) < 0.1
    assert abs(L0 / last - 0.67) < 0.02
    # pass 1: the first chunk (with outputs) against the middle chunks without
    # readout (0.67 of the cost) spread over the free slots; pass 2 likewise
    pass1_mid = (J - 2) * 160 * Lm * 0.67 / (592 - 160)
    pass2_mid = (J - 2) * 160 * Lm / (592 - 160)
    assert abs(L0 / pass1_mid - 1) < 0.02 and abs(last / pass2_mid - 1) < 0.02
