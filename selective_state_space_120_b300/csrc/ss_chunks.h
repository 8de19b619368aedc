// L-chunk geometry of the chunked single-direction path (host code only, so
// that it can be compiled and checked without the CUDA toolchain).
#pragma once

#include <algorithm>
#include <cmath>
#include <cstdint>

namespace ssi {

// Steps of the L-chunks of the chunked single-direction path: chunk 0 covers
// [0, L0), chunks 1..J-2 Lm steps each after it, chunk J-1 the rest up to L.
struct ChunkGeom {
    int J;
    int64_t L0, Lm;
};

// Cost of a chunk of the chunk-local pass (no readout, no C tiles, no gate)
// relative to a chunk that writes outputs: 284.6 us for one chunk with outputs
// and ten without against 408.7 us for eleven with, on 5120 rows of 16384 steps.
inline constexpr double kMidNoReadoutCost = 0.67;

// L-chunk geometry of the chunked path for a request of J chunks of R CTAs
// each on a GPU of S CTA slots.  Chunk 0 has no pass-2 rescan and chunk J-1
// no pass-1 scan, so making them longer than the middle chunks removes
// rescanned steps -- as long as each pass still keeps every slot busy: its
// long chunk's R CTAs run the whole pass while the other S - R slots work
// through the R*(J-2) middle CTAs.  Balancing the two gives the last chunk
// (J-2)*R/(S-R) middle lengths, and the first chunk that times the relative
// cost of a middle chunk in pass 1 (no readout: about two thirds of one with
// it, measured on the B300).  Every chunk starts on a multiple of T.
inline ChunkGeom chunk_geom(int64_t L, int J, int64_t R, int64_t S, int T) {
    if (J <= 1) return {1, L, L};
    const int mid = J - 2;
    double wf = 1.0, wl = 1.0;
    if (mid > 0 && 2 * R <= S) {
        wl = std::max(1.0, (double)mid * (double)R / (double)(S - R));
        wf = std::max(1.0, wl * kMidNoReadoutCost);
    }
    const double wsum = wf + mid + wl;
    const int64_t Lm = std::max<int64_t>(T, ((int64_t)std::ceil((double)L / wsum) + T - 1) / T * T);
    const int64_t L0 = std::max<int64_t>(T, ((int64_t)std::ceil(wf * (double)L / wsum) + T - 1) / T * T);
    int m = mid;
    while (m >= 0 && L - L0 - (int64_t)m * Lm <= 0) --m;
    if (m < 0) return {1, L, L};
    return {m + 2, L0, Lm};
}

}  // namespace ssi
