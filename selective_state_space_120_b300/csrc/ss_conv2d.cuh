// Depthwise 3 x 3 convolution + SiLU: the input branch of VMamba's SS2D block
// ("Mamba Series from Selective State Spaces to Visual State Space Models", VSS
// block structure and SS2Dv0.forwardv0: DWConv 3x3 -> SiLU before the
// four-direction scan), sm_103a.
//
//   u[b, d, r, c] = SiLU(bias[d] + sum_{i,j in -1..1} w[d, i+1, j+1] * x[b, d, r+i, c+j])
//
// with zero padding of one cell (a cross-correlation, as a framework's conv2d
// computes it).  It is a memory-bound stencil.  Maps up to 256 wide take the
// band kernel (whole rows of a plane staged in shared memory); wider ones the
// tile kernel, which stages a (TH + 2) x (TW + 2) window of one channel plane
// with coalesced row loads, each thread forming TH*TW/256 outputs from it.
#pragma once

#include "ss_device.cuh"

namespace ssk {

constexpr int DWC_TW = 64, DWC_TH = 16, DWC_THREADS = 256;

template <typename IO>
__global__ void __launch_bounds__(DWC_THREADS)
k_dwconv3x3_silu(const IO *__restrict__ x, const float *__restrict__ w, const float *__restrict__ bias,
                 IO *__restrict__ u, int64_t planes, int dim, int H, int W) {
    __shared__ float tile[DWC_TH + 2][DWC_TW + 3];
    const int tid = threadIdx.x;
    const int tx = tid % DWC_TW, ty = tid / DWC_TW;  // 64 x 4
    const int c0 = blockIdx.x * DWC_TW, r0 = blockIdx.y * DWC_TH;
    for (int64_t pl = blockIdx.z; pl < planes; pl += gridDim.z) {
        const int d = (int)(pl % dim);
        const IO *xp = x + pl * H * W;
        for (int i = tid; i < (DWC_TH + 2) * (DWC_TW + 2); i += DWC_THREADS) {
            const int rr = i / (DWC_TW + 2), cc = i - rr * (DWC_TW + 2);
            const int r = r0 + rr - 1, c = c0 + cc - 1;
            tile[rr][cc] = (r >= 0 && r < H && c >= 0 && c < W) ? IOT<IO>::load(xp + (int64_t)r * W + c) : 0.f;
        }
        float wk[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) wk[k] = __ldg(w + (int64_t)d * 9 + k);
        const float bd = bias ? __ldg(bias + d) : 0.f;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < DWC_TH / 4; ++k) {
            const int rr = ty + 4 * k;
            const int r = r0 + rr, c = c0 + tx;
            float v = bd;
#pragma unroll
            for (int i = 0; i < 3; ++i)
#pragma unroll
                for (int j = 0; j < 3; ++j) v = fmaf(wk[i * 3 + j], tile[rr + i][tx + j], v);
            if (r < H && c < W) u[pl * H * W + (int64_t)r * W + c] = IOT<IO>::from_f(silu(v));
        }
        __syncthreads();
    }
}

// Whole rows at a time, for maps up to DWC_BAND_MAXW wide: a CTA stages rows
// r0-1 .. r0+RB of one channel plane, zero-padded to W + 2 columns, in dynamic
// shared memory, and writes rows r0 .. r0+RB-1.  Rows that are a multiple of 16
// bytes arrive with 16-byte loads.  Blocks (band, plane) stride over the planes.
constexpr int DWC_BAND_MAXW = 256;

template <typename IO>
__global__ void __launch_bounds__(DWC_THREADS)
k_dwconv3x3_silu_band(const IO *__restrict__ x, const float *__restrict__ w,
                      const float *__restrict__ bias, IO *__restrict__ u, int64_t planes, int dim,
                      int H, int W, int RB) {
    extern __shared__ float band[];  // [RB + 2][W + 2]
    const int tid = threadIdx.x;
    const int WP = W + 2;
    const int r0 = blockIdx.y * RB;
    const int rows = min(RB, H - r0);  // output rows of this band
    constexpr int VPC = 16 / (int)sizeof(IO);  // elements per 16-byte chunk
    const bool vec = (W % VPC) == 0;
    for (int64_t pl = blockIdx.x; pl < planes; pl += gridDim.x) {
        const int d = (int)(pl % dim);
        const IO *xp = x + pl * H * W;
        // zero the halo columns, then the rows (zero outside the map)
        for (int i = tid; i < rows + 2; i += DWC_THREADS) {
            band[i * WP] = 0.f;
            band[i * WP + W + 1] = 0.f;
        }
        if (vec) {
            const int cpr = W / VPC;  // chunks per row
            for (int i = tid; i < (rows + 2) * cpr; i += DWC_THREADS) {
                const int rr = i / cpr, q = i - rr * cpr;
                const int r = r0 + rr - 1;
                float v[VPC];
                if (r >= 0 && r < H) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(xp + (int64_t)r * W + q * VPC);
                    const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) unpack_word(wds[k], v + k * (VPC / 4), (IO *)nullptr);
                } else {
#pragma unroll
                    for (int k = 0; k < VPC; ++k) v[k] = 0.f;
                }
#pragma unroll
                for (int k = 0; k < VPC; ++k) band[rr * WP + 1 + q * VPC + k] = v[k];
            }
        } else {
            for (int i = tid; i < (rows + 2) * W; i += DWC_THREADS) {
                const int rr = i / W, c = i - rr * W;
                const int r = r0 + rr - 1;
                band[rr * WP + 1 + c] = (r >= 0 && r < H) ? IOT<IO>::load(xp + (int64_t)r * W + c) : 0.f;
            }
        }
        float wk[9];
#pragma unroll
        for (int k = 0; k < 9; ++k) wk[k] = __ldg(w + (int64_t)d * 9 + k);
        const float bd = bias ? __ldg(bias + d) : 0.f;
        __syncthreads();
        // thread = (column c, run of consecutive rows): the 3 x 3 window slides
        // down the run, three new values per output row
        IO *up = u + pl * H * W + (int64_t)r0 * W;
        const int nseg = DWC_THREADS / W;  // runs side by side (W <= 256)
        const int seg = tid / W, c = tid - seg * W;
        const int run = (rows + nseg - 1) / nseg;
        const int ra = seg * run, rb = min(rows, ra + run);
        if (seg < nseg && ra < rb) {
            float t0[3], t1[3], t2[3];
#pragma unroll
            for (int b2 = 0; b2 < 3; ++b2) {
                t0[b2] = band[ra * WP + c + b2];
                t1[b2] = band[(ra + 1) * WP + c + b2];
            }
            for (int rr = ra; rr < rb; ++rr) {
#pragma unroll
                for (int b2 = 0; b2 < 3; ++b2) t2[b2] = band[(rr + 2) * WP + c + b2];
                float v = bd;
#pragma unroll
                for (int b2 = 0; b2 < 3; ++b2) {
                    v = fmaf(wk[b2], t0[b2], v);
                    v = fmaf(wk[3 + b2], t1[b2], v);
                    v = fmaf(wk[6 + b2], t2[b2], v);
                }
                up[(int64_t)rr * W + c] = IOT<IO>::from_f(silu(v));
#pragma unroll
                for (int b2 = 0; b2 < 3; ++b2) {
                    t0[b2] = t1[b2];
                    t1[b2] = t2[b2];
                }
            }
        }
        __syncthreads();
    }
}

}  // namespace ssk
