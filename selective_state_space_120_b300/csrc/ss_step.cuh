// One step of the selective recurrence for token-by-token inference (sm_103a).
//
// "Mamba论文" reading notes (recurrent mode for inference) and "Mamba Series
// ...", mathematical form of the selective SSM: per (batch b, channel d),
//   dt = softplus(Delta + bias);  h_n = exp(dt A_n) h_n + Bbar_n x;
//   y = (sum_n C_n h_n + D x) * SiLU(z).
// One thread owns one channel and its N fp32 states: the step is a few hundred
// bytes of state traffic per channel, so the kernel is a plain streaming pass
// with 16-byte state and A accesses; B/C of a group are read by all its
// channels and stay in L1/L2.
#pragma once

#include "ss_device.cuh"

namespace ssk {

struct StepParams {
    int64_t rows, dim;
    int G, dpg;
    const void *x, *delta, *B, *C, *z;
    const float *A, *D, *bias;
    int softplus, zoh;
    float *state;
    void *out;
};

template <typename IO, int N>
__global__ void __launch_bounds__(128) k_step(const StepParams p) {
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= p.rows) return;
    const int64_t b = row / p.dim, d = row - b * p.dim;
    const int64_t grp = d / p.dpg;
    const IO *B = reinterpret_cast<const IO *>(p.B) + (b * p.G + grp) * N;
    const IO *C = reinterpret_cast<const IO *>(p.C) + (b * p.G + grp) * N;
    const float x = IOT<IO>::load(reinterpret_cast<const IO *>(p.x) + row);
    float dt = IOT<IO>::load(reinterpret_cast<const IO *>(p.delta) + row) + (p.bias ? __ldg(p.bias + d) : 0.f);
    if (p.softplus) dt = softplus(dt);
    float *h = p.state + row * N;
    const float *A = p.A + d * N;
    float y = 0.f;
#pragma unroll
    for (int n0 = 0; n0 < N; n0 += 4) {
        float hv[4], av[4];
        if constexpr (N >= 4) {
            const float4 h4 = *reinterpret_cast<const float4 *>(h + n0);
            const float4 a4 = __ldg(reinterpret_cast<const float4 *>(A + n0));
            hv[0] = h4.x; hv[1] = h4.y; hv[2] = h4.z; hv[3] = h4.w;
            av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                hv[j] = n0 + j < N ? h[n0 + j] : 0.f;
                av[j] = n0 + j < N ? __ldg(A + n0 + j) : 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (n0 + j >= N) break;
            const float abar = ex2(dt * av[j] * kLog2e);
            float bbar = dt;  // Euler: Bbar = dt * B
            if (p.zoh) {
                // (exp(dt A) - 1) / A, with the series of expm1(v)/v near 0
                const float v = dt * av[j];
                bbar = fabsf(v) < 0.0625f ? dt * fmaf(v, fmaf(v, fmaf(v, 1.f / 24.f, 1.f / 6.f), 0.5f), 1.f)
                                          : (abar - 1.f) / av[j];
            }
            hv[j] = fmaf(abar, hv[j], bbar * IOT<IO>::load(B + n0 + j) * x);
            y = fmaf(IOT<IO>::load(C + n0 + j), hv[j], y);
        }
        if constexpr (N >= 4) {
            *reinterpret_cast<float4 *>(h + n0) = make_float4(hv[0], hv[1], hv[2], hv[3]);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (n0 + j < N) h[n0 + j] = hv[j];
        }
    }
    if (p.D) y = fmaf(__ldg(p.D + d), x, y);
    if (p.z) y *= silu(IOT<IO>::load(reinterpret_cast<const IO *>(p.z) + row));
    reinterpret_cast<IO *>(p.out)[row] = IOT<IO>::from_f(y);
}

}  // namespace ssk
