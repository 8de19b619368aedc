// Multi-direction selective scan with the merge fused (sm_103a):
//   K = 2: Vision Mamba bidirectional scan (forward + reversed, summed);
//   K = 4: VMamba SS2D (row-major, column-major, and both reversed, summed);
//   K = 1: a single direction for shapes the TMA path does not take.
//
// Sources: "Mamba Series from Selective State Spaces to Visual State Space
// Models", section "key code" (cross_scan_fwd builds the four orders by
// flattening the map and its transpose and flipping both; the merge flips and
// transposes each output back and sums them); "From LSTM to Mamba" (Vision
// Mamba), section 3.1 (forward scan + scan of the reversed sequence).
//
// Design: one CTA owns CB channels of one (batch, group) and runs all K
// directions at once, one group of WPD warps per direction.  No permuted copy of
// the map is made: each direction reads u at the position its traversal visits
// (index arithmetic on the H x W map), reads its own Delta_k, B_k and C_k in its
// scan order (as the key code's projections of the reordered sequences produce
// them), and adds its readout y_k into an fp32 accumulator of the channel's
// whole map in shared memory.  After the last step the CTA adds (sum_k D_k) * u, applies the gate
// and writes the map once.  Each accumulator receives at most two addends per
// position (K = 4 uses one accumulator for the two row-major directions and one
// for the two column-major ones), so the sum does not depend on the order in
// which the directions reach a position: the result is deterministic.
//
// Inputs of the next chunk are gathered into registers while the current chunk
// is scanned.
#pragma once

#include "ss_device.cuh"
#include "ss_scan1d.cuh"

namespace ssk {

template <typename IO_, int N_, int NPT_, int K_, int WPD_, int T_ = 32>
struct CfgM {
    using IO = IO_;
    static constexpr int N = N_, NPT = NPT_, K = K_, WPD = WPD_;
    static constexpr int R = N / NPT;
    static constexpr int CPW = 32 / R;
    static constexpr int CL = 1;                // channels per lane (scan_chunk_pipe)
    static constexpr bool BCW = false;          // B/C staged as fp32 pairs
    static constexpr int CB = WPD * CPW;        // channels per CTA
    static constexpr int DT = 32 * WPD;         // threads per direction
    static constexpr int THREADS = K * DT;
    static constexpr int T = T_;                // steps per chunk
    static constexpr int TP = T / 2;
    static constexpr int E = T / R;             // steps gathered and prepped by one lane
    static constexpr int NACC = (K == 4) ? 2 : 1;
    static constexpr int NBC = 2 * N * T;               // B/C values of one chunk
    static constexpr int BCV = (NBC + DT - 1) / DT;     // gathered by one thread per chunk
    static_assert(R >= 1 && R <= 8 && (R & (R - 1)) == 0, "1..8 lanes per channel");
    static_assert(E >= 2 && E % 2 == 0, "a prep lane owns whole step pairs");
    static constexpr int BCBUF = TP * 4 * N * 4;
    static constexpr int DXROW = (TP + 1) * 16;
    static constexpr int DIRBYTES = 2 * BCBUF + CB * DXROW;
    // accumulator row stride (floats): >= L, == 8 (mod 32) so the CPW channels of
    // a warp land on different banks
    static __host__ __device__ int64_t acc_stride(int64_t L) { return ((L + 31) / 32) * 32 + 8; }
    static __host__ __device__ int64_t acc_bytes(int64_t L) { return NACC * CB * acc_stride(L) * 4; }
    static __host__ int64_t smem_bytes(int64_t L) { return acc_bytes(L) + K * DIRBYTES + 16; }
};

struct MultiParams {
    int64_t dim, L;
    int H, W;
    int G, dpg;
    int orders[4];
    FastDiv divH;
    const void *u, *delta, *B, *C, *z;
    const float *A, *D, *bias;
    int softplus;
    int zoh;            // single direction only: zero-order-hold input matrix
    const float *h0;    // single direction only: initial state [batch*dim, N]
    void *out;
    float *last_state;
};

template <class C>
__global__ void __launch_bounds__(C::THREADS) k_multidir(const MultiParams p) {
    using IO = typename C::IO;
    constexpr int N = C::N, NPT = C::NPT, R = C::R, T = C::T, E = C::E, K = C::K;
    extern __shared__ __align__(16) uint8_t smem_m[];
    uint8_t *smem = smem_m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int k = warp / C::WPD;                  // direction of this warp
    const int td = tid - k * C::DT;               // thread index within the direction
    const int c = lane % C::CPW, g = lane / C::CPW;  // slice-major lanes
    const int ch = (warp % C::WPD) * C::CPW + c;  // channel within the CTA
    const int cblk = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / p.G, grp = bg % p.G;
    const int dg = cblk * C::CB + ch;
    const bool valid = dg < p.dpg;
    const int64_t d = (int64_t)grp * p.dpg + (valid ? dg : p.dpg - 1);
    const int64_t L = p.L;
    const int order = p.orders[k];
    const int64_t LS = C::acc_stride(L);
    const int nchunks = (int)((L + T - 1) / T);

    const IO *u = reinterpret_cast<const IO *>(p.u);
    const IO *u_row = u + ((int64_t)b * p.dim + d) * L;
    const IO *dl_row = reinterpret_cast<const IO *>(p.delta) + (((int64_t)b * K + k) * p.dim + d) * L;
    const IO *Bk = reinterpret_cast<const IO *>(p.B) + (((int64_t)b * K + k) * p.G + grp) * N * L;
    const IO *Ck = reinterpret_cast<const IO *>(p.C) + (((int64_t)b * K + k) * p.G + grp) * N * L;

    float2 A2p[1][NPT];
    float h[1][NPT];
    float iAv[NPT];  // 1/A (0 where A = 0), for the zero-order hold
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        const float araw = __ldg(p.A + ((int64_t)k * p.dim + d) * N + g * NPT + j);
        A2p[0][j] = make_float2(araw * kLog2e, araw * kLog2e);
        iAv[j] = araw != 0.f ? 1.f / araw : 0.f;
        h[0][j] = (K == 1 && p.h0) ? __ldg(p.h0 + ((int64_t)b * p.dim + d) * N + g * NPT + j) : 0.f;
    }
    const bool zoh = K == 1 && p.zoh;
    const float bk = p.bias ? __ldg(p.bias + (int64_t)k * p.dim + d) : 0.f;

    float *acc = reinterpret_cast<float *>(smem);
    float *my_acc = acc + ((C::NACC == 2 && (order == 1 || order == 3)) ? C::CB * LS : 0) + ch * LS;
    uint8_t *dir = smem + C::acc_bytes(L) + k * C::DIRBYTES;
    float *bcbuf0 = reinterpret_cast<float *>(dir);
    float4 *dxrow = reinterpret_cast<float4 *>(dir + 2 * C::BCBUF + ch * C::DXROW);

    // zero the accumulators
    {
        float4 *a4 = reinterpret_cast<float4 *>(acc);
        const int64_t n4 = C::acc_bytes(L) / 16;
        for (int64_t i = tid; i < n4; i += C::THREADS) a4[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }

    // register prefetch of one chunk: this lane's E steps of u and Delta_k, and
    // BCV values of B_k / C_k for this direction
    float ru[E], rd[E], rbc[C::BCV];
    auto fetch = [&](int i) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int64_t s = (int64_t)i * T + E * g + e;
            if (s < L) {
                const int64_t pos = position_of(order, s, L, p.H, p.W, p.divH);
                ru[e] = IOT<IO>::load(u_row + pos);
                rd[e] = IOT<IO>::load(dl_row + s);
            } else {
                ru[e] = 0.f;
                rd[e] = 0.f;
            }
        }
#pragma unroll
        for (int m = 0; m < C::BCV; ++m) {
            const int vi = td + m * C::DT;
            const int e = vi % T;
            const int rest = vi / T;
            const int n = rest % N;
            const int isC = rest / N;
            const int64_t s = (int64_t)i * T + e;
            float v = 0.f;
            if (vi < C::NBC && s < L) v = IOT<IO>::load((isC ? Ck : Bk) + (int64_t)n * L + s);
            rbc[m] = v;
        }
    };
    fetch(0);
    __syncthreads();

#pragma unroll 1
    for (int i = 0; i < nchunks; ++i) {
        float *bc = bcbuf0 + (i & 1) * (C::BCBUF / 4);
        // prep this lane's steps: Delta' and x = Delta' * u
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            float dlv[2], xv[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float v = rd[e + q] + bk;
                if (p.softplus) v = softplus(v);
                if ((int64_t)i * T + E * g + e + q >= L) v = 0.f;
                dlv[q] = v;
                xv[q] = zoh ? ru[e + q] : v * ru[e + q];
            }
            dxrow[swz_slot((E * g + e) >> 1)] = make_float4(dlv[0], dlv[1], xv[0], xv[1]);
        }
#pragma unroll
        for (int m = 0; m < C::BCV; ++m) {
            const int vi = td + m * C::DT;
            const int e = vi % T;
            const int rest = vi / T;
            const int n = rest % N;
            const int isC = rest / N;
            if (vi < C::NBC) bc[(e >> 1) * 4 * N + isC * 2 * N + 2 * n + (e & 1)] = rbc[m];
        }
        if (i + 1 < nchunks) fetch(i + 1);
        __syncthreads();

        const float4 *const dxrows[1] = {dxrow};
        auto emit = [&](int, float y, int t) {
            const int64_t s = (int64_t)i * T + t;
            if (s < L) {
                const int64_t pos = position_of(order, s, L, p.H, p.W, p.divH);
                if constexpr (K == 1)
                    my_acc[pos] = y;
                else
                    atomicAdd(my_acc + pos, y);
            }
        };
        if (zoh) scan_chunk_pipe<C, true, true>(dxrows, bc, g, h, A2p, emit, iAv);
        else scan_chunk_pipe<C, true>(dxrows, bc, g, h, A2p, emit);
    }
    __syncthreads();

    // merge: out = (sum of accumulators + sum_k D_k * u) * gate
    {
        const IO *z = reinterpret_cast<const IO *>(p.z);
        IO *out = reinterpret_cast<IO *>(p.out);
        const int64_t total = (int64_t)C::CB * L;
        for (int64_t idx = tid; idx < total; idx += C::THREADS) {
            const int chm = (int)(idx / L);
            const int64_t pos = idx - (int64_t)chm * L;
            const int dgm = cblk * C::CB + chm;
            if (dgm >= p.dpg) continue;
            const int64_t dm = (int64_t)grp * p.dpg + dgm;
            float y = acc[chm * LS + pos];
            if (C::NACC == 2) y += acc[(C::CB + chm) * LS + pos];
            float dsum = 0.f;
            if (p.D) {
#pragma unroll
                for (int kk = 0; kk < K; ++kk) dsum += __ldg(p.D + kk * p.dim + dm);
            }
            const int64_t gi = ((int64_t)b * p.dim + dm) * L + pos;
            y = fmaf(dsum, IOT<IO>::load(u + gi), y);
            if (z) y *= silu(IOT<IO>::load(z + gi));
            out[gi] = IOT<IO>::from_f(y);
        }
    }
    if (valid && p.last_state) {
#pragma unroll
        for (int j = 0; j < NPT; ++j)
            p.last_state[(((int64_t)b * K + k) * p.dim + d) * N + g * NPT + j] = h[0][j];
    }
}

}  // namespace ssk
