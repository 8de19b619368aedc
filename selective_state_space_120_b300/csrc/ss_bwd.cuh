// Backward pass of the selective scan (sm_103a): one direction, and the
// directions of multi-direction calls (MULTI = true, below the description).
//
// Forward (Euler input matrix, zero initial state), per channel d and state n:
//   Delta'_t = softplus(delta_t + bias_d)     Abar_t = exp(Delta'_t A_n)
//   h_t = Abar_t h_{t-1} + Delta'_t B_t u_t   s_t = C_t . h_t + D_d u_t
//   out_t = s_t SiLU(z_t)
// Reverse mode for an upstream gradient dout, with ds_t = dout_t SiLU(z_t):
//   dh_t      = ds_t C_t + Abar_{t+1} (.) dh_{t+1}        (runs backwards in t)
//   dDelta'_t = sum_n dh_{t,n} (h_{t-1,n} Abar_{t,n} A_n + B_{t,n} u_t)
//   ddelta_t  = dDelta'_t softplus'(delta_t + bias_d)
//   du_t      = ds_t D_d + Delta'_t sum_n dh_{t,n} B_{t,n}
//   dz_t      = dout_t s_t SiLU'(z_t)
//   dA_n     += dh_{t,n} h_{t-1,n} Abar_{t,n} Delta'_t    (summed over batch and time)
//   dB_{t,n} += dh_{t,n} Delta'_t u_t,  dC_{t,n} += ds_t h_{t,n}   (over a group's channels)
//   dD_d     += ds_t u_t,  dbias_d += ddelta_t              (over batch and time)
// The review of the Mamba series (core insight 1) and the Mamba reading notes
// (section 3.3.2) describe the backward pass of the hardware-aware scan: the
// intermediate states are recomputed on chip rather than stored in HBM and
// read back.  This kernel recomputes them from sparse checkpoints.
//
// Work split: a CTA owns CB channels of one (batch, group).  Inside a warp,
// lane = g*CPW + q holds NPT of the N states (slice g) of CL channels (group q).
// Each CTA walks its rows twice through one TMA ring:
//   pass F, tiles 0 .. nt-1: the states only, storing them every TS steps as
//     checkpoints in the workspace (fp32);
//   pass B, tiles nt-1 .. 0, each tile's TS-step blocks last to first: from the
//     block's checkpoint the lane recomputes its chains' TS states into
//     registers together with the readout s_t, then runs the reverse recurrence
//     over the block; Abar (.) dh is carried in registers from block to block.
// State math runs on pairs of states with packed f32x2 operations.  Sums over
// the N states (s_t, dDelta'_t, sum_n dh B) are combined across a channel's R
// lanes by the transposing butterfly, R steps at a time, so that lane g
// finishes step g of each R-step group.  dB and dC are sums over the channels
// of a group: in registers over a lane's CL channels, then per step a
// transposing butterfly over the CPW lanes of a state slice, then per-warp sums
// in shared memory that the CTA adds up after each block and adds to the fp32
// outputs with 16-byte atomic adds.  The shared-memory footprint is kept small
// enough (two ring stages, one sums buffer) for three CTAs of the N = 16
// configuration to share an SM: a Mamba-layer call then runs in a single wave.
// dA, dD and dbias are per-channel sums over time held in registers, added
// over the batch with atomics at the end.
//
// Multi-direction calls: direction k's gradients are those of one direction
// over its inputs taken in its traversal order.  Two directions run side by
// side over grid z; u, dout and z come as row-order tiles, forward or back to
// front, of the call's maps or of copies permuted into the direction's step
// order (k_transpose_planes or k_transpose_maps for the column order); du goes
// by scan step to an fp32 buffer per direction, which k_merge_bwd sums by
// position while forming dz from the sum of all directions' outputs before the
// gate.
#pragma once

#include <type_traits>
#include "ss_device.cuh"

namespace ssk {

template <typename IO_, int N_, int W_, int CL_ = 1, int NPT_ = 4, int TS_ = 16 / CL_,
          int MINB_ = 1, int STAGES_ = 2>
struct CfgB {
    using IO = IO_;
    static constexpr int N = N_, W = W_, CL = CL_, STAGES = STAGES_;
    static constexpr int MINB = MINB_;             // CTAs per SM the register budget allows
    static constexpr int NPT = N < NPT_ ? N : NPT_;  // states per lane
    static constexpr int NPE = NPT < 2 ? 2 : NPT;  // padded to whole pairs (N = 1: a phantom state)
    static constexpr int NP = NPE / 2;             // state pairs per lane
    static constexpr int NB = N < 2 ? 2 : N;       // B (and C) slots per step in shared memory
    static constexpr int R = N / NPT;              // lanes per channel group
    static constexpr int CPW = 32 / R;             // channel groups per warp
    static constexpr int CHW = CPW * CL;           // channels per warp
    static constexpr int CB = W * CHW;             // channels per CTA
    static constexpr int THREADS = 32 * W;
    static constexpr int ES = sizeof(IO);
    static constexpr int T = 64 / ES;              // steps per tile (64-byte raw rows)
    static constexpr int TS = TS_;                 // steps per register block = checkpoint interval
    static constexpr int NS = T / TS;              // register blocks per tile
    static constexpr int RB = TS / R;              // R-step readout groups per block
    static constexpr int PT = R / CL;              // prep threads per channel
    static constexpr int E = T / PT;               // steps one thread preps
    static constexpr int EP = E < 8 ? E : 8;       // steps converted at a time
    static constexpr int V = 2 * NPE;              // dB and dC terms of a lane per step
    static_assert(N % NPT == 0 && (R & (R - 1)) == 0 && R <= TS && TS % R == 0, "lane split");
    static_assert(CL >= 1 && R % CL == 0 && T % TS == 0 && TS % 4 == 0, "block split");
    static_assert(E % EP == 0 && EP * ES >= 4, "prep split");
    static_assert(CB <= 256 && N <= 256, "TMA box rows");

    static constexpr int al(int x) { return (x + 1023) & ~1023; }
    static constexpr int TILE_CH = al(CB * 64);
    static constexpr int TILE_BC = al(N * 64);
    static constexpr int STAGE = 4 * TILE_CH + 2 * TILE_BC;
    static constexpr int OFF_U = 0, OFF_DL = TILE_CH, OFF_Z = 2 * TILE_CH, OFF_DY = 3 * TILE_CH;
    static constexpr int OFF_B = 4 * TILE_CH, OFF_C = 4 * TILE_CH + TILE_BC;
    static constexpr int BCF = T * 2 * NB * 4;      // fp32 B, C of a tile: [t][B_0..NB-1 | C_0..NB-1]
    static constexpr int OFF_BCF = STAGES * STAGE;  // two tiles' worth (tile parity)
    static constexpr int P0ROW = (T + 1) * 16;      // per step {Delta', Delta'u, ds, softplus'}
    static constexpr int P1ROW = (T + 1) * 8;       // per step {u, dout SiLU'(z)}
    static constexpr int OFF_P0 = OFF_BCF + 2 * BCF;
    static constexpr int OFF_P1 = OFF_P0 + CB * P0ROW;
    static constexpr int OBROW = 64 + 16;           // staged du / ddelta / dz rows (I/O type)
    static constexpr int OFF_OB = OFF_P1 + CB * P1ROW;
    static constexpr int REDW = TS * 2 * N * 4;     // one warp's dB/dC sums over one block
    static constexpr int OFF_RED = OFF_OB + 3 * CB * OBROW;
    static constexpr int OFF_BAR = (OFF_RED + W * REDW + 7) & ~7;
    static constexpr int SMEM = OFF_BAR + 8 * STAGES + 1024;  // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
    // Per-step rows of channel ch sit in order (ch % CL, ch / CL): the CPW lanes
    // of a quarter-warp read CPW consecutive rows, whose odd 16-byte stride
    // spreads them over all banks.
    static __device__ __forceinline__ int prow(int ch) { return (ch % CL) * (CB / CL) + ch / CL; }
};

struct BwdParams {
    int64_t dim, L;
    int G, dpg;
    int nblk;                 // checkpoint blocks per row
    const float *A, *D, *bias;
    int softplus, has_z;
    float *ckpt;              // [batch*dim, nblk, N]: state after each block (pass F)
    void *du, *ddelta, *dz;   // [batch, dim, L], I/O type
    float *dA;                // [dim, N]
    float *dB, *dC;           // [batch, G, N, L]
    float *dD, *dbias;        // [dim], nullable
    // multi-direction calls (MULTI kernels): direction k of K.  Delta, B, C,
    // ddelta, dB, dC are direction k's (scan order); u, z, dout come as tiles of
    // maps in direction k's step order, read forward (order 0) or back to front
    // (order 2); du goes by scan step, in fp32, to du_acc [batch*dim, L]; dz is
    // left to the merge.
    // Two directions may run side by side: blockIdx.z = j scans direction k_z[j]
    // with order_z[j] over the u, z, dout maps of the launch, its checkpoints at
    // ckpt + j*ck_zstride and its du at du_acc + k_z[j]*du_zstride.
    int K;
    int k_z[2], order_z[2];
    float *du_acc;
    int64_t du_zstride, ck_zstride;
    // single direction, option instantiations (EXT kernels): the zero-order-hold
    // input matrix, an initial state h0 [batch*dim, N] (nullable) and the
    // gradient of the loss with respect to it, dh0 [batch*dim, N] (nullable)
    int zoh;
    const float *h0;
    float *dh0;
};

// Zero-order hold: Bbar u = psi * B u with psi = (exp(x) - 1)/A, x = Delta' A,
// and its derivative with respect to A, (Delta' exp(x) - psi)/A.  For |x| <
// 1/16 both come from the Taylor series of (exp(x) - 1)/x (truncation below
// x^4/120 relative), which avoids the cancellation of exp(x) - 1:
//   psi = Delta' (1 + x/2 + x^2/6 + x^3/24),  dpsi/dA = Delta'^2 (1/2 + x/3 + x^2/8 + x^3/30).
// A = 0 gives psi = Delta' (x = 0) through the series.  ia = 1/A (0 for A = 0).
__device__ __forceinline__ float zoh_psi(float dl, float a, float xn, float ia) {
    return fabsf(xn) < 0.0625f ? dl * fmaf(xn, fmaf(xn, fmaf(xn, 1.f / 24.f, 1.f / 6.f), 0.5f), 1.f)
                               : (a - 1.f) * ia;
}
__device__ __forceinline__ float zoh_dpsi_dA(float dl, float a, float xn, float ia, float psi) {
    return fabsf(xn) < 0.0625f
               ? dl * dl * fmaf(xn, fmaf(xn, fmaf(xn, 1.f / 30.f, 0.125f), 1.f / 3.f), 0.5f)
               : (dl * a - psi) * ia;
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 ex2x2(float2 v) { return make_float2(ex2(v.x), ex2(v.y)); }

// Sums the V dB/dC terms of one step over the P channel-group lanes of a state
// slice (lanes g*P + q, q = 0..P-1) and writes the sums to dst = [dB_0..N-1 |
// dC_0..N-1] of that step.  Term vi is dB of state g*NPT + vi for vi < NPE and
// dC of state g*NPT + vi - NPE otherwise (padded states are dropped).
template <int V, int P, int N, int NPT, int NPE>
__device__ __forceinline__ void reduce_bc_store(float (&v)[V], int q, int g, float *dst) {
    auto put = [&](int vi, float x) {
        const int j = vi % NPE;
        if (j < NPT) dst[(vi < NPE ? 0 : N) + g * NPT + j] = x;
    };
    if constexpr (P == 1) {
#pragma unroll
        for (int vi = 0; vi < V; ++vi) put(vi, v[vi]);
    } else if constexpr (V >= P) {
#pragma unroll
        for (int m = 0; m < V / P; ++m) {
            float part[P];
#pragma unroll
            for (int k = 0; k < P; ++k) part[k] = v[m * P + k];
            put(m * P + q, transpose_reduce<P, 1>(part, q));
        }
    } else {
        float r = transpose_reduce<V, 1>(v, q & (V - 1));
#pragma unroll
        for (int m = V; m < P; m <<= 1) r += __shfl_xor_sync(kFull, r, m);
        if (q < V) put(q, r);
    }
}

// EXT (single direction only) compiles the options: the zero-order hold and the
// initial state with its gradient; the plain instantiations carry none of
// their code.
template <class C, bool MULTI = false, bool EXT = false>
__global__ void __launch_bounds__(C::THREADS, C::MINB)
k_scan_bwd(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
           const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dy,
           const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
           const BwdParams p) {
    using IO = typename C::IO;
    constexpr int N = C::N, NPT = C::NPT, NPE = C::NPE, NP = C::NP, NB = C::NB, R = C::R;
    constexpr int CPW = C::CPW, CL = C::CL, T = C::T, TS = C::TS, E = C::E, EP = C::EP;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = lane % CPW, g = lane / CPW;
    const int cblk = blockIdx.x, bg = blockIdx.y;
    const int b = bg / p.G, grp = bg % p.G;
    const int64_t L = p.L;
    const int64_t row0 = (int64_t)b * p.dim + (int64_t)grp * p.dpg;  // the group's channel 0
    const int row_tma = (int)(row0 + (int64_t)cblk * C::CB);          // u, z, dout rows
    const int zsl = MULTI ? (int)blockIdx.z : 0;                      // direction slice of the grid
    const int Kd = MULTI ? p.K : 1, kdir = MULTI ? (zsl ? p.k_z[1] : p.k_z[0]) : 0;  // directions, this one
    const int order = MULTI ? (zsl ? p.order_z[1] : p.order_z[0]) : 0;
    // Delta / ddelta rows [batch, K, dim]; B/C rows [batch, K, G, N]
    const int64_t dlrow0 = ((int64_t)b * Kd + kdir) * p.dim + (int64_t)grp * p.dpg;
    const int dlrow_tma = (int)(dlrow0 + (int64_t)cblk * C::CB);
    const int bcrow_tma = (int)((((int64_t)b * Kd + kdir) * p.G + grp) * N);
    const int64_t poff = (int64_t)kdir * p.dim;  // direction offset of A, D, bias and their gradients
    const int nt = (int)((L + T - 1) / T);
    const int nq = 2 * nt;  // ring order: pass F tiles 0..nt-1, then pass B tiles nt-1..0

    // scan role: states g*NPT .. of channels chs[c]
    int chs[CL];
    bool valid[CL];
    int64_t dch[CL];
    float2 A2[CL][NP], carry[CL][NP], dA[CL][NP];
    float2 iA2[EXT ? CL : 1][EXT ? NP : 1];  // 1/A per state (0 for A = 0), zero-order hold
    const bool zoh = EXT && p.zoh;
    float Dd[CL], dD_acc[CL], dbias_acc[CL];
    float *ck[CL];
    const float4 *P0[CL];
    const float2 *P1[CL];
#pragma unroll
    for (int c = 0; c < CL; ++c) {
        chs[c] = warp * C::CHW + q * CL + c;
        const int dg = cblk * C::CB + chs[c];
        valid[c] = dg < p.dpg;
        dch[c] = (int64_t)grp * p.dpg + (valid[c] ? dg : p.dpg - 1);
#pragma unroll
        for (int k = 0; k < NP; ++k) {
            const int j0 = 2 * k, j1 = 2 * k + 1;
            const float a0 = __ldg(p.A + (poff + dch[c]) * N + g * NPT + j0) * kLog2e;
            const float a1 = j1 < NPT ? __ldg(p.A + (poff + dch[c]) * N + g * NPT + j1) * kLog2e : 0.f;
            A2[c][k] = make_float2(a0, a1);
            carry[c][k] = make_float2(0.f, 0.f);
            dA[c][k] = make_float2(0.f, 0.f);
            if constexpr (EXT)
                iA2[c][k] = make_float2(a0 != 0.f ? kLog2e / a0 : 0.f, a1 != 0.f ? kLog2e / a1 : 0.f);
        }
        Dd[c] = p.D ? __ldg(p.D + poff + dch[c]) : 0.f;
        dD_acc[c] = 0.f;
        dbias_acc[c] = 0.f;
        ck[c] = p.ckpt + (MULTI ? zsl * p.ck_zstride : 0) + ((int64_t)b * p.dim + dch[c]) * p.nblk * N +
                g * NPT;
        P0[c] = reinterpret_cast<const float4 *>(smem + C::OFF_P0 + C::prow(chs[c]) * C::P0ROW);
        P1[c] = reinterpret_cast<const float2 *>(smem + C::OFF_P1 + C::prow(chs[c]) * C::P1ROW);
    }
    float *red0 = reinterpret_cast<float *>(smem + C::OFF_RED);
    float *bcf0 = reinterpret_cast<float *>(smem + C::OFF_BCF);

    // prep role: E consecutive steps of channel pch (a channel of this warp)
    const int pch = tid / C::PT;
    const int pt0 = (tid % C::PT) * E;
    const int pdg = cblk * C::CB + pch;
    const bool pvalid = pdg < p.dpg;
    const int64_t pd = (int64_t)grp * p.dpg + (pvalid ? pdg : p.dpg - 1);
    const float pbias = p.bias ? __ldg(p.bias + poff + pd) : 0.f;
    const int64_t prow = (int64_t)b * p.dim + pd;  // the prep channel's row of u, z, dout
    float4 *q0row = reinterpret_cast<float4 *>(smem + C::OFF_P0 + C::prow(pch) * C::P0ROW);
    float2 *q1row = reinterpret_cast<float2 *>(smem + C::OFF_P1 + C::prow(pch) * C::P1ROW);

    const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t nuF = 1u;                           // u
    const uint32_t nuB = 2u + (p.has_z ? 1u : 0u);     // u, dout, z
    const uint32_t txF = (nuF + 1u) * C::CB * 64u + N * 64u;
    const uint32_t txB = (nuB + 1u) * C::CB * 64u + 2u * N * 64u;
    const uint64_t budget = g_wait_budget_ns;

    if (tid == 0) {
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_dl);
        prefetch_tensormap(&tm_dy);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        if (p.has_z) prefetch_tensormap(&tm_z);
#pragma unroll 1
        for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    // padded B/C slots (N = 1) stay zero, so the padded state stays zero
    if (NB > N) {
        for (int i = tid; i < 2 * T * 2 * NB; i += C::THREADS)
            if (i % NB >= N) bcf0[i] = 0.f;
    }
    __syncthreads();

    // diagnostics: this CTA leaves its first tile's barrier without arrivals
    const bool skip_first = (g_debug_flags & 1u) && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0;
    auto tile_of = [&](int qs) { return qs < nt ? qs : nq - 1 - qs; };
    auto issue = [&](int qs) {
        if (qs == 0 && skip_first) return;
        const int s = qs % STAGES;
        const uint32_t bar = bar0 + 8 * s;
        const uint32_t st = smem0 + s * C::STAGE;
        const bool bwd = qs >= nt;
        const int x = tile_of(qs) * T;
        // u, z, dout of a reversed row order: positions L-(i+1)T .. L-1-iT (the
        // last tile may start below 0; the copy fills zeros there)
        const int xu = order == 2 ? (int)(L - (int64_t)(tile_of(qs) + 1) * T) : x;
        mbar_expect_tx(bar, bwd ? txB : txF);
        tma_load_2d(st + C::OFF_U, &tm_u, xu, row_tma, bar);
        tma_load_2d(st + C::OFF_DL, &tm_dl, x, dlrow_tma, bar);
        tma_load_2d(st + C::OFF_B, &tm_B, x, bcrow_tma, bar);
        if (bwd) {
            tma_load_2d(st + C::OFF_DY, &tm_dy, xu, row_tma, bar);
            if (p.has_z) tma_load_2d(st + C::OFF_Z, &tm_z, xu, row_tma, bar);
            tma_load_2d(st + C::OFF_C, &tm_C, x, bcrow_tma, bar);
        }
    };
    if (tid == 0) {
#pragma unroll 1
        for (int qs = 0; qs < STAGES && qs < nq; ++qs) issue(qs);
    }

    // Converts ring item qs (tile i) into fp32 B (and C) and per-step rows.
    auto prep = [&](int qs, int i, bool bwd) {
        const uint8_t *st = smem + (qs % STAGES) * C::STAGE;
        float *bcf = bcf0 + (qs & 1) * (C::BCF / 4);
        constexpr int VPC = 16 / C::ES;
        const int na = bwd ? 2 : 1;
#pragma unroll 1
        for (int task = tid; task < na * N * 4; task += C::THREADS) {
            const int n = task % N;
            const int arr = (task / N) % na;
            const int qq = task / (N * na);  // 16-byte chunk of the 64-byte row
            float v[VPC];
            load_tile_row<IO, VPC>(st + (arr ? C::OFF_C : C::OFF_B), n, qq * VPC, v);
#pragma unroll
            for (int e = 0; e < VPC; ++e) bcf[(qq * VPC + e) * 2 * NB + arr * NB + n] = v[e];
        }
        const int64_t tb0 = (int64_t)i * T;
#pragma unroll
        for (int e0 = 0; e0 < E; e0 += EP) {
            float uu[EP], dd[EP], zz[EP], gy[EP];
            load_tile_row<IO, EP>(st + C::OFF_DL, pch, pt0 + e0, dd);
            if (!MULTI || order == 0) {
                load_tile_row<IO, EP>(st + C::OFF_U, pch, pt0 + e0, uu);
                if (bwd) {
                    load_tile_row<IO, EP>(st + C::OFF_DY, pch, pt0 + e0, gy);
                    if (p.has_z) load_tile_row<IO, EP>(st + C::OFF_Z, pch, pt0 + e0, zz);
                }
            } else {
                // reversed tile: step pt0+e0+e sits at tile column T-1-(pt0+e0+e)
                float tmp[EP];
                const int col = T - (pt0 + e0) - EP;
                load_tile_row<IO, EP>(st + C::OFF_U, pch, col, tmp);
#pragma unroll
                for (int e = 0; e < EP; ++e) uu[e] = tmp[EP - 1 - e];
                if (bwd) {
                    load_tile_row<IO, EP>(st + C::OFF_DY, pch, col, tmp);
#pragma unroll
                    for (int e = 0; e < EP; ++e) gy[e] = tmp[EP - 1 - e];
                    if (p.has_z) {
                        load_tile_row<IO, EP>(st + C::OFF_Z, pch, col, tmp);
#pragma unroll
                        for (int e = 0; e < EP; ++e) zz[e] = tmp[EP - 1 - e];
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const int tl = pt0 + e0 + e;
                // steps past the sequence end and channels past the group leave h
                // unchanged and contribute nothing
                const bool in = pvalid && tb0 + tl < L;
                const float v = dd[e] + pbias;
                float dl = v, dsp = 1.f;
                if (p.softplus) {
                    // softplus and its derivative (the logistic function) from one exponential
                    const float ev = ex2(v * kLog2e);
                    dl = softplus_from_exp(v, ev);
                    dsp = v > 15.f ? 1.f - rcp(ev) : ev * rcp(1.f + ev);
                }
                if (!in) dl = 0.f;
                // the state's input term per unit B: Delta' u (Euler), or u, to be
                // scaled by psi per state (zero-order hold)
                const float x = zoh ? uu[e] : dl * uu[e];
                if (!bwd) {
                    *reinterpret_cast<float2 *>(q0row + tl) = make_float2(dl, x);
                } else {
                    float ds = gy[e], dzf = 0.f;
                    if (p.has_z) {
                        const float sg = rcp(1.f + ex2(-zz[e] * kLog2e));
                        ds = gy[e] * zz[e] * sg;
                        dzf = gy[e] * sg * fmaf(zz[e], 1.f - sg, 1.f);
                    }
                    q0row[tl] = make_float4(dl, x, in ? ds : 0.f, dsp);
                    q1row[tl] = make_float2(uu[e], dzf);
                }
            }
        }
    };
    // Bounded wait for ring item qs; on timeout the whole CTA drains its copies
    // and exits (returns true then).
    auto abandon = [&](int qs, bool ok) -> bool {
        if (!__syncthreads_or(!ok)) return false;
        if (tid == 0) {
            report_timeout();
#pragma unroll 1
            for (int k = qs; k < nq && k < qs + STAGES; ++k)
                if (!(k == 0 && skip_first))
                    (void)mbar_wait_bounded(bar0 + 8 * (k % STAGES), (k / STAGES) & 1, 1000000000ull);
        }
        return true;
    };
    // this lane's B or C pairs at tile-local step t
    auto ld_pairs = [&](const float *bcf, int t, int arr, float2 (&v)[NP]) {
        const float *src = bcf + t * 2 * NB + arr * NB + g * NPE;
        if constexpr (NP == 2) {
            const float4 w = *reinterpret_cast<const float4 *>(src);
            v[0] = make_float2(w.x, w.y);
            v[1] = make_float2(w.z, w.w);
        } else {
#pragma unroll
            for (int k = 0; k < NP; ++k) v[k] = *reinterpret_cast<const float2 *>(src + 2 * k);
        }
    };

    // checkpoint kc of channel c (the state after block kc; before block 0 the
    // initial state: zero, or h0)
    auto ld_ckpt = [&](int c, int kc, float2 (&v)[NP]) {
#pragma unroll
        for (int kk = 0; kk < NP; ++kk) v[kk] = make_float2(0.f, 0.f);
        const float *base = nullptr;
        if (kc >= 0) base = ck[c] + (int64_t)kc * N;
        else if (EXT && p.h0) base = p.h0 + ((int64_t)b * p.dim + dch[c]) * N + g * NPT;
        if (base) {
#pragma unroll
            for (int kk = 0; kk < NP; ++kk) {
                const float *src = base + 2 * kk;
                v[kk].x = src[0];
                if (2 * kk + 1 < NPT) v[kk].y = src[1];
            }
        }
    };
    // Bbar u of the lane's state pair kk of channel c at a step: (Delta' B) u, or
    // psi (B u) for the zero-order hold (pp = {Delta', x}, da = Delta' A log2 e)
    auto bx_pair = [&](int c, int kk, float2 pp, float2 da, float2 a, const float2 &B2) -> float2 {
        const float2 bu = __fmul2_rn(f2(pp.y), B2);
        if (!zoh) return bu;
        const float psi0 = zoh_psi(pp.x, a.x, da.x * kLn2, iA2[c][kk].x);
        const float psi1 = zoh_psi(pp.x, a.y, da.y * kLn2, iA2[c][kk].y);
        return __fmul2_rn(make_float2(psi0, psi1), bu);
    };

    float2 h[CL][NP], hbn[CL][NP];
#pragma unroll
    for (int c = 0; c < CL; ++c) ld_ckpt(c, -1, h[c]);

#pragma unroll 1
    for (int qs = 0; qs < nq; ++qs) {
        const bool bwd = qs >= nt;
        const int i = tile_of(qs);
        const bool ok = mbar_wait_bounded(bar0 + 8 * (qs % STAGES), (qs / STAGES) & 1, budget);
        if (ok) prep(qs, i, bwd);
        if (abandon(qs, ok)) return;
        if (tid == 0 && qs + STAGES < nq) {
            fence_proxy_async_smem();
            issue(qs + STAGES);
        }
        const float *bcf = bcf0 + (qs & 1) * (C::BCF / 4);

        if (!bwd) {
            // ---------------- pass F: checkpoints after each block
#pragma unroll 1
            for (int s = 0; s < C::NS; ++s) {
                const int k = i * C::NS + s;
                if (k >= p.nblk - 1) break;  // no later block starts from this state
#pragma unroll
                for (int tb = 0; tb < TS; ++tb) {
                    const int t = s * TS + tb;
                    float2 B2[NP];
                    ld_pairs(bcf, t, 0, B2);
#pragma unroll
                    for (int c = 0; c < CL; ++c) {
                        const float2 pp = *reinterpret_cast<const float2 *>(P0[c] + t);
#pragma unroll
                        for (int kk = 0; kk < NP; ++kk) {
                            const float2 da = __fmul2_rn(f2(pp.x), A2[c][kk]);
                            const float2 a = ex2x2(da);
                            h[c][kk] = __ffma2_rn(a, h[c][kk], bx_pair(c, kk, pp, da, a, B2[kk]));
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    if (!valid[c]) continue;
                    float *dst = ck[c] + (int64_t)k * N;
#pragma unroll
                    for (int kk = 0; kk < NP; ++kk) {
                        dst[2 * kk] = h[c][kk].x;
                        if (2 * kk + 1 < NPT) dst[2 * kk + 1] = h[c][kk].y;
                    }
                }
            }
            __syncwarp();
            continue;
        }

        // ---------------- pass B: blocks of tile i, last to first
        if (qs == nt) {
            // state entering the first block scanned backwards
            const int kf = p.nblk - 1;
#pragma unroll
            for (int c = 0; c < CL; ++c) ld_ckpt(c, kf - 1, hbn[c]);
        }
#pragma unroll 1
        for (int s = C::NS - 1; s >= 0; --s) {
            const int k = i * C::NS + s;
            if (k >= p.nblk) continue;  // the block lies past the sequence end
            const int t0b = s * TS;
            float2 hb[CL][NP];
#pragma unroll
            for (int c = 0; c < CL; ++c) {
#pragma unroll
                for (int kk = 0; kk < NP; ++kk) hb[c][kk] = hbn[c][kk];
                ld_ckpt(c, k - 2, hbn[c]);  // for the next block, one block ahead
            }

            // recompute the block's states and readouts
            float2 hs[TS][CL][NP];
            float sv[CL][C::RB];
            {
                float2 hc[CL][NP];
#pragma unroll
                for (int c = 0; c < CL; ++c)
#pragma unroll
                    for (int kk = 0; kk < NP; ++kk) hc[c][kk] = hb[c][kk];
#pragma unroll
                for (int rb = 0; rb < C::RB; ++rb) {
                    float sp[CL][R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int tb = rb * R + r;
                        float2 B2[NP], C2[NP];
                        ld_pairs(bcf, t0b + tb, 0, B2);
                        ld_pairs(bcf, t0b + tb, 1, C2);
#pragma unroll
                        for (int c = 0; c < CL; ++c) {
                            const float2 pp = *reinterpret_cast<const float2 *>(P0[c] + t0b + tb);
                            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                            for (int kk = 0; kk < NP; ++kk) {
                                const float2 da = __fmul2_rn(f2(pp.x), A2[c][kk]);
                                const float2 a = ex2x2(da);
                                hc[c][kk] = __ffma2_rn(a, hc[c][kk], bx_pair(c, kk, pp, da, a, B2[kk]));
                                hs[tb][c][kk] = hc[c][kk];
                                acc = __ffma2_rn(C2[kk], hc[c][kk], acc);
                            }
                            sp[c][r] = acc.x + acc.y;
                        }
                    }
#pragma unroll
                    for (int c = 0; c < CL; ++c) sv[c][rb] = transpose_reduce<R, CPW>(sp[c], g);
                }
            }

            // reverse recurrence over the block
            float *redw = red0 + warp * (TS * 2 * N);
#pragma unroll
            for (int rb = C::RB - 1; rb >= 0; --rb) {
                float p1v[CL][R], p2v[CL][R];
                float p3v[EXT ? CL : 1][EXT ? R : 1];  // zero-order hold: sum_n dh psi B (du)
#pragma unroll
                for (int r = R - 1; r >= 0; --r) {
                    const int tb = rb * R + r;
                    float2 B2[NP], C2[NP], vb[NP], vc[NP];
                    ld_pairs(bcf, t0b + tb, 0, B2);
                    ld_pairs(bcf, t0b + tb, 1, C2);
#pragma unroll
                    for (int c = 0; c < CL; ++c) {
                        const float4 pp = P0[c][t0b + tb];  // Delta', Delta'u, ds, softplus'
                        const float2 dl2 = f2(pp.x), x2 = f2(pp.y), ds2 = f2(pp.z);
                        float2 p1 = make_float2(0.f, 0.f), p2 = make_float2(0.f, 0.f);
                        float2 p3 = make_float2(0.f, 0.f);
#pragma unroll
                        for (int kk = 0; kk < NP; ++kk) {
                            const float2 da = __fmul2_rn(dl2, A2[c][kk]);
                            const float2 a = ex2x2(da);
                            const float2 dh = __ffma2_rn(ds2, C2[kk], carry[c][kk]);
                            const float2 hp = tb > 0 ? hs[tb - 1][c][kk] : hb[c][kk];
                            const float2 w = __fmul2_rn(__fmul2_rn(dh, hp), a);
                            p1 = __ffma2_rn(w, A2[c][kk], p1);
                            dA[c][kk] = __ffma2_rn(w, dl2, dA[c][kk]);
                            float2 db;
                            if (zoh) {
                                // Bbar u = psi B u: d/dDelta' = Abar B u, d/du = psi B,
                                // d/dB = psi u, d/dA = (dpsi/dA) B u
                                const float2 xn = __fmul2_rn(da, f2(kLn2));
                                const float ps0 = zoh_psi(pp.x, a.x, xn.x, iA2[c][kk].x);
                                const float ps1 = zoh_psi(pp.x, a.y, xn.y, iA2[c][kk].y);
                                const float2 psi = make_float2(ps0, ps1);
                                const float2 dpa = make_float2(zoh_dpsi_dA(pp.x, a.x, xn.x, iA2[c][kk].x, ps0),
                                                               zoh_dpsi_dA(pp.x, a.y, xn.y, iA2[c][kk].y, ps1));
                                const float2 dhb = __fmul2_rn(dh, B2[kk]);
                                p2 = __ffma2_rn(dhb, a, p2);
                                p3 = __ffma2_rn(dhb, psi, p3);
                                dA[c][kk] = __ffma2_rn(__fmul2_rn(dhb, x2), dpa, dA[c][kk]);
                                db = __fmul2_rn(__fmul2_rn(dh, psi), x2);
                            } else {
                                p2 = __ffma2_rn(dh, B2[kk], p2);
                                db = __fmul2_rn(dh, x2);
                            }
                            const float2 dc = __fmul2_rn(ds2, hs[tb][c][kk]);
                            vb[kk] = c == 0 ? db : __fadd2_rn(vb[kk], db);
                            vc[kk] = c == 0 ? dc : __fadd2_rn(vc[kk], dc);
                            carry[c][kk] = __fmul2_rn(a, dh);
                        }
                        p1v[c][r] = p1.x + p1.y;
                        p2v[c][r] = p2.x + p2.y;
                        if constexpr (EXT) p3v[c][r] = p3.x + p3.y;
                    }
                    float vals[C::V];
#pragma unroll
                    for (int kk = 0; kk < NP; ++kk) {
                        vals[2 * kk] = vb[kk].x;
                        vals[2 * kk + 1] = vb[kk].y;
                        vals[NPE + 2 * kk] = vc[kk].x;
                        vals[NPE + 2 * kk + 1] = vc[kk].y;
                    }
                    reduce_bc_store<C::V, CPW, N, NPT, NPE>(vals, q, g, redw + tb * 2 * N);
                }
                // lane g finishes step rb*R + g of the block for each of its channels
                const int tl = t0b + rb * R + g;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    const float P1s = transpose_reduce<R, CPW>(p1v[c], g) * kLn2;  // sum dh h Abar A
                    // sum dh B (Euler), sum dh Abar B (zero-order hold)
                    const float P2s = transpose_reduce<R, CPW>(p2v[c], g);
                    const float4 pp = P0[c][tl];
                    const float2 q1 = P1[c][tl];
                    const float ddelta = fmaf(P2s, q1.x, P1s) * pp.w;
                    dD_acc[c] = fmaf(pp.z, q1.x, dD_acc[c]);
                    dbias_acc[c] += ddelta;
                    IO *ob = reinterpret_cast<IO *>(smem + C::OFF_OB + chs[c] * C::OBROW);
                    float du_in = pp.x * P2s;  // sum_n dh Delta' B
                    if constexpr (EXT) {
                        const float P3s = transpose_reduce<R, CPW>(p3v[c], g);  // sum_n dh psi B
                        if (zoh) du_in = P3s;
                    }
                    const float du = fmaf(pp.z, Dd[c], du_in);
                    if (MULTI || (EXT && p.du_acc)) {
                        // this direction's du by scan step, in fp32: the merge sums by
                        // position (multi-direction), or the fused Conv1D's backward
                        // reads it (single direction)
                        const int64_t t = (int64_t)i * T + tl;
                        if (valid[c] && t < L)
                            p.du_acc[kdir * p.du_zstride + ((int64_t)b * p.dim + dch[c]) * L + t] = du;
                    } else {
                        ob[tl] = IOT<IO>::from_f(du);
                    }
                    ob[C::CB * C::OBROW / C::ES + tl] = IOT<IO>::from_f(ddelta);
                    if (!MULTI && p.has_z)                                          // dz
                        ob[2 * C::CB * C::OBROW / C::ES + tl] =
                            IOT<IO>::from_f(fmaf(Dd[c], q1.x, sv[c][rb]) * q1.y);
                }
            }

            // dB, dC of the block: sum the warps' terms, add to the outputs
            __syncthreads();
            {
                const float *rb_all = red0;
#pragma unroll 1
                for (int gi = tid; gi < 2 * N * (TS / 4); gi += C::THREADS) {
                    const int n = gi % N;
                    const int arr = (gi / N) & 1;
                    const int t4 = gi / (2 * N);
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int w = 0; w < C::W; ++w) {
                        const float *src = rb_all + (w * TS + 4 * t4) * 2 * N + arr * N + n;
                        acc.x += src[0];
                        acc.y += src[2 * N];
                        acc.z += src[4 * N];
                        acc.w += src[6 * N];
                    }
                    const int64_t t = (int64_t)k * TS + 4 * t4;
                    float *dBC = arr ? p.dC : p.dB;
                    if (t < L)
                        atomicAdd(reinterpret_cast<float4 *>(
                                      dBC + ((((int64_t)b * Kd + kdir) * p.G + grp) * N + n) * L + t),
                                  acc);
                }
            }
            __syncthreads();  // the sums buffer is refilled by the next block
        }

        // the tile's du, ddelta (and dz) rows: 16-byte stores of this warp's channels
        __syncwarp();
        {
            constexpr int VPC = 16 / C::ES;
            // single direction: du, ddelta (and dz); multi-direction: ddelta only
            const int narr = MULTI ? 1 : (p.has_z ? 3 : 2);
#pragma unroll 1
            for (int kk = lane; kk < narr * C::CHW * 4; kk += 32) {
                const int arr = MULTI ? 1 : kk / (C::CHW * 4);
                if (EXT && arr == 0 && p.du_acc) continue;  // du went out in fp32
                const int rem = kk % (C::CHW * 4);
                const int rr = rem >> 2, qq = rem & 3;
                const int chr = warp * C::CHW + rr;
                const int dgr = cblk * C::CB + chr;
                const int64_t t = (int64_t)i * T + qq * VPC;
                if (dgr < p.dpg && t < L) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        smem + C::OFF_OB + (arr * C::CB + chr) * C::OBROW + qq * 16);
                    void *base = arr == 0 ? p.du : (arr == 1 ? p.ddelta : p.dz);
                    const int64_t orow = (arr == 1 ? dlrow0 : row0) + dgr;  // ddelta: direction k's row
                    *reinterpret_cast<uint4 *>(reinterpret_cast<IO *>(base) + orow * L + t) = v;
                }
            }
        }
        __syncwarp();
    }

    // the gradient with respect to the initial state: Abar_0 (.) dh_0, the carry
    // left by the first step
    if (EXT && p.dh0) {
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            if (!valid[c]) continue;
            float *dst = p.dh0 + ((int64_t)b * p.dim + dch[c]) * N + g * NPT;
#pragma unroll
            for (int kk = 0; kk < NP; ++kk) {
                dst[2 * kk] = carry[c][kk].x;
                if (2 * kk + 1 < NPT) dst[2 * kk + 1] = carry[c][kk].y;
            }
        }
    }

    // per-channel sums: over the channel's R lanes, then over the batch (atomics)
#pragma unroll
    for (int c = 0; c < CL; ++c) {
#pragma unroll
        for (int m = 1; m < R; m <<= 1) {
            dD_acc[c] += __shfl_xor_sync(kFull, dD_acc[c], m * CPW);
            dbias_acc[c] += __shfl_xor_sync(kFull, dbias_acc[c], m * CPW);
        }
        if (!valid[c]) continue;
#pragma unroll
        for (int kk = 0; kk < NP; ++kk) {
            atomicAdd(p.dA + (poff + dch[c]) * N + g * NPT + 2 * kk, dA[c][kk].x);
            if (2 * kk + 1 < NPT) atomicAdd(p.dA + (poff + dch[c]) * N + g * NPT + 2 * kk + 1, dA[c][kk].y);
        }
        if (g == 0) {
            if (p.dD) atomicAdd(p.dD + poff + dch[c], dD_acc[c]);
            if (p.dbias) atomicAdd(p.dbias + poff + dch[c], dbias_acc[c]);
        }
    }
}

// Transposes each [H, W] plane of src [rows, H, W] into dst [rows, W, H], so that
// a column-order direction can read its inputs as tiles of a row order.  32 x 32
// tiles through shared memory; grid (rows, ceil(H/32), ceil(W/32)).
template <typename IO>
__global__ void __launch_bounds__(256) k_transpose_maps(const IO *__restrict__ src, IO *__restrict__ dst,
                                                        int H, int W) {
    __shared__ IO tile[32][33];
    const int64_t row = blockIdx.x;
    const int64_t L = (int64_t)H * W;
    const int r0 = blockIdx.y * 32, c0 = blockIdx.z * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const IO *s = src + row * L;
    IO *d = dst + row * L;
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int r = r0 + ty + k, c = c0 + tx;
        if (r < H && c < W) tile[ty + k][tx] = s[(int64_t)r * W + c];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int c = c0 + ty + k, r = r0 + tx;
        if (r < H && c < W) d[(int64_t)c * H + r] = tile[tx][ty + k];
    }
}

// k_transpose_maps for planes that fit in shared memory whole, H a multiple of
// the V = 16 / sizeof(IO) elements of a 16-byte vector, and 16-byte aligned
// planes.  One CTA per plane copies it into shared memory as 16-byte vectors
// (all of a thread's loads issued before its stores), then each thread gathers
// V consecutive rows of one column and writes them as one 16-byte vector of the
// [W, H] plane; consecutive lanes take consecutive columns, so a warp's
// shared-memory reads are consecutive.  Dynamic shared memory: H * W elements.
template <typename IO>
__global__ void __launch_bounds__(256) k_transpose_planes(const IO *__restrict__ src, IO *__restrict__ dst,
                                                          int H, int W) {
    using R = typename std::conditional<sizeof(IO) == 2, unsigned short, unsigned int>::type;
    constexpr int V = 16 / (int)sizeof(IO);
    constexpr int U = 4;
    extern __shared__ uint4 plane_v[];
    const R *plane = reinterpret_cast<const R *>(plane_v);
    const int t = threadIdx.x;
    const int L = H * W;
    const int nv = L / V;
    const uint4 *s = reinterpret_cast<const uint4 *>(src + blockIdx.x * (int64_t)L);
    for (int i0 = t; i0 < nv; i0 += U * 256) {
        uint4 v[U];
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (i0 + j * 256 < nv) v[j] = __ldg(s + i0 + j * 256);
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (i0 + j * 256 < nv) plane_v[i0 + j * 256] = v[j];
    }
    __syncthreads();
    uint4 *d = reinterpret_cast<uint4 *>(dst + blockIdx.x * (int64_t)L);
    const int nb = H / V;  // 16-byte vectors in a row of the [W, H] plane
    for (int k = t; k < nv; k += 256) {
        const int rb = k / W, c = k - rb * W;  // column c, rows rb*V .. rb*V + V - 1
        union {
            uint4 v;
            R e[V];
        } o;
#pragma unroll
        for (int j = 0; j < V; ++j) o.e[j] = plane[(rb * V + j) * W + c];
        d[c * nb + rb] = o.v;
    }
}

// Merge of a multi-direction backward pass: du[p] = sum_k du_k[step_k(p)] (each
// direction's du was stored by scan step) and, with a gate, dz[p] = dout[p] *
// s[p] * SiLU'(z[p]), s being the sum of all directions' pre-gate outputs.  A
// thread owns one position (the traversals are the same for every row) and
// walks rows blockIdx.y, blockIdx.y + gridDim.y, ...
struct BwdOrderSet {
    int K, H, W, win;
    int orders[8];
};
template <typename IO>
__global__ void __launch_bounds__(256)
k_merge_bwd(const float *__restrict__ du_acc, int64_t rows, const BwdOrderSet os,
            const IO *__restrict__ dout, const IO *__restrict__ z, const IO *__restrict__ s,
            IO *__restrict__ du, IO *__restrict__ dz) {
    const int64_t L = (int64_t)os.H * os.W;
    const int pos = blockIdx.x * blockDim.x + threadIdx.x;
    if (pos >= L) return;
    const int r = pos / os.W, c = pos - r * os.W;
    uint32_t st[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) st[k] = k < os.K ? step_of(os.orders[k], r, c, os.H, os.W, os.win) : 0u;
    for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
        float g = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < os.K) g += du_acc[((int64_t)k * rows + row) * L + st[k]];
        const int64_t i = row * L + pos;
        du[i] = IOT<IO>::from_f(g);
        if (z) {
            const float zz = IOT<IO>::load(z + i);
            const float sg = rcp(1.f + ex2(-zz * kLog2e));
            dz[i] = IOT<IO>::from_f(IOT<IO>::load(dout + i) * IOT<IO>::load(s + i) * sg *
                                    fmaf(zz, 1.f - sg, 1.f));
        }
    }
}

}  // namespace ssk

namespace ssk {

// The Mamba block's Conv1D + SiLU input branch (causal depthwise convolution
// of width 4 with bias, then SiLU) as passes of their own, for the backward
// pass of a scan that fused it in front: k_conv_silu_fwd recomputes the scan's
// input u, and k_conv_silu_bwd turns the scan's du into the gradients of the
// convolution's input x, weights, bias and history x0.
//   v_t = b + sum_{j<4} w_j x_{t-3+j}   (x_s for s < 0 is x0[3+s], or 0)
//   u_t = SiLU(v_t)
//   dv_t = du_t SiLU'(v_t),  SiLU'(v) = sigmoid(v) (1 + v (1 - sigmoid(v)))
//   dx_s = sum_j w_j dv_{s+3-j},  dx0_k = sum_{j<=k} w_j dv_{k-j}
//   dw_j = sum_t dv_t x_{t-3+j},  db = sum_t dv_t      (over batch and time)
struct ConvSiluParams {
    int64_t rows, dim, L;
    const void *x;
    const float *w, *bias, *x0;  // [dim, 4], [dim] (nullable), [rows, 3] (nullable)
    void *u;                     // k_conv_silu_fwd: [rows, L] (I/O type)
    const float *du;             // k_conv_silu_bwd: [rows, L] fp32 (the scan's du)
    void *dx;                    // [rows, L] (I/O type)
    float *dw, *dbias, *dx0;     // [dim, 4] and [dim] summed with atomics; [rows, 3]
};

template <typename IO>
__device__ __forceinline__ float conv_x(const ConvSiluParams &p, int64_t row, int64_t s) {
    if (s >= 0) return IOT<IO>::load(reinterpret_cast<const IO *>(p.x) + row * p.L + s);
    return p.x0 ? __ldg(p.x0 + row * 3 + 3 + s) : 0.f;
}

template <typename IO>
__device__ __forceinline__ float conv_pre(const ConvSiluParams &p, int64_t row, int64_t t, const float4 &w,
                                          float b) {
    return fmaf(w.w, conv_x<IO>(p, row, t),
                fmaf(w.z, conv_x<IO>(p, row, t - 1), fmaf(w.y, conv_x<IO>(p, row, t - 2),
                                                          fmaf(w.x, conv_x<IO>(p, row, t - 3), b))));
}

// One thread per element, grid-stride over [rows, L].
template <typename IO>
__global__ void __launch_bounds__(256) k_conv_silu_fwd(const ConvSiluParams p) {
    const int64_t n = p.rows * p.L;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / p.L, t = i - row * p.L;
        const int64_t d = row % p.dim;
        const float4 w = __ldg(reinterpret_cast<const float4 *>(p.w) + d);
        const float b = p.bias ? __ldg(p.bias + d) : 0.f;
        reinterpret_cast<IO *>(p.u)[i] = IOT<IO>::from_f(silu(conv_pre<IO>(p, row, t, w, b)));
    }
}

// One block of CONV_TS threads per (row, tile of CONV_TS steps): dv of the
// tile's steps and of the three after it (the taps reaching back into the
// tile) go to shared memory; each thread then forms dx of its step and its
// partial dw and db, which the block sums and adds with atomics.
constexpr int CONV_TS = 256;
template <typename IO>
__global__ void __launch_bounds__(CONV_TS) k_conv_silu_bwd(const ConvSiluParams p) {
    __shared__ float dv[CONV_TS + 3];
    __shared__ float red[5][CONV_TS / 32];
    const int64_t row = blockIdx.y;
    const int64_t d = row % p.dim;
    const int64_t t0 = (int64_t)blockIdx.x * CONV_TS;
    const float4 w = __ldg(reinterpret_cast<const float4 *>(p.w) + d);
    const float b = p.bias ? __ldg(p.bias + d) : 0.f;
    const float *dur = p.du + row * p.L;
    for (int k = threadIdx.x; k < CONV_TS + 3; k += CONV_TS) {
        const int64_t t = t0 + k;
        float g = 0.f;
        if (t < p.L) {
            const float v = conv_pre<IO>(p, row, t, w, b);
            const float sg = rcp(1.f + ex2(-v * kLog2e));
            g = __ldg(dur + t) * sg * fmaf(v, 1.f - sg, 1.f);
        }
        dv[k] = g;
    }
    __syncthreads();
    const int k = threadIdx.x;
    const int64_t t = t0 + k;
    float pw[4] = {0.f, 0.f, 0.f, 0.f}, pb = 0.f;
    if (t < p.L) {
        // dx_t = w_0 dv_{t+3} + w_1 dv_{t+2} + w_2 dv_{t+1} + w_3 dv_t
        const float dxt = fmaf(w.x, dv[k + 3], fmaf(w.y, dv[k + 2], fmaf(w.z, dv[k + 1], w.w * dv[k])));
        reinterpret_cast<IO *>(p.dx)[row * p.L + t] = IOT<IO>::from_f(dxt);
        const float g = dv[k];
        pw[0] = g * conv_x<IO>(p, row, t - 3);
        pw[1] = g * conv_x<IO>(p, row, t - 2);
        pw[2] = g * conv_x<IO>(p, row, t - 1);
        pw[3] = g * conv_x<IO>(p, row, t);
        pb = g;
    }
    if (t0 == 0 && p.dx0 && k < 3) {
        // the history: dx0_k = sum_{j <= k} w_j dv_{k-j}
        const float wj[4] = {w.x, w.y, w.z, w.w};
        float acc = 0.f;
        for (int j = 0; j <= k; ++j) acc = fmaf(wj[j], dv[k - j], acc);
        p.dx0[row * 3 + k] = acc;
    }
    // block sums of dw and db
    float vals[5] = {pw[0], pw[1], pw[2], pw[3], pb};
#pragma unroll
    for (int i = 0; i < 5; ++i) {
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) vals[i] += __shfl_xor_sync(kFull, vals[i], m);
        if ((threadIdx.x & 31) == 0) red[i][threadIdx.x >> 5] = vals[i];
    }
    __syncthreads();
    if (threadIdx.x < 5) {
        float s = 0.f;
        for (int i = 0; i < CONV_TS / 32; ++i) s += red[threadIdx.x][i];
        if (threadIdx.x < 4) atomicAdd(p.dw + d * 4 + threadIdx.x, s);
        else if (p.dbias) atomicAdd(p.dbias + d, s);
    }
}

}  // namespace ssk
