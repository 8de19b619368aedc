// Backward pass of the single-direction selective scan (sm_103a).
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
// Work split as in the forward scan: a CTA owns CB channels of one (batch,
// group); lane = g*CPW + c holds NPT of the N states of channel c of its warp.
// Each CTA walks its rows twice through one TMA ring:
//   pass F, tiles 0 .. nt-1: the states only, storing them every TS = 16 steps
//     as checkpoints (fp32, N values per channel per 16 steps: 4 bytes per
//     element at N = 16);
//   pass B, tiles nt-1 .. 0, each tile's 16-step blocks last to first: from
//     the block's checkpoint the lane recomputes its chains' 16 states into
//     registers together with the readout s_t, then runs the reverse
//     recurrence over the block; Abar (.) dh is carried in registers from block
//     to block.
// Sums over the N states (s_t, dDelta'_t, sum_n dh B) are combined across a
// channel's R lanes by the transposing butterfly, R steps at a time, so that
// lane g finishes step g of each R-step group.  dB and dC are sums over the
// channels of a group: per step a transposing butterfly over the CPW lanes of
// a state slice, then per-warp sums in shared memory that the CTA adds up after
// each block and adds to the fp32 outputs with 16-byte atomic adds.  dA, dD and
// dbias are per-channel sums over time held in registers, added over the batch
// with atomics at the end.
#pragma once

#include "ss_device.cuh"

namespace ssk {

template <typename IO_, int N_, int W_, int STAGES_ = 3>
struct CfgB {
    using IO = IO_;
    static constexpr int N = N_, W = W_, STAGES = STAGES_;
    static constexpr int NPT = N < 4 ? N : 4;  // states per lane
    static constexpr int R = N / NPT;          // lanes per channel
    static constexpr int CPW = 32 / R;         // channels per warp
    static constexpr int CB = W * CPW;         // channels per CTA
    static constexpr int THREADS = 32 * W;
    static constexpr int ES = sizeof(IO);
    static constexpr int T = 64 / ES;          // steps per tile (64-byte raw rows)
    static constexpr int TS = 16;              // steps per register block = checkpoint interval
    static constexpr int NS = T / TS;          // register blocks per tile
    static constexpr int RB = TS / R;          // R-step readout groups per block
    static constexpr int E = T / R;            // steps one thread preps (R threads per channel)
    static constexpr int EP = E < 8 ? E : 8;   // steps converted at a time
    static constexpr int V = 2 * NPT;          // dB and dC terms of a lane per step
    static_assert(N % NPT == 0 && (R & (R - 1)) == 0 && R <= TS && TS % R == 0, "lane split");
    static_assert(T % TS == 0 && E % EP == 0 && EP * ES >= 4, "tile split");
    static_assert(CB <= 256 && N <= 256, "TMA box rows");

    static constexpr int al(int x) { return (x + 1023) & ~1023; }
    static constexpr int TILE_CH = al(CB * 64);
    static constexpr int TILE_BC = al(N * 64);
    static constexpr int STAGE = 4 * TILE_CH + 2 * TILE_BC;
    static constexpr int OFF_U = 0, OFF_DL = TILE_CH, OFF_Z = 2 * TILE_CH, OFF_DY = 3 * TILE_CH;
    static constexpr int OFF_B = 4 * TILE_CH, OFF_C = 4 * TILE_CH + TILE_BC;
    static constexpr int BCF = T * 2 * N * 4;       // fp32 B, C of a tile: [t][B_0..N-1 | C_0..N-1]
    static constexpr int OFF_BCF = STAGES * STAGE;  // two tiles' worth (tile parity)
    static constexpr int P0ROW = (T + 1) * 16;      // per step {Delta', Delta'u, ds, softplus'}
    static constexpr int P1ROW = (T + 2) * 8;       // per step {u, dout SiLU'(z)}
    static constexpr int OFF_P0 = OFF_BCF + 2 * BCF;
    static constexpr int OFF_P1 = OFF_P0 + CB * P0ROW;
    static constexpr int OBROW = 64 + 16;           // staged du / ddelta / dz rows (I/O type)
    static constexpr int OFF_OB = OFF_P1 + CB * P1ROW;
    static constexpr int REDW = TS * 2 * N * 4;     // one warp's dB/dC sums over one block
    static constexpr int OFF_RED = OFF_OB + 3 * CB * OBROW;
    static constexpr int OFF_BAR = (OFF_RED + 2 * W * REDW + 7) & ~7;
    static constexpr int SMEM = OFF_BAR + 8 * STAGES + 1024;  // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

struct BwdParams {
    int64_t dim, L;
    int G, dpg;
    int nblk;                 // 16-step blocks per row
    const float *A, *D, *bias;
    int softplus, has_z;
    float *ckpt;              // [batch*dim, nblk, N]: state after each block (pass F)
    void *du, *ddelta, *dz;   // [batch, dim, L], I/O type
    float *dA;                // [dim, N]
    float *dB, *dC;           // [batch, G, N, L]
    float *dD, *dbias;        // [dim], nullable
};

template <int NPT>
__device__ __forceinline__ void lds_npt(const float *p, float (&v)[NPT]) {
    if constexpr (NPT == 4) {
        const float4 q = *reinterpret_cast<const float4 *>(p);
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    } else {
#pragma unroll
        for (int j = 0; j < NPT; ++j) v[j] = p[j];
    }
}

__device__ __forceinline__ float sigmoid(float x) { return rcp(1.0f + ex2(-x * kLog2e)); }

// Sums the V dB/dC terms of one step over the P channel lanes of a state slice
// (lanes g*P + c, c = 0..P-1) and writes the sums to dst = [dB_0..N-1 | dC_0..N-1]
// of that step.  Term vi of a lane is dB of state g*NPT + vi for vi < NPT and
// dC of state g*NPT + vi - NPT otherwise.
template <int V, int P, int N, int NPT>
__device__ __forceinline__ void reduce_bc_store(float (&v)[V], int c, int g, float *dst) {
    auto slot = [&](int vi) { return (vi < NPT ? 0 : N) + g * NPT + (vi % NPT); };
    if constexpr (P == 1) {
#pragma unroll
        for (int vi = 0; vi < V; ++vi) dst[slot(vi)] = v[vi];
    } else if constexpr (V >= P) {
#pragma unroll
        for (int m = 0; m < V / P; ++m) {
            float part[P];
#pragma unroll
            for (int k = 0; k < P; ++k) part[k] = v[m * P + k];
            const float r = transpose_reduce<P, 1>(part, c);
            dst[slot(m * P + c)] = r;
        }
    } else {
        float r = transpose_reduce<V, 1>(v, c & (V - 1));
#pragma unroll
        for (int m = V; m < P; m <<= 1) r += __shfl_xor_sync(kFull, r, m);
        if (c < V) dst[slot(c)] = r;
    }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS)
k_scan_bwd(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
           const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_dy,
           const __grid_constant__ CUtensorMap tm_B, const __grid_constant__ CUtensorMap tm_C,
           const BwdParams p) {
    using IO = typename C::IO;
    constexpr int N = C::N, NPT = C::NPT, R = C::R, CPW = C::CPW, T = C::T, TS = C::TS;
    constexpr int E = C::E, EP = C::EP, STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = lane % CPW, g = lane / CPW;
    const int cblk = blockIdx.x, bg = blockIdx.y;
    const int b = bg / p.G, grp = bg % p.G;
    const int64_t L = p.L;
    const int64_t row0 = (int64_t)b * p.dim + (int64_t)grp * p.dpg;  // the group's channel 0
    const int row_tma = (int)(row0 + (int64_t)cblk * C::CB);
    const int bcrow_tma = (int)(((int64_t)b * p.G + grp) * N);
    const int nt = (int)((L + T - 1) / T);
    const int nq = 2 * nt;  // ring order: pass F tiles 0..nt-1, then pass B tiles nt-1..0

    // scan role: NPT states of channel ch
    const int ch = warp * CPW + c;
    const int dg = cblk * C::CB + ch;
    const bool valid = dg < p.dpg;
    const int64_t d = (int64_t)grp * p.dpg + (valid ? dg : p.dpg - 1);
    const int64_t row = (int64_t)b * p.dim + d;
    float A2[NPT], h[NPT], carry[NPT], dA[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        A2[j] = __ldg(p.A + d * N + g * NPT + j) * kLog2e;
        h[j] = 0.f;
        carry[j] = 0.f;
        dA[j] = 0.f;
    }
    const float Dd = p.D ? __ldg(p.D + d) : 0.f;
    float dD_acc = 0.f, dbias_acc = 0.f;
    float *ck = p.ckpt + row * p.nblk * N + g * NPT;  // this lane's checkpoint slots
    const float4 *P0 = reinterpret_cast<const float4 *>(smem + C::OFF_P0 + ch * C::P0ROW);
    const float2 *P1 = reinterpret_cast<const float2 *>(smem + C::OFF_P1 + ch * C::P1ROW);
    IO *ob0 = reinterpret_cast<IO *>(smem + C::OFF_OB + ch * C::OBROW);
    IO *ob1 = reinterpret_cast<IO *>(smem + C::OFF_OB + (C::CB + ch) * C::OBROW);
    IO *ob2 = reinterpret_cast<IO *>(smem + C::OFF_OB + (2 * C::CB + ch) * C::OBROW);
    float *red0 = reinterpret_cast<float *>(smem + C::OFF_RED);
    float *bcf0 = reinterpret_cast<float *>(smem + C::OFF_BCF);

    // prep role: E consecutive steps of channel pch (a channel of this warp)
    const int pch = tid / R;
    const int pt0 = (tid % R) * E;
    const int pdg = cblk * C::CB + pch;
    const bool pvalid = pdg < p.dpg;
    const int64_t pd = (int64_t)grp * p.dpg + (pvalid ? pdg : p.dpg - 1);
    const float pbias = p.bias ? __ldg(p.bias + pd) : 0.f;
    float4 *q0row = reinterpret_cast<float4 *>(smem + C::OFF_P0 + pch * C::P0ROW);
    float2 *q1row = reinterpret_cast<float2 *>(smem + C::OFF_P1 + pch * C::P1ROW);

    const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t txF = 2u * C::CB * 64u + N * 64u;
    const uint32_t txB = (3u + (p.has_z ? 1u : 0u)) * C::CB * 64u + 2u * N * 64u;
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
    __syncthreads();

    // diagnostics: this CTA leaves its first tile's barrier without arrivals
    const bool skip_first = (g_debug_flags & 1u) && blockIdx.x == 0 && blockIdx.y == 0;
    auto tile_of = [&](int q) { return q < nt ? q : nq - 1 - q; };
    auto issue = [&](int q) {
        if (q == 0 && skip_first) return;
        const int s = q % STAGES;
        const uint32_t bar = bar0 + 8 * s;
        const uint32_t st = smem0 + s * C::STAGE;
        const bool bwd = q >= nt;
        const int x = tile_of(q) * T;
        mbar_expect_tx(bar, bwd ? txB : txF);
        tma_load_2d(st + C::OFF_U, &tm_u, x, row_tma, bar);
        tma_load_2d(st + C::OFF_DL, &tm_dl, x, row_tma, bar);
        tma_load_2d(st + C::OFF_B, &tm_B, x, bcrow_tma, bar);
        if (bwd) {
            tma_load_2d(st + C::OFF_DY, &tm_dy, x, row_tma, bar);
            if (p.has_z) tma_load_2d(st + C::OFF_Z, &tm_z, x, row_tma, bar);
            tma_load_2d(st + C::OFF_C, &tm_C, x, bcrow_tma, bar);
        }
    };
    if (tid == 0) {
#pragma unroll 1
        for (int q = 0; q < STAGES && q < nq; ++q) issue(q);
    }

    // Converts ring item q (tile i) into fp32 B (and C) and per-step rows.
    auto prep = [&](int q, int i, bool bwd) {
        const uint8_t *st = smem + (q % STAGES) * C::STAGE;
        float *bcf = bcf0 + (q & 1) * (C::BCF / 4);
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
            for (int e = 0; e < VPC; ++e) bcf[(qq * VPC + e) * 2 * N + arr * N + n] = v[e];
        }
        const int64_t tb0 = (int64_t)i * T;
#pragma unroll
        for (int e0 = 0; e0 < E; e0 += EP) {
            float uu[EP], dd[EP], zz[EP], gy[EP];
            load_tile_row<IO, EP>(st + C::OFF_U, pch, pt0 + e0, uu);
            load_tile_row<IO, EP>(st + C::OFF_DL, pch, pt0 + e0, dd);
            if (bwd) {
                load_tile_row<IO, EP>(st + C::OFF_DY, pch, pt0 + e0, gy);
                if (p.has_z) load_tile_row<IO, EP>(st + C::OFF_Z, pch, pt0 + e0, zz);
            }
#pragma unroll
            for (int e = 0; e < EP; ++e) {
                const int tl = pt0 + e0 + e;
                // steps past the sequence end and channels past the group leave h
                // unchanged and contribute nothing
                const bool in = pvalid && tb0 + tl < L;
                const float v = dd[e] + pbias;
                const float dl = in ? (p.softplus ? softplus(v) : v) : 0.f;
                const float x = dl * uu[e];
                if (!bwd) {
                    *reinterpret_cast<float2 *>(q0row + tl) = make_float2(dl, x);
                } else {
                    const float dsp = p.softplus ? sigmoid(v) : 1.f;
                    float ds = gy[e], dzf = 0.f;
                    if (p.has_z) {
                        const float sg = sigmoid(zz[e]);
                        ds = gy[e] * zz[e] * sg;
                        dzf = gy[e] * sg * fmaf(zz[e], 1.f - sg, 1.f);
                    }
                    q0row[tl] = make_float4(dl, x, in ? ds : 0.f, dsp);
                    q1row[tl] = make_float2(uu[e], dzf);
                }
            }
        }
    };
    // Bounded wait for ring item q; on timeout the whole CTA drains its copies
    // and exits (returns true then).
    auto abandon = [&](int q, bool ok) -> bool {
        if (!__syncthreads_or(!ok)) return false;
        if (tid == 0) {
            report_timeout();
#pragma unroll 1
            for (int k = q; k < nq && k < q + STAGES; ++k)
                if (!(k == 0 && skip_first))
                    (void)mbar_wait_bounded(bar0 + 8 * (k % STAGES), (k / STAGES) & 1, 1000000000ull);
        }
        return true;
    };

#pragma unroll 1
    for (int q = 0; q < nq; ++q) {
        const bool bwd = q >= nt;
        const int i = tile_of(q);
        const bool ok = mbar_wait_bounded(bar0 + 8 * (q % STAGES), (q / STAGES) & 1, budget);
        if (ok) prep(q, i, bwd);
        if (abandon(q, ok)) return;
        if (tid == 0 && q + STAGES < nq) {
            fence_proxy_async_smem();
            issue(q + STAGES);
        }
        const float *bcf = bcf0 + (q & 1) * (C::BCF / 4);

        if (!bwd) {
            // ---------------- pass F: checkpoints after each block
#pragma unroll 1
            for (int s = 0; s < C::NS; ++s) {
                const int k = i * C::NS + s;
                if (k >= p.nblk - 1) break;  // no later block starts from this state
#pragma unroll
                for (int tb = 0; tb < TS; ++tb) {
                    const float2 pp = *reinterpret_cast<const float2 *>(P0 + s * TS + tb);
                    float Bv[NPT];
                    lds_npt<NPT>(bcf + (s * TS + tb) * 2 * N + g * NPT, Bv);
#pragma unroll
                    for (int j = 0; j < NPT; ++j) h[j] = fmaf(ex2(pp.x * A2[j]), h[j], pp.y * Bv[j]);
                }
                if (valid) {
#pragma unroll
                    for (int j = 0; j < NPT; ++j) ck[(int64_t)k * N + j] = h[j];
                }
            }
            __syncwarp();
            continue;
        }

        // ---------------- pass B: blocks of tile i, last to first
#pragma unroll 1
        for (int s = C::NS - 1; s >= 0; --s) {
            const int k = i * C::NS + s;
            if (k >= p.nblk) continue;  // the block lies past the sequence end
            const int t0b = s * TS;
            float hb[NPT];
#pragma unroll
            for (int j = 0; j < NPT; ++j) hb[j] = k > 0 ? ck[(int64_t)(k - 1) * N + j] : 0.f;

            // recompute the block's states and readouts
            float hs[TS][NPT];
            float sv[C::RB];
            {
                float hc[NPT];
#pragma unroll
                for (int j = 0; j < NPT; ++j) hc[j] = hb[j];
#pragma unroll
                for (int rb = 0; rb < C::RB; ++rb) {
                    float sp[R];
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const int tb = rb * R + r;
                        const float4 pp = P0[t0b + tb];
                        float Bv[NPT], Cv[NPT];
                        lds_npt<NPT>(bcf + (t0b + tb) * 2 * N + g * NPT, Bv);
                        lds_npt<NPT>(bcf + (t0b + tb) * 2 * N + N + g * NPT, Cv);
                        float acc = 0.f;
#pragma unroll
                        for (int j = 0; j < NPT; ++j) {
                            hc[j] = fmaf(ex2(pp.x * A2[j]), hc[j], pp.y * Bv[j]);
                            hs[tb][j] = hc[j];
                            acc = fmaf(Cv[j], hc[j], acc);
                        }
                        sp[r] = acc;
                    }
                    sv[rb] = transpose_reduce<R, CPW>(sp, g);
                }
            }

            // reverse recurrence over the block
            float *redw = red0 + ((k & 1) * C::W + warp) * (TS * 2 * N);
#pragma unroll
            for (int rb = C::RB - 1; rb >= 0; --rb) {
                float p1v[R], p2v[R];
#pragma unroll
                for (int r = R - 1; r >= 0; --r) {
                    const int tb = rb * R + r;
                    const float4 pp = P0[t0b + tb];  // Delta', Delta'u, ds, softplus'
                    float Bv[NPT], Cv[NPT];
                    lds_npt<NPT>(bcf + (t0b + tb) * 2 * N + g * NPT, Bv);
                    lds_npt<NPT>(bcf + (t0b + tb) * 2 * N + N + g * NPT, Cv);
                    float vals[C::V];
                    float p1 = 0.f, p2 = 0.f;
#pragma unroll
                    for (int j = 0; j < NPT; ++j) {
                        const float a = ex2(pp.x * A2[j]);
                        const float dh = fmaf(pp.z, Cv[j], carry[j]);
                        const float hp = tb > 0 ? hs[tb - 1][j] : hb[j];
                        const float w = dh * hp * a;
                        p1 = fmaf(w, A2[j], p1);
                        dA[j] = fmaf(w, pp.x, dA[j]);
                        p2 = fmaf(dh, Bv[j], p2);
                        vals[j] = dh * pp.y;
                        vals[NPT + j] = pp.z * hs[tb][j];
                        carry[j] = a * dh;
                    }
                    p1v[r] = p1;
                    p2v[r] = p2;
                    reduce_bc_store<C::V, CPW, N, NPT>(vals, c, g, redw + tb * 2 * N);
                }
                // lane g finishes step rb*R + g of the block
                const float P1s = transpose_reduce<R, CPW>(p1v, g) * kLn2;  // sum dh h Abar A
                const float P2s = transpose_reduce<R, CPW>(p2v, g);         // sum dh B
                const int tl = t0b + rb * R + g;
                const float4 pp = P0[tl];
                const float2 q1 = P1[tl];
                const float ddl = fmaf(P2s, q1.x, P1s);
                const float ddelta = ddl * pp.w;
                const float du = fmaf(pp.z, Dd, pp.x * P2s);
                dD_acc = fmaf(pp.z, q1.x, dD_acc);
                dbias_acc += ddelta;
                ob0[tl] = IOT<IO>::from_f(du);
                ob1[tl] = IOT<IO>::from_f(ddelta);
                if (p.has_z) ob2[tl] = IOT<IO>::from_f(fmaf(Dd, q1.x, sv[rb]) * q1.y);
            }

            // dB, dC of the block: sum the warps' terms, add to the outputs
            __syncthreads();
            {
                const float *rb_all = red0 + (k & 1) * C::W * (TS * 2 * N);
                float *dBC = nullptr;
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
                    dBC = arr ? p.dC : p.dB;
                    if (t < L)
                        atomicAdd(reinterpret_cast<float4 *>(dBC + (((int64_t)b * p.G + grp) * N + n) * L + t),
                                  acc);
                }
            }
        }

        // the tile's du, ddelta (and dz) rows: 16-byte stores of this warp's channels
        __syncwarp();
        {
            constexpr int VPC = 16 / C::ES;
            const int narr = p.has_z ? 3 : 2;
#pragma unroll 1
            for (int kk = lane; kk < narr * CPW * 4; kk += 32) {
                const int arr = kk / (CPW * 4);
                const int rem = kk % (CPW * 4);
                const int rr = rem >> 2, qq = rem & 3;
                const int chr = warp * CPW + rr;
                const int dgr = cblk * C::CB + chr;
                const int64_t t = (int64_t)i * T + qq * VPC;
                if (dgr < p.dpg && t < L) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(
                        smem + C::OFF_OB + (arr * C::CB + chr) * C::OBROW + qq * 16);
                    void *base = arr == 0 ? p.du : (arr == 1 ? p.ddelta : p.dz);
                    *reinterpret_cast<uint4 *>(reinterpret_cast<IO *>(base) + (row0 + dgr) * L + t) = v;
                }
            }
        }
        __syncwarp();
    }

    // per-channel sums: over the channel's R lanes, then over the batch (atomics)
#pragma unroll
    for (int m = 1; m < R; m <<= 1) {
        dD_acc += __shfl_xor_sync(kFull, dD_acc, m * CPW);
        dbias_acc += __shfl_xor_sync(kFull, dbias_acc, m * CPW);
    }
    if (valid) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) atomicAdd(p.dA + d * N + g * NPT + j, dA[j]);
        if (g == 0) {
            if (p.dD) atomicAdd(p.dD + d, dD_acc);
            if (p.dbias) atomicAdd(p.dbias + d, dbias_acc);
        }
    }
}

}  // namespace ssk
