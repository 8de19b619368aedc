// Single-direction selective scan, TMA-staged (sm_103a).
//
// Work split: a CTA owns CB consecutive channels of one (batch, group) and
// walks the sequence in chunks of T steps.  Inside a warp, lane = c*R + g:
// channel c of the warp, and state slice g holding NPT of the N states.  The
// fp32 states stay in registers for the whole sequence; Abar and Bbar are
// formed on the fly and never stored (the "do not materialise Abar, Bbar"
// point of the hardware-aware scan: "Mamba Series ..." review, core insight 1,
// and the Mamba reading notes, section 3.3.2).
//
// Per chunk:
//   1. TMA (64-byte rows, 64B swizzle) has landed the u, Delta, z tiles
//      [CB x T] and the B, C tiles [N x T] of this chunk in a STAGES-deep ring.
//   2. All threads convert B and C to fp32 in a pair-interleaved layout
//      (B[t], B[t+1]) so a lane reads its NPT states' inputs for two steps with
//      vector loads; every lane "preps" its own E steps of its channel:
//      Delta' = softplus(Delta + bias), x = Delta'*u, gate = SiLU(z), D*u*gate.
//   3. Barrier; thread 0 refills the ring slot just consumed.
//   4. Each warp scans its channels: per step pair and state n,
//         (a_t, a_t+1) = ex2(Delta' * A*log2e)   h = a*h + x*B   y += C*h
//      with packed f32x2 multiplies over the two steps.  Every R steps the R
//      partial readouts of a channel are combined by a butterfly so that lane g
//      ends with the full y of step g, applies y*gate + D*u*gate and stages it.
//   5. The warp writes its staged outputs with 16-byte coalesced stores.
//
// The same kernel runs the long-sequence chunked path: pass 1 scans L-chunks
// from a zero state and records each chunk's end state and sum of Delta';
// a carry kernel chains them; pass 2 rescans each chunk from its carried state.
#pragma once

#include "ss_device.cuh"

namespace ssk {

template <typename IO_, int N_, int NPT_, int W_, int STAGES_>
struct Cfg1 {
    using IO = IO_;
    static constexpr int N = N_, NPT = NPT_, W = W_, STAGES = STAGES_;
    static constexpr int R = N / NPT;    // lanes sharing one channel
    static constexpr int CPW = 32 / R;   // channels per warp
    static constexpr int CB = W * CPW;   // channels per CTA
    static constexpr int THREADS = 32 * W;
    static constexpr int ES = sizeof(IO);
    static constexpr int T = 64 / ES;    // steps per chunk (raw rows are 64 bytes)
    static constexpr int TP = T / 2;     // step pairs per chunk
    static constexpr int E = T / R;      // consecutive steps prepped by one lane
    static_assert(N % NPT == 0 && R >= 1 && R <= 32 && (R & (R - 1)) == 0, "lane split");
    static_assert(E >= 2 && E % 2 == 0 && E * ES >= 4, "a prep lane owns whole step pairs");
    static_assert(CB <= 256 && N <= 256, "TMA box rows");

    static constexpr int al(int x) { return (x + 1023) & ~1023; }
    static constexpr int TILE_CH = al(CB * 64);
    static constexpr int TILE_BC = al(N * 64);
    static constexpr int STAGE = 3 * TILE_CH + 2 * TILE_BC;
    static constexpr int OFF_U = 0, OFF_DL = TILE_CH, OFF_Z = 2 * TILE_CH;
    static constexpr int OFF_B = 3 * TILE_CH, OFF_C = 3 * TILE_CH + TILE_BC;
    static constexpr int BCBUF = TP * 4 * N * 4;  // fp32 B/C of one chunk
    static constexpr int OFF_BC = STAGES * STAGE;
    static constexpr int DXROW = (TP + 1) * 16;  // one padding slot per row
    static constexpr int OFF_DX = OFF_BC + 2 * BCBUF;
    static constexpr int OFF_GD = OFF_DX + CB * DXROW;
    static constexpr int OBROW = T * ES + 16;
    static constexpr int OFF_OB = OFF_GD + CB * DXROW;
    static constexpr int OFF_BAR = (OFF_OB + CB * OBROW + 7) & ~7;
    static constexpr int SMEM = OFF_BAR + 8 * STAGES + 1024;  // + alignment slack
};

struct Scan1dParams {
    int64_t dim, L;
    int G, dpg;
    int64_t Lc;   // steps per L-chunk (multiple of T); L for the direct path
    int J;        // number of L-chunks
    int jbase;    // L-chunk index of blockIdx.z == 0
    int pass;     // 0 direct, 1 chunk-local pass, 2 chunk fix-up pass
    const float *A, *D, *bias;
    int softplus, has_z;
    void *out;
    float *last_state;
    float *hend;          // [rows, J, N] end state of an L-chunk scanned from zero
    float *sdt;           // [rows, J]    sum of Delta' over an L-chunk
    const float *carry;   // [rows, J, N] state entering an L-chunk
};

// B/C tiles -> fp32, layout per step pair tp: [B: N pairs (t, t+1)][C: N pairs].
template <class C>
__device__ __forceinline__ void convert_bc(const uint8_t *tB, const uint8_t *tC, float *bc, int tid) {
    using IO = typename C::IO;
    constexpr int VPC = 16 / C::ES;  // values per 16-byte chunk
#pragma unroll 1
    for (int task = tid; task < 8 * C::N; task += C::THREADS) {
        const int n = task % C::N;
        const int isC = (task / C::N) & 1;
        const int q = task / (2 * C::N);  // 16-byte chunk of the 64-byte row
        float v[VPC];
        load_tile_row<IO, VPC>(isC ? tC : tB, n, q * VPC, v);
#pragma unroll
        for (int e = 0; e < VPC; e += 2) {
            const int tp = (q * VPC + e) >> 1;
            *reinterpret_cast<float2 *>(bc + tp * 4 * C::N + isC * 2 * C::N + 2 * n) =
                make_float2(v[e], v[e + 1]);
        }
    }
}

// Scans one chunk of T steps for this lane's channel slice.  DO_Y selects the
// readout (off in the chunk-local pass, which only needs the end state).
// `emit(y, t)` receives the full readout y of local step t (one lane per step).
template <class C, bool DO_Y, class Emit>
__device__ __forceinline__ void scan_chunk(const float4 *dxrow, const float *bc, int g,
                                           float (&h)[C::NPT], const float2 (&A2p)[C::NPT],
                                           Emit &&emit) {
    constexpr int R = C::R, NPT = C::NPT, N = C::N;
    constexpr int BS = R >= 2 ? R : 2;  // steps per readout block
    constexpr int PPB = BS / 2;
#pragma unroll
    for (int blk = 0; blk < C::T / BS; ++blk) {
        float v[BS];
#pragma unroll
        for (int pp = 0; pp < PPB; ++pp) {
            const int tp = blk * PPB + pp;
            const float4 d4 = dxrow[swz_slot(tp)];
            const float2 dl = make_float2(d4.x, d4.y);
            const float2 xx = make_float2(d4.z, d4.w);
            const float *bB = bc + tp * 4 * N + 2 * NPT * g;
            const float *bC = bB + 2 * N;
            float Bv[2 * NPT], Cv[2 * NPT];
            if constexpr (NPT == 1) {
                const float2 b2 = *reinterpret_cast<const float2 *>(bB);
                Bv[0] = b2.x; Bv[1] = b2.y;
                if constexpr (DO_Y) {
                    const float2 c2 = *reinterpret_cast<const float2 *>(bC);
                    Cv[0] = c2.x; Cv[1] = c2.y;
                }
            } else {
#pragma unroll
                for (int k = 0; k < NPT / 2; ++k) {
                    const float4 b4 = reinterpret_cast<const float4 *>(bB)[k];
                    Bv[4 * k] = b4.x; Bv[4 * k + 1] = b4.y; Bv[4 * k + 2] = b4.z; Bv[4 * k + 3] = b4.w;
                    if constexpr (DO_Y) {
                        const float4 c4 = reinterpret_cast<const float4 *>(bC)[k];
                        Cv[4 * k] = c4.x; Cv[4 * k + 1] = c4.y; Cv[4 * k + 2] = c4.z; Cv[4 * k + 3] = c4.w;
                    }
                }
            }
            float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                const float2 da = __fmul2_rn(dl, A2p[j]);
                const float a0 = ex2(da.x), a1 = ex2(da.y);
                const float2 bx = __fmul2_rn(xx, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                const float h0 = fmaf(a0, h[j], bx.x);
                const float h1 = fmaf(a1, h0, bx.y);
                h[j] = h1;
                if constexpr (DO_Y)
                    y2 = __ffma2_rn(make_float2(Cv[2 * j], Cv[2 * j + 1]), make_float2(h0, h1), y2);
            }
            v[2 * pp] = y2.x;
            v[2 * pp + 1] = y2.y;
        }
        if constexpr (DO_Y) {
            if constexpr (R >= 2) {
                const float y = transpose_reduce<R>(v, g);
                emit(y, blk * R + g);
            } else {
                emit(v[0], blk * 2);
                emit(v[1], blk * 2 + 1);
            }
        }
    }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS)
k_scan1d(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
         const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
         const __grid_constant__ CUtensorMap tm_C, const Scan1dParams p) {
    using IO = typename C::IO;
    constexpr int N = C::N, NPT = C::NPT, R = C::R, T = C::T, E = C::E;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = lane / R, g = lane % R;
    const int cblk = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / p.G, grp = bg % p.G;
    const int jc = p.jbase + blockIdx.z;
    const int ch = warp * C::CPW + c;
    const int dg = cblk * C::CB + ch;
    const bool valid = dg < p.dpg;
    const int d = grp * p.dpg + (valid ? dg : p.dpg - 1);
    const int64_t row = (int64_t)b * p.dim + d;
    const int row_tma = (int)((int64_t)b * p.dim + (int64_t)grp * p.dpg + (int64_t)cblk * C::CB);
    const int bcrow_tma = bg * N;
    const int64_t t_begin = (int64_t)jc * p.Lc;
    const int64_t t_end = min(p.L, t_begin + p.Lc);
    const int nchunks = (int)((t_end - t_begin + T - 1) / T);
    const bool do_y = (p.pass != 1) || (jc == 0);

    float2 A2p[NPT];
    float h[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
        const int n = g * NPT + j;
        const float a = __ldg(p.A + (int64_t)d * N + n) * kLog2e;
        A2p[j] = make_float2(a, a);
        h[j] = (p.pass == 2) ? __ldg(p.carry + (row * p.J + jc) * N + n) : 0.f;
    }
    const float Dd = p.D ? __ldg(p.D + d) : 0.f;
    const float bd = p.bias ? __ldg(p.bias + d) : 0.f;

    float *bcbuf0 = reinterpret_cast<float *>(smem + C::OFF_BC);
    const float4 *dxrow_c = reinterpret_cast<const float4 *>(smem + C::OFF_DX + ch * C::DXROW);
    float4 *dxrow = reinterpret_cast<float4 *>(smem + C::OFF_DX + ch * C::DXROW);
    float4 *gdrow = reinterpret_cast<float4 *>(smem + C::OFF_GD + ch * C::DXROW);
    uint8_t *obrow = smem + C::OFF_OB + ch * C::OBROW;
    const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
    const uint32_t smem0 = smem_u32(smem);
    const uint32_t tx_bytes = (p.has_z ? 3u : 2u) * C::CB * 64u + 2u * N * 64u;
    const uint64_t budget = g_wait_budget_ns;

    if (tid == 0) {
        prefetch_tensormap(&tm_u);
        prefetch_tensormap(&tm_dl);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        if (p.has_z) prefetch_tensormap(&tm_z);
#pragma unroll 1
        for (int s = 0; s < C::STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    __syncthreads();

    // diagnostics: this CTA leaves its first tile's barrier without arrivals
    const bool skip_first = (g_debug_flags & 1u) && blockIdx.x == 0 && blockIdx.y == 0 &&
                            blockIdx.z == 0;
    auto issue = [&](int i) {
        if (i == 0 && skip_first) return;
        const int s = i % C::STAGES;
        const uint32_t bar = bar0 + 8 * s;
        const uint32_t st = smem0 + s * C::STAGE;
        const int x = (int)(t_begin + (int64_t)i * T);
        mbar_expect_tx(bar, tx_bytes);
        tma_load_2d(st + C::OFF_U, &tm_u, x, row_tma, bar);
        tma_load_2d(st + C::OFF_DL, &tm_dl, x, row_tma, bar);
        if (p.has_z) tma_load_2d(st + C::OFF_Z, &tm_z, x, row_tma, bar);
        tma_load_2d(st + C::OFF_B, &tm_B, x, bcrow_tma, bar);
        tma_load_2d(st + C::OFF_C, &tm_C, x, bcrow_tma, bar);
    };
    if (tid == 0) {
#pragma unroll 1
        for (int i = 0; i < C::STAGES && i < nchunks; ++i) issue(i);
    }

    float sdt_acc = 0.f;
#pragma unroll 1
    for (int i = 0; i < nchunks; ++i) {
        const int s = i % C::STAGES;
        const bool ok = mbar_wait_bounded(bar0 + 8 * s, (i / C::STAGES) & 1, budget);
        const uint8_t *st = smem + s * C::STAGE;
        float *bc = bcbuf0 + (i & 1) * (C::BCBUF / 4);
        convert_bc<C>(st + C::OFF_B, st + C::OFF_C, bc, tid);

        // prep: this lane's E consecutive steps of its channel
        {
            float uu[E], dd[E], zz[E];
            load_tile_row<IO, E>(st + C::OFF_U, ch, E * g, uu);
            load_tile_row<IO, E>(st + C::OFF_DL, ch, E * g, dd);
            if (p.has_z) load_tile_row<IO, E>(st + C::OFF_Z, ch, E * g, zz);
            const int64_t t0 = t_begin + (int64_t)i * T + E * g;
#pragma unroll
            for (int e = 0; e < E; e += 2) {
                float dl[2], xx[2], ga[2], du[2];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    float v = dd[e + k] + bd;
                    if (p.softplus) v = softplus(v);
                    if (t0 + e + k >= t_end) v = 0.f;  // steps past the end leave h unchanged
                    dl[k] = v;
                    xx[k] = v * uu[e + k];
                    ga[k] = p.has_z ? silu(zz[e + k]) : 1.f;
                    du[k] = Dd * uu[e + k] * ga[k];
                    sdt_acc += v;
                }
                const int slot = swz_slot((E * g + e) >> 1);
                dxrow[slot] = make_float4(dl[0], dl[1], xx[0], xx[1]);
                gdrow[slot] = make_float4(ga[0], du[0], ga[1], du[1]);
            }
        }
        const int any_fail = __syncthreads_or(!ok);
        if (any_fail) {
            if (tid == 0) {
                report_timeout();
                // let every copy this CTA issued land before its smem goes away
#pragma unroll 1
                for (int k = i; k < nchunks && k < i + C::STAGES; ++k)
                    if (!(k == 0 && skip_first))
                        (void)mbar_wait_bounded(bar0 + 8 * (k % C::STAGES), (k / C::STAGES) & 1,
                                            1000000000ull);
            }
            return;
        }
        if (tid == 0 && i + C::STAGES < nchunks) {
            fence_proxy_async_smem();
            issue(i + C::STAGES);
        }

        if (do_y) {
            scan_chunk<C, true>(dxrow_c, bc, g, h, A2p, [&](float y, int t) {
                const float2 ge = reinterpret_cast<const float2 *>(gdrow + swz_slot(t >> 1))[t & 1];
                reinterpret_cast<IO *>(obrow)[t] = IOT<IO>::from_f(fmaf(y, ge.x, ge.y));
            });
        } else {
            scan_chunk<C, false>(dxrow_c, bc, g, h, A2p, [](float, int) {});
        }
        __syncwarp();

        if (do_y) {
            constexpr int VPC = 16 / C::ES;
#pragma unroll 1
            for (int k = lane; k < C::CPW * 4; k += 32) {
                const int rr = k >> 2, q = k & 3;
                const int chr = warp * C::CPW + rr;
                const int dgr = cblk * C::CB + chr;
                const int64_t t = t_begin + (int64_t)i * T + q * VPC;
                if (dgr < p.dpg && t < t_end) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(smem + C::OFF_OB + chr * C::OBROW + q * 16);
                    IO *dst = reinterpret_cast<IO *>(p.out) +
                              ((int64_t)b * p.dim + (int64_t)grp * p.dpg + dgr) * p.L + t;
                    *reinterpret_cast<uint4 *>(dst) = v;
                }
            }
            __syncwarp();
        }
    }

    if (!valid) return;
    const bool last_chunk = (jc == p.J - 1);
    if (p.last_state && (p.pass == 0 || (p.pass == 2 && last_chunk))) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) p.last_state[row * N + g * NPT + j] = h[j];
    }
    if (p.pass == 1) {
#pragma unroll
        for (int j = 0; j < NPT; ++j) p.hend[(row * p.J + jc) * N + g * NPT + j] = h[j];
#pragma unroll
        for (int m = 1; m < R; m <<= 1) sdt_acc += __shfl_xor_sync(kFull, sdt_acc, m);
        if (g == 0) p.sdt[row * p.J + jc] = sdt_acc;
    }
}

// Chains the L-chunks: carry[j] = state entering chunk j, from the chunk-local
// end states and the chunk decays exp(A * sum Delta').
__global__ void k_carry(int64_t rows, int64_t dim, int J, int N, const float *__restrict__ A,
                        const float *__restrict__ hend, const float *__restrict__ sdt,
                        float *__restrict__ carry) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= rows * N) return;
    const int64_t row = idx / N;
    const int n = (int)(idx % N);
    const int64_t d = row % dim;
    const float a = A[d * N + n];
    float hc = 0.f;
#pragma unroll 1
    for (int j = 0; j < J; ++j) {
        carry[(row * J + j) * N + n] = hc;
        if (j + 1 < J) hc = expf(a * sdt[row * J + j]) * hc + hend[(row * J + j) * N + n];
    }
}

}  // namespace ssk
