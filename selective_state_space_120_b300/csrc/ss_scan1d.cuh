// Single-direction selective scan, TMA-staged (sm_103a).
//
// Work split: a CTA owns CB consecutive channels of one (batch, group) and
// walks the sequence in chunks of T steps.  Inside a warp, lane = g*CPW + q:
// state slice g (NPT of the N states) of channel group q (CL consecutive
// channels).  Slice-major lanes put eight lanes that read the same B/C words
// in each quarter-warp, which halves the shared-memory wavefronts of the
// 16-byte B/C loads (the hardware serves a 16-byte load per quarter-warp and
// broadcasts a single address within it).  The fp32 states stay
// in registers for the whole sequence; Abar and Bbar are formed on the fly and
// never stored (the "do not materialise Abar, Bbar" point of the
// hardware-aware scan: "Mamba Series ..." review, core insight 1, and the
// Mamba reading notes, section 3.3.2).
//
// Why CL channels per lane: B and C are shared by every channel of a group,
// and shared memory delivers at most 128 bytes of lane data per clock per SM.
// A lane that reads its NPT states' B/C once and uses them for CL channels
// divides that traffic by CL, which is what bounds this kernel otherwise.
//
// Per chunk i (the prep of chunk i+1 runs in the same barrier interval as the
// scan of chunk i, so the two independent instruction streams interleave):
//   1. TMA (64-byte rows, 64B swizzle) has landed the u, Delta, z tiles
//      [CB x T] and the B, C tiles [N x T] of chunk i+1 in a STAGES-deep ring.
//   2. All threads convert chunk i+1's B and C to fp32 in a pair-interleaved
//      layout (B[t], B[t+1]) so a lane reads its NPT states' inputs for two
//      steps with vector loads; each thread "preps" E consecutive steps of one
//      channel: Delta' = softplus(Delta + bias), x = Delta'*u, gate = SiLU(z),
//      D*u*gate -- into the other half of double-buffered rows.
//   3. Each warp scans chunk i for its channels: per step pair, state n and
//      channel c,
//         (a_t, a_t+1) = ex2(Delta' * A*log2e)   h = a*h + x*B   y += C*h
//      with packed f32x2 multiplies over the two steps.  Every R steps the R
//      partial readouts of a channel are combined by a butterfly so that lane g
//      ends with the full y of step g, applies y*gate + D*u*gate and stages it.
//   4. The warp writes its staged outputs with 16-byte coalesced stores.
//   5. Barrier; thread 0 refills the ring slot of chunk i+1.
//
// The same kernel runs the long-sequence chunked path: pass 1 scans L-chunks
// from a zero state and records each chunk's end state and sum of Delta';
// a carry kernel chains them; pass 2 rescans each chunk from its carried state.
//
// It also runs the directions of multi-direction calls (MULTI = true): two
// directions side by side over grid z, each reading u as row-order tiles,
// forward or back to front, of u itself or of a copy of u permuted into its
// traversal's step order, and merging through fp32 accumulators (the merge
// modes below; the final sums by position are k_merge2_map, k_merge2 and
// k_merge_steps at the end of this file).
#pragma once

#include "ss_device.cuh"

namespace ssk {

template <typename IO_, int N_, int NPT_, int W_, int STAGES_, int CL_ = 1, int PIPE_ = 0,
          int OVL_ = 0, int VIEW_ = 0>
struct Cfg1 {
    using IO = IO_;
    static constexpr int N = N_, NPT = NPT_, W = W_, STAGES = STAGES_, CL = CL_;
    static constexpr bool PIPE = PIPE_ != 0;  // software-pipelined step loop
    // OVL: the prep of chunk i+1 shares a barrier interval with the scan of
    // chunk i (double-buffered prep rows); otherwise prep, barrier, scan.
    static constexpr bool OVL = OVL_ != 0;
    static constexpr int R = N / NPT;    // lanes sharing one channel group
    static constexpr int CPW = 32 / R;   // channel groups per warp
    static constexpr int CHW = CPW * CL; // channels per warp
    static constexpr int CB = W * CHW;   // channels per CTA
    static constexpr int THREADS = 32 * W;
    static constexpr int ES = sizeof(IO);
    static constexpr int T = 64 / ES;    // steps per chunk (raw rows are 64 bytes)
    static constexpr int TP = T / 2;     // step pairs per chunk
    static constexpr int PT = R / CL;    // prep threads per channel
    static constexpr int E = T / PT;     // consecutive steps prepped by one thread
    static constexpr int VPC = 16 / ES;  // values per 16 bytes
    static_assert(N % NPT == 0 && R >= 1 && R <= 32 && (R & (R - 1)) == 0, "lane split");
    static_assert(CL >= 1 && CL <= R && R % CL == 0, "channels per lane");
    static_assert(E >= 2 && E % 2 == 0 && E * ES >= 4, "a prep thread owns whole step pairs");
    static_assert(CB <= 256 && N <= 256, "TMA box rows");

    // VIEW: rows whose length is not a multiple of 16 bytes, read in place
    // through a view of the tensor whose rows hold P consecutive rows of it
    // (P * L * ES a multiple of 16, P a power of two dividing CB and N).  Each
    // chunk is P boxes, one per residue of the row index mod P, each starting
    // at the 16-byte boundary at or below its first step: tile rows hold
    // BW = T + VPC values, unswizzled, with the chunk's first step at a per-box
    // offset below VPC.  VIEW_ = 1: the direction-pair launch (no z tile, no
    // gate in the prep); VIEW_ = 2: the single-direction scan (with both).
    // A box lands at a 128-byte boundary (the copy's rule for its shared-memory
    // address): box j of a tile of `rows` rows starts at j * box_stride.
    static constexpr bool VIEW = VIEW_ != 0;
    static constexpr bool VIEWZ = VIEW_ == 2;      // a z tile and the gate in the prep
    static constexpr int BW = VIEW ? T + VPC : T;  // values per tile row
    static constexpr int ROWB = BW * ES;           // bytes per tile row
    static constexpr int al(int x) { return VIEW ? (x + 127) & ~127 : (x + 1023) & ~1023; }
    static __host__ __device__ constexpr int box_stride(int rows, int vshift) {
        return (((rows >> vshift) * ROWB) + 127) & ~127;
    }
    static constexpr int view_tile(int rows) {  // the largest over P = 2, 4, 8
        int m = 0;
        for (int vs = 1; vs <= 3; ++vs)
            if ((rows >> vs) > 0 && (1 << vs) * box_stride(rows, vs) > m) m = (1 << vs) * box_stride(rows, vs);
        return m;
    }
    static constexpr int TILE_CH = VIEW ? view_tile(CB) : al(CB * ROWB);
    static constexpr int TILE_BC = VIEW ? view_tile(N) : al(N * ROWB);
    static constexpr int NCHT = (VIEW && !VIEWZ) ? 2 : 3;  // channel tiles per stage: u, Delta (, z)
    static constexpr int STAGE = NCHT * TILE_CH + 2 * TILE_BC;
    static constexpr int OFF_U = 0, OFF_DL = TILE_CH, OFF_Z = 2 * TILE_CH;
    static constexpr int OFF_B = NCHT * TILE_CH, OFF_C = NCHT * TILE_CH + TILE_BC;
    // BCW: keep B/C as bf16 pairs (B[t], B[t+1]) in one 32-bit word (exact for
    // bf16 inputs), halving the shared-memory bytes each lane reads at the cost
    // of two integer ops per word to widen them.  Measured slower on the B300
    // for N = 16 (the step loop is issue-bound, not shared-memory-bound), so off.
    static constexpr bool BCW = false;
    static constexpr int BCBUF = TP * (BCW ? 2 : 4) * N * 4;  // B/C of one chunk
    static_assert(!BCW || PIPE, "packed B/C words are read by the pipelined step loop");
    static constexpr int OFF_BC = STAGES * STAGE;
    static constexpr int DXROW = (TP + 1) * 16;  // one padding slot per row
    // gd rows: (gate, D*u*gate) per step; a direction-pair VIEW launch has no
    // gate: D*u only (two padding slots: the channels of a warp start on
    // distinct 16-byte groups)
    static constexpr bool DU_ONLY = VIEW && !VIEWZ;
    static constexpr int GDROW = DU_ONLY ? (TP + 2) * 8 : DXROW;
    static constexpr int PREPBUF = CB * (DXROW + GDROW);  // dx and gd rows of one chunk
    static constexpr int NPREP = OVL ? 2 : 1;      // prep row buffers
    static constexpr int OFF_DX = OFF_BC + 2 * BCBUF;
    static constexpr int OFF_GD = OFF_DX + CB * DXROW;
    static constexpr int OBROW = T * 4 + 16;  // staged outputs (I/O type, or fp32 partials)
    static constexpr int OFF_OB = OFF_DX + NPREP * PREPBUF;
    // fused Conv1D: each channel's last three inputs of a chunk, double-buffered
    static constexpr int OFF_HALO = OFF_OB + CB * OBROW;
    static constexpr int HALO = VIEW ? 0 : 2 * CB * 16;
    static constexpr int OFF_BAR = (OFF_HALO + HALO + 7) & ~7;
    // alignment of the tiles: 1024 bytes for the swizzled ones, 128 for VIEW
    static constexpr int SALIGN = VIEW ? 128 : 1024;
    static constexpr int SMEM = OFF_BAR + 8 * STAGES + SALIGN;  // + alignment slack
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA");
};

// Output modes of one launch.  A single-direction scan stores its gated output
// (OUT_STORE).  A K-direction scan runs K launches in direction order over one
// fp32 accumulator of y_k + D_k*u by position: the first stores it, the middle
// ones add to it, and the last adds its own term, applies the gate and writes
// the I/O-typed output.  Each position receives its terms in launch order, so
// the merged result is deterministic.
// OUT_STEP (directions of any order, merged by a separate kernel): store
// y_k + D_k*u in fp32 by scan step, i.e. in the direction's own order.
enum { OUT_STORE = 0, OUT_ACC_FIRST = 1, OUT_ACC_ADD = 2, OUT_ACC_LAST = 3, OUT_STEP = 4 };

struct Scan1dParams {
    int64_t dim, L;
    int G, dpg;
    // L-chunks: chunk 0 covers steps [0, L0), chunk j in 1..J-2 the Lc steps
    // from L0 + (j-1)*Lc, chunk J-1 the rest up to L (L0 and Lc multiples of
    // T; J = 1 and L0 = Lc = L for the direct path).  Pass 1 runs chunks
    // 0..J-2 as blockIdx.z = 0..J-2; pass 2 runs chunk J-1 as blockIdx.z = 0
    // and chunks 1..J-2 as blockIdx.z = 1..J-2, so that each pass's longest
    // chunk is dispatched first.
    int64_t L0, Lc;
    int J;        // number of L-chunks
    int pass;     // 0 direct, 1 chunk-local pass, 2 chunk fix-up pass
    int K, k;     // directions of the call, and the one this launch scans
    int order;    // 0: u tiles in step order; 2: the same, read back to front
    int mode;     // OUT_*
    float *acc;   // [batch*dim, L] fp32 merge accumulator by position (modes 1-3)
    int64_t pitch;  // row pitch (elements) of the accumulators; L unless the inputs are re-pitched
    int vshift;     // VIEW tiles: log2 of the rows folded into one view row
    // Multi-direction launches may scan several directions side by side:
    // blockIdx.z = d selects direction k0 + d with its own order, mode and
    // accumulator (entries [0, nz)); odd d read u through the second map.
    int nz, k0;
    int orders_z[4], modes_z[4];
    float *accs_z[4];
    const void *u_g;        // u (the fused Conv1D's history across L-chunks)
    const void *z_g;        // z (the gate of the last direction of a merge)
    const float *A, *D, *bias;
    int softplus, has_z;
    int zoh;                // zero-order-hold input matrix (single direction)
    const float *h0;        // initial state [batch*dim, N] (single direction; nullable)
    int conv;               // fused Conv1D(k=4) + SiLU before the scan (single direction)
    const float *conv_w, *conv_b, *conv_x0;  // [dim, 4], [dim], [batch*dim, 3]
    void *out;
    float *last_state;      // [batch, K, dim, N]
    float *hend;          // [rows, J, N] end state of an L-chunk scanned from zero
    float *sdt;           // [rows, J]    sum of Delta' over an L-chunk
    const float *carry;   // [rows, J, N] state entering an L-chunk
};

// B/C tiles -> per step pair tp: [B: N pairs (t, t+1)][C: N pairs], as fp32
// pairs, or (C::BCW) as bf16 pairs packed in one 32-bit word -- which is
// exactly the word the tile holds at columns (t, t+1), so it is only moved.
template <class C>
__device__ __forceinline__ void convert_bc(const uint8_t *tB, const uint8_t *tC, float *bc, int tid,
                                           bool with_c = true) {
    using IO = typename C::IO;
    constexpr int VPC = 16 / C::ES;  // values per 16-byte chunk
    if constexpr (C::BCW) {
        uint32_t *bw = reinterpret_cast<uint32_t *>(bc);
#pragma unroll 1
        for (int task = tid; task < 8 * C::N; task += C::THREADS) {
            const int n = task % C::N;
            const int isC = (task / C::N) & 1;
            const int q = task / (2 * C::N);  // 16-byte chunk of the 64-byte row
            const uint4 w = *reinterpret_cast<const uint4 *>((isC ? tC : tB) + swz64(n * 64 + q * 16));
            const int tp0 = q * 4;            // four step pairs per 16 bytes
            uint32_t *dst = bw + tp0 * 2 * C::N + isC * C::N + n;
            dst[0] = w.x;
            dst[2 * C::N] = w.y;
            dst[4 * C::N] = w.z;
            dst[6 * C::N] = w.w;
        }
        return;
    }
#pragma unroll 1
    for (int task = tid; task < 8 * C::N; task += C::THREADS) {
        const int n = task % C::N;
        const int isC = (task / C::N) & 1;
        const int q = task / (2 * C::N);  // 16-byte chunk of the 64-byte row
        if (isC && !with_c) continue;
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

// One element of row `row`, column `col` of a swizzled 64-byte-row tile.
template <typename IO>
__device__ __forceinline__ float load_tile_elem(const uint8_t *tile, int row, int col) {
    const int off = swz64(row * 64 + col * (int)sizeof(IO));
    if constexpr (sizeof(IO) == 2)
        return __uint_as_float((uint32_t)(*reinterpret_cast<const unsigned short *>(tile + off)) << 16);
    else
        return *reinterpret_cast<const float *>(tile + off);
}

// VIEW tiles.  Byte offset of row r of a tile of `rows` rows: box r mod P,
// row r / P of that box.
template <class C>
__device__ __forceinline__ int view_row_off(int r, int rows, int vshift) {
    return (r & ((1 << vshift) - 1)) * C::box_stride(rows, vshift) + (r >> vshift) * C::ROWB;
}
// Offset of a chunk's first step in the box of row residue j: the distance
// from view column j*L + x down to a 16-byte boundary.  Chunks start on
// multiples of T (forward) or end on L less one (back to front), so the offset
// is (j*L) mod VPC forward and ((j+1)*L) mod VPC back to front for every chunk.
template <class C>
__device__ __forceinline__ int view_mis(int j, int L) {
    return (j * L) & (C::VPC - 1);
}
// E consecutive values from column col0 of the tile row at byte offset rowoff
// (ROWB bytes a row, no swizzle), which need not start on a 16-byte boundary:
// aligned 32-bit words, shifted into place (a shift of 0 or 16 bits for bf16).
// Callers keep col0 + E <= BW - 1, which keeps every word read inside the row.
template <class C, int E>
__device__ __forceinline__ void load_view_row(const uint8_t *tile, int rowoff, int col0, float *v) {
    using IO = typename C::IO;
    constexpr int PER = 4 / C::ES;
    constexpr int NW = E * C::ES / 4;  // whole words of output
    const int off = rowoff + col0 * C::ES;
    const uint32_t *w = reinterpret_cast<const uint32_t *>(tile + (off & ~3));
    if constexpr (C::ES == 4) {
#pragma unroll
        for (int k = 0; k < NW; ++k) unpack_word(w[k], v + k * PER, (IO *)nullptr);
    } else {
        const uint32_t sh = (uint32_t)(off & 3) * 8u;
        uint32_t ww[NW + 1];
#pragma unroll
        for (int k = 0; k <= NW; ++k) ww[k] = w[k];
#pragma unroll
        for (int k = 0; k < NW; ++k) unpack_word(__funnelshift_r(ww[k], ww[k + 1], sh), v + k * PER, (IO *)nullptr);
    }
}

// convert_bc over VIEW tiles: the B/C rows of a chunk of T steps starting on a
// multiple of T, of which the first `nvalid` exist (the rest are zeroed: in the
// view they are the next row's values or past the tensor).
template <class C>
__device__ __forceinline__ void convert_bc_view(const uint8_t *tB, const uint8_t *tC, float *bc, int tid,
                                                bool with_c, int L, int vshift, int nvalid) {
    constexpr int VPC = C::VPC;
    // segment-fastest tasks: the rows of one LDS start on the same bank (boxes
    // sit on 128-byte boundaries), so a warp spreads over segments first
#pragma unroll 1
    for (int task = tid; task < 8 * C::N; task += C::THREADS) {
        const int q = task & 3;  // VPC steps of the chunk
        const int n = (task >> 2) % C::N;
        const int isC = (task >> 2) / C::N;
        if (isC && !with_c) continue;
        float v[VPC];
        const int col0 = view_mis<C>(n & ((1 << vshift) - 1), L) + q * VPC;
        load_view_row<C, VPC>(isC ? tC : tB, view_row_off<C>(n, C::N, vshift), col0, v);
        if (nvalid < C::T) {
#pragma unroll
            for (int e = 0; e < VPC; ++e)
                if (q * VPC + e >= nvalid) v[e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < VPC; e += 2) {
            const int tp = (q * VPC + e) >> 1;
            *reinterpret_cast<float2 *>(bc + tp * 4 * C::N + isC * 2 * C::N + 2 * n) = make_float2(v[e], v[e + 1]);
        }
    }
}

// Scans one chunk of T steps, or its first nblk readout blocks (TAIL: a
// chunk that runs past the end of the sequence, whose later steps would leave
// h unchanged), for this lane's CL channels and state slice, one readout block
// at a time without the step pipeline of scan_chunk_pipe.  DO_Y selects the
// readout (off in the chunk-local pass, which only needs the end states).
// `emit(c, y, t)` receives the full readout y of channel c of the lane's group
// at local step t (one lane per step).
template <class C, bool DO_Y, bool TAIL = false, class Emit>
__device__ __forceinline__ void scan_chunk_cl(const float4 *const (&dxrow)[C::CL], const float *bc,
                                              int g, float (&h)[C::CL][C::NPT],
                                              const float2 (&A2p)[C::CL][C::NPT], Emit &&emit,
                                              int nblk = 0) {
    constexpr int R = C::R, NPT = C::NPT, N = C::N, CL = C::CL;
    constexpr int BS = R >= 2 ? R : 2;  // steps per readout block
    constexpr int PPB = BS / 2;
    auto block = [&](int blk) {
        float v[CL][BS];
#pragma unroll
        for (int pp = 0; pp < PPB; ++pp) {
            const int tp = blk * PPB + pp;
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
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                const float4 d4 = dxrow[c][swz_slot(tp)];
                const float2 dl = make_float2(d4.x, d4.y);
                const float2 xx = make_float2(d4.z, d4.w);
                float2 y2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int j = 0; j < NPT; ++j) {
                    const float2 da = __fmul2_rn(dl, A2p[c][j]);
                    const float a0 = ex2(da.x), a1 = ex2(da.y);
                    const float2 bx = __fmul2_rn(xx, make_float2(Bv[2 * j], Bv[2 * j + 1]));
                    const float h0 = fmaf(a0, h[c][j], bx.x);
                    const float h1 = fmaf(a1, h0, bx.y);
                    h[c][j] = h1;
                    if constexpr (DO_Y)
                        y2 = __ffma2_rn(make_float2(Cv[2 * j], Cv[2 * j + 1]), make_float2(h0, h1), y2);
                }
                v[c][2 * pp] = y2.x;
                v[c][2 * pp + 1] = y2.y;
            }
        }
        if constexpr (DO_Y) {
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                if constexpr (R >= 2) {
                    const float y = transpose_reduce<R, C::CPW>(v[c], g);
                    emit(c, y, blk * R + g);
                } else {
                    emit(c, v[c][0], blk * 2);
                    emit(c, v[c][1], blk * 2 + 1);
                }
            }
        }
    };
    if constexpr (TAIL) {
#pragma unroll 1
        for (int blk = 0; blk < nblk; ++blk) block(blk);
    } else {
#pragma unroll
        for (int blk = 0; blk < C::T / BS; ++blk) block(blk);
    }
}

// Registers of one step pair of scan_chunk_pipe: the exponentials, the input
// terms x*B and the readout weights C for the lane's channels and states.
template <class C>
struct StepRegs {
    float a[C::CL][C::NPT][2];
    float2 bx[C::CL][C::NPT];
    float Cv[2 * C::NPT];
};

// Loads and evaluates everything of step pair tp that does not depend on the
// state: smem loads, Delta'*A, ex2, x*B.
template <class C, bool DO_Y, bool ZOH>
__device__ __forceinline__ void stage_step(StepRegs<C> &r, const float4 *const (&dxrow)[C::CL],
                                           const float *bc, int g, int tp,
                                           const float2 (&A2p)[C::CL][C::NPT], const float *iA) {
    constexpr int NPT = C::NPT, N = C::N, CL = C::CL;
    float Bv[2 * NPT];
    if constexpr (C::BCW) {
        // bf16 pairs: low half step t, high half step t+1
        const uint32_t *wB = reinterpret_cast<const uint32_t *>(bc) + tp * 2 * N + NPT * g;
        const uint32_t *wC = wB + N;
        uint32_t bw[NPT], cw[NPT];
        if constexpr (NPT % 4 == 0) {
#pragma unroll
            for (int k = 0; k < NPT / 4; ++k) {
                const uint4 b4 = reinterpret_cast<const uint4 *>(wB)[k];
                bw[4 * k] = b4.x; bw[4 * k + 1] = b4.y; bw[4 * k + 2] = b4.z; bw[4 * k + 3] = b4.w;
                if constexpr (DO_Y) {
                    const uint4 c4 = reinterpret_cast<const uint4 *>(wC)[k];
                    cw[4 * k] = c4.x; cw[4 * k + 1] = c4.y; cw[4 * k + 2] = c4.z; cw[4 * k + 3] = c4.w;
                }
            }
        } else {
#pragma unroll
            for (int j = 0; j < NPT; ++j) {
                bw[j] = wB[j];
                if constexpr (DO_Y) cw[j] = wC[j];
            }
        }
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            Bv[2 * j] = __uint_as_float(bw[j] << 16);
            Bv[2 * j + 1] = __uint_as_float(bw[j] & 0xffff0000u);
            if constexpr (DO_Y) {
                r.Cv[2 * j] = __uint_as_float(cw[j] << 16);
                r.Cv[2 * j + 1] = __uint_as_float(cw[j] & 0xffff0000u);
            }
        }
    } else {
    const float *bB = bc + tp * 4 * N + 2 * NPT * g;
    const float *bC = bB + 2 * N;
    if constexpr (NPT == 1) {
        const float2 b2 = *reinterpret_cast<const float2 *>(bB);
        Bv[0] = b2.x; Bv[1] = b2.y;
        if constexpr (DO_Y) {
            const float2 c2 = *reinterpret_cast<const float2 *>(bC);
            r.Cv[0] = c2.x; r.Cv[1] = c2.y;
        }
    } else {
#pragma unroll
        for (int k = 0; k < NPT / 2; ++k) {
            const float4 b4 = reinterpret_cast<const float4 *>(bB)[k];
            Bv[4 * k] = b4.x; Bv[4 * k + 1] = b4.y; Bv[4 * k + 2] = b4.z; Bv[4 * k + 3] = b4.w;
            if constexpr (DO_Y) {
                const float4 c4 = reinterpret_cast<const float4 *>(bC)[k];
                r.Cv[4 * k] = c4.x; r.Cv[4 * k + 1] = c4.y; r.Cv[4 * k + 2] = c4.z; r.Cv[4 * k + 3] = c4.w;
            }
        }
    }
    }
#pragma unroll
    for (int c = 0; c < CL; ++c) {
        const float4 d4 = dxrow[c][swz_slot(tp)];
        const float2 dl = make_float2(d4.x, d4.y);
        const float2 xx = make_float2(d4.z, d4.w);
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const float2 da = __fmul2_rn(dl, A2p[c][j]);
            r.a[c][j][0] = ex2(da.x);
            r.a[c][j][1] = ex2(da.y);
            r.bx[c][j] = __fmul2_rn(xx, make_float2(Bv[2 * j], Bv[2 * j + 1]));
            if constexpr (ZOH) {
                // zero-order hold: Bbar*u = (exp(x) - 1)/A * B*u with x = Delta'*A
                // (the slots hold u, not Delta'*u).  For |x| < 1/16 use
                // Delta' * expm1(x)/x = Delta' (1 + x/2 + x^2/6 + x^3/24), whose
                // truncation error x^4/120 < 1.3e-7 avoids the cancellation of
                // exp(x) - 1; otherwise (exp(x) - 1) * (1/A).
                const float ia = iA[c * NPT + j];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const float x = (q ? da.y : da.x) * kLn2;
                    const float dlt = q ? dl.y : dl.x;
                    const float series = dlt * fmaf(x, fmaf(x, fmaf(x, 1.f / 24.f, 1.f / 6.f), 0.5f), 1.f);
                    const float coef = fabsf(x) < 0.0625f ? series : (r.a[c][j][q] - 1.f) * ia;
                    if (q) r.bx[c][j].y *= coef;
                    else r.bx[c][j].x *= coef;
                }
            }
        }
    }
}

// scan_chunk_cl with a one-step-pair software pipeline: the loads and
// exponentials of step pair tp+1 are issued before the state updates of tp, so
// their latency overlaps the dependent FMA chain.  With DEFER the per-step
// partial readouts of the whole chunk stay in registers and are combined
// (butterflies, then emit) after the chunk's last step: the step loop then
// holds no shuffle chains, and the T/R butterflies of a chunk are independent
// of one another -- faster when the kernel may use the registers it needs
// (the plain single-direction scan); otherwise (DEFER false) every R-step block
// is combined as soon as its partials are complete.
// ZOH selects the zero-order-hold input matrix at compile time (iA = 1/A per
// state); a runtime branch inside the unrolled step loop costs the scheduler
// its freedom to interleave across states and step pairs.
template <class C, bool DO_Y, bool ZOH = false, bool DEFER = false, class Emit>
__device__ __forceinline__ void scan_chunk_pipe(const float4 *const (&dxrow)[C::CL], const float *bc,
                                                int g, float (&h)[C::CL][C::NPT],
                                                const float2 (&A2p)[C::CL][C::NPT], Emit &&emit,
                                                const float *iA = nullptr) {
    constexpr int R = C::R, NPT = C::NPT, CL = C::CL;
    constexpr int BS = R >= 2 ? R : 2;  // steps per readout block
    constexpr int PPB = BS / 2;
    constexpr int VN = DEFER ? C::T : BS;
    StepRegs<C> cur, nxt;
    stage_step<C, DO_Y, ZOH>(nxt, dxrow, bc, g, 0, A2p, iA);
    float v[CL][VN];  // partial readouts: of the chunk (DEFER) or of one block
#pragma unroll
    for (int tp = 0; tp < C::TP; ++tp) {
        cur = nxt;
        if (tp + 1 < C::TP) stage_step<C, DO_Y, ZOH>(nxt, dxrow, bc, g, tp + 1, A2p, iA);
        const int vi = DEFER ? 2 * tp : 2 * (tp % PPB);
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            // written phase by phase (every state's first step, then every
            // state's second step, then the readout) so that independent FMAs
            // sit between each dependent pair
            float hs0[NPT];
#pragma unroll
            for (int j = 0; j < NPT; ++j) hs0[j] = fmaf(cur.a[c][j][0], h[c][j], cur.bx[c][j].x);
#pragma unroll
            for (int j = 0; j < NPT; ++j) h[c][j] = fmaf(cur.a[c][j][1], hs0[j], cur.bx[c][j].y);
            if constexpr (DO_Y) {
                // two readout accumulators halve the dependent FMA chain
                float2 y2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                for (int j = 0; j < NPT; ++j)
                    y2[j & 1] = __ffma2_rn(make_float2(cur.Cv[2 * j], cur.Cv[2 * j + 1]),
                                           make_float2(hs0[j], h[c][j]), y2[j & 1]);
                if constexpr (NPT > 1) y2[0] = __fadd2_rn(y2[0], y2[1]);
                v[c][vi] = y2[0].x;
                v[c][vi + 1] = y2[0].y;
            }
        }
        if constexpr (DO_Y && !DEFER) {
            if (tp % PPB == PPB - 1) {
                const int blk = tp / PPB;
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    if constexpr (R >= 2) {
                        const float y = transpose_reduce<R, C::CPW>(v[c], g);
                        emit(c, y, blk * R + g);
                    } else {
                        emit(c, v[c][0], blk * 2);
                        emit(c, v[c][1], blk * 2 + 1);
                    }
                }
            }
        }
    }
    if constexpr (DO_Y && DEFER) {
#pragma unroll
        for (int blk = 0; blk < C::T / BS; ++blk) {
#pragma unroll
            for (int c = 0; c < CL; ++c) {
                if constexpr (R >= 2) {
                    float w[BS];
#pragma unroll
                    for (int i = 0; i < BS; ++i) w[i] = v[c][blk * BS + i];
                    const float y = transpose_reduce<R, C::CPW>(w, g);
                    emit(c, y, blk * R + g);
                } else {
                    emit(c, v[c][blk * 2], blk * 2);
                    emit(c, v[c][blk * 2 + 1], blk * 2 + 1);
                }
            }
        }
    }
}

// Epilogue of the merge modes for one chunk (steps s0 .. s0+T-1 of direction
// k): the warp's staged fp32 partials y_k + D_k*u go to the accumulator
// (stored, added, or -- for the last direction -- added, gated by SiLU(z) and
// written to out in the I/O type).  An accumulator is indexed in its pair's
// traversal: by position for the row orders, by column-major index (the
// transposed map) for the column orders, so that in both cases step s of the
// forward order sits at index s and of the reversed order at index L-1-s; four
// steps are one 16-byte access.  Only row orders run the last mode (the column
// pair is transposed back by the final merge).  MergeRegs holds what a task
// reads from global memory (the accumulator and z), loaded one chunk early by
// load_partials so the latency hides behind the scan.
template <class C>
struct MergeRegs {
    static constexpr int QG = C::T / 4;  // groups of four steps per chunk
    static constexpr int TPL = (C::CHW * QG + 31) / 32;
    float4 acc[TPL];
    typename IOT<typename C::IO>::Raw z[TPL][4];
    // per task, fixed for the whole launch: the row offset (row * L, or -1 when
    // the task has no channel), the staged row in shared memory, the group
    int64_t rowL[TPL];
    int chr[TPL], qq[TPL];

    __device__ __forceinline__ void init(const Scan1dParams &p, int warp, int lane, int cblk, int64_t row0) {
#pragma unroll
        for (int m = 0; m < TPL; ++m) {
            const int task = lane + 32 * m;
            const int rr = task / QG;
            qq[m] = task % QG;
            chr[m] = warp * C::CHW + rr;
            const int dgr = cblk * C::CB + chr[m];
            rowL[m] = (task < C::CHW * QG && dgr < p.dpg) ? (row0 + dgr) * p.pitch : -1;
        }
    }
};

// Task m of this lane in the chunk starting at step s0: false if it has no
// channel or lies past the end; sg = its first step.
template <class C>
__device__ __forceinline__ bool merge_task(const Scan1dParams &p, const MergeRegs<C> &mr, int64_t s0,
                                           int m, int64_t &sg) {
    sg = s0 + mr.qq[m] * 4;
    return mr.rowL[m] >= 0 && sg < p.L;
}

template <class C>
__device__ __forceinline__ void load_partials(const Scan1dParams &p, MergeRegs<C> &mr, int64_t s0) {
    using IO = typename C::IO;
    if (p.mode == OUT_ACC_FIRST || p.mode == OUT_STEP) return;
#pragma unroll
    for (int m = 0; m < MergeRegs<C>::TPL; ++m) {
        int64_t sg;
        if (!merge_task<C>(p, mr, s0, m, sg)) continue;
        const float *accr = p.acc + mr.rowL[m];
        const IO *zr = reinterpret_cast<const IO *>(p.z_g) + mr.rowL[m];
        const bool gate = p.mode == OUT_ACC_LAST && p.has_z;
        const bool rev = p.order >= 2;
        const int64_t pos0 = rev ? p.L - 4 - sg : sg;
        mr.acc[m] = ld_pref_v4(accr + pos0);
        if (gate) {
#pragma unroll
            for (int j = 0; j < 4; ++j) mr.z[m][j] = IOT<IO>::load_raw(zr + pos0 + j);
        }
    }
}

template <class C>
__device__ __forceinline__ void store_partials(const Scan1dParams &p, const MergeRegs<C> &mr,
                                               const uint8_t *smem, int64_t s0) {
    using IO = typename C::IO;
#pragma unroll
    for (int m = 0; m < MergeRegs<C>::TPL; ++m) {
        int64_t sg;
        if (!merge_task<C>(p, mr, s0, m, sg)) continue;
        const float4 v = *reinterpret_cast<const float4 *>(smem + C::OFF_OB + mr.chr[m] * C::OBROW +
                                                           mr.qq[m] * 16);
        float *accr = p.acc + mr.rowL[m];
        if (p.mode == OUT_STEP) {  // by scan step: steps sg .. sg+3
            *reinterpret_cast<float4 *>(accr + sg) = v;
            continue;
        }
        IO *outr = reinterpret_cast<IO *>(p.out) + mr.rowL[m];
        const bool gate = p.mode == OUT_ACC_LAST && p.has_z;
        // w[j] is the term of step sg + j; a reversed order runs back to front
        const bool rev = p.order >= 2;
        float w[4] = {v.x, v.y, v.z, v.w};
        if (p.mode != OUT_ACC_FIRST) {
            const float4 o = mr.acc[m];  // prefetched, in accumulator order
            if (rev) {
                w[0] += o.w; w[1] += o.z; w[2] += o.y; w[3] += o.x;
            } else {
                w[0] += o.x; w[1] += o.y; w[2] += o.z; w[3] += o.w;
            }
        }
        if (gate) {
#pragma unroll
            for (int j = 0; j < 4; ++j) w[j] *= silu(IOT<IO>::widen(mr.z[m][rev ? 3 - j : j]));
        }
        const int64_t pos0 = rev ? p.L - 4 - sg : sg;
        float q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) q[j] = rev ? w[3 - j] : w[j];  // accumulator order
        if (p.mode != OUT_ACC_LAST) {
            *reinterpret_cast<float4 *>(accr + pos0) = make_float4(q[0], q[1], q[2], q[3]);
        } else if constexpr (sizeof(IO) == 2) {
            uint2 packed;
            packed.x = pack_bf16x2(q[0], q[1]);
            packed.y = pack_bf16x2(q[2], q[3]);
            *reinterpret_cast<uint2 *>(outr + pos0) = packed;
        } else {
            *reinterpret_cast<float4 *>(outr + pos0) = make_float4(q[0], q[1], q[2], q[3]);
        }
    }
}

// MULTI = false: a single-direction scan (order 0, OUT_STORE, one direction),
// with those fields fixed at compile time; MULTI = true: one direction of a
// multi-direction call, as the params say.
// Every traversal other than the row order and its reverse reaches the kernel
// as one of those two over a copy of u permuted into its step order, so u
// always arrives as TMA tiles.
// EXT = true compiles the optional paths of a single direction, the
// zero-order hold and the fused Conv1D; the plain instantiations carry none of
// their code, which keeps the default scans' registers and schedule.
// The body of the scan kernels; DEFER selects the chunk-deferred readout
// combination of scan_chunk_pipe.
template <class C, bool MULTI, bool EXT, bool DEFER>
__device__ __forceinline__ void scan1d_body(const CUtensorMap &tm_u, const CUtensorMap &tm_dl,
                                            const CUtensorMap &tm_z, const CUtensorMap &tm_B,
                                            const CUtensorMap &tm_C, const CUtensorMap &tm_u2,
                                            const Scan1dParams &p_in) {
    using IO = typename C::IO;
    Scan1dParams p = p_in;
    if constexpr (!MULTI) {
        p.K = 1;
        p.k = 0;
        p.order = 0;
        p.mode = OUT_STORE;
    } else {
        // direction of this slice of the grid: selects, not a dynamic index
        // (which would copy the params to the stack)
        const unsigned zi = blockIdx.z;
        const bool z1 = zi & 1u, z2 = zi & 2u;
        p.k = p.k0 + (int)zi;
        p.order = z2 ? (z1 ? p_in.orders_z[3] : p_in.orders_z[2]) : (z1 ? p_in.orders_z[1] : p_in.orders_z[0]);
        p.mode = z2 ? (z1 ? p_in.modes_z[3] : p_in.modes_z[2]) : (z1 ? p_in.modes_z[1] : p_in.modes_z[0]);
        p.acc = z2 ? (z1 ? p_in.accs_z[3] : p_in.accs_z[2]) : (z1 ? p_in.accs_z[1] : p_in.accs_z[0]);
    }
    constexpr int N = C::N, NPT = C::NPT, T = C::T, E = C::E, CL = C::CL;
    // u tiles: the two slices of a multi-direction launch may read different
    // maps (u, or the copies of u permuted into other traversals' step orders)
    const CUtensorMap *umap = (MULTI && (blockIdx.z & 1u)) ? &tm_u2 : &tm_u;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + ((C::SALIGN - (raw_addr & (C::SALIGN - 1u))) & (C::SALIGN - 1u));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = lane % C::CPW, g = lane / C::CPW;
    const int cblk = blockIdx.x;
    const int bg = blockIdx.y;
    const int b = bg / p.G, grp = bg % p.G;
    const int jc = MULTI ? 0 : (p.pass == 2 && blockIdx.z == 0) ? p.J - 1 : (int)blockIdx.z;
    const int64_t row0 = (int64_t)b * p.dim + (int64_t)grp * p.dpg;  // row of the group's channel 0
    const int row_tma = (int)(row0 + (int64_t)cblk * C::CB);          // u, z, out rows
    // Delta rows of direction k: [batch, K, dim]; B/C rows: [batch, K, G, N]
    const int dlrow_tma = (int)(((int64_t)b * p.K + p.k) * p.dim + (int64_t)grp * p.dpg +
                                (int64_t)cblk * C::CB);
    const int bcrow_tma = (int)((((int64_t)b * p.K + p.k) * p.G + grp) * N);
    const int64_t t_begin = jc == 0 ? 0 : p.L0 + (int64_t)(jc - 1) * p.Lc;
    const int64_t t_end = jc == p.J - 1 ? p.L : jc == 0 ? p.L0 : t_begin + p.Lc;
    const int nchunks = (int)((t_end - t_begin + T - 1) / T);
    // the chunk-local pass needs only the end states of chunks 1..J-2: no
    // readout, so no C tiles, no gate and no skip term
    const bool do_y = (p.pass != 1) || (jc == 0);
    const bool gate_in_prep = !C::DU_ONLY && do_y && (p.mode == OUT_STORE) && p.has_z;
    static_assert(!C::VIEW || (MULTI != C::VIEWZ), "pair VIEW tiles for multi-direction launches, "
                  "z-carrying ones for the single direction");
    static_assert(!(C::VIEW && EXT), "VIEW tiles carry no optional input paths");

    // scan role: channels ch[c] (within the CTA) of this lane's group
    int chs[CL];
    bool valid[CL];
    int64_t rows[CL];
    float2 A2p[CL][NPT];
    float h[CL][NPT];
    float iAv[CL * NPT];  // 1/A (0 where A = 0), for the zero-order hold
#pragma unroll
    for (int c = 0; c < CL; ++c) {
        chs[c] = warp * C::CHW + q * CL + c;
        const int dg = cblk * C::CB + chs[c];
        valid[c] = dg < p.dpg;
        const int64_t d = (int64_t)grp * p.dpg + (valid[c] ? dg : p.dpg - 1);
        rows[c] = (int64_t)b * p.dim + d;
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
            const int n = g * NPT + j;
            const float araw = __ldg(p.A + ((int64_t)p.k * p.dim + d) * N + n);
            const float a = araw * kLog2e;
            A2p[c][j] = make_float2(a, a);
            if (EXT) iAv[c * NPT + j] = araw != 0.f ? 1.f / araw : 0.f;
            h[c][j] = (p.pass == 2) ? __ldg(p.carry + (rows[c] * p.J + jc) * N + n)
                      : (p.h0 && jc == 0) ? __ldg(p.h0 + rows[c] * N + n) : 0.f;
        }
    }
    // prep role: E consecutive steps of channel pch, starting at step pt0 of the chunk
    const int pch = tid / C::PT;
    const int pt0 = (tid % C::PT) * E;
    // VIEW tiles: the prep channel's row in a tile and its chunks' offsets
    // there (forward, and back to front for u of a reversed order)
    const int vj = C::VIEW ? pch & ((1 << p.vshift) - 1) : 0;
    const int vroff = C::VIEW ? view_row_off<C>(pch, C::CB, p.vshift) : 0;
    const int vmis_f = C::VIEW ? view_mis<C>(vj, (int)p.L) : 0;
    const int vmis_r = C::VIEW ? view_mis<C>(vj + 1, (int)p.L) : 0;
    const int pdg = cblk * C::CB + pch;
    const bool pvalid = pdg < p.dpg;
    const int64_t pd = (int64_t)grp * p.dpg + (pvalid ? pdg : p.dpg - 1);
    const float Dd = p.D ? __ldg(p.D + (int64_t)p.k * p.dim + pd) : 0.f;
    const float bd = p.bias ? __ldg(p.bias + (int64_t)p.k * p.dim + pd) : 0.f;
    const int64_t prow = (int64_t)b * p.dim + pd;  // u/z row of the prep channel
    // fused Conv1D: weights of the prep channel and the three inputs before this
    // launch's first step (the given history at the start of the sequence, the
    // previous L-chunk's last inputs otherwise)
    // (loaded inside the prep, so they hold no registers across the chunk loop)
    const bool conv = EXT && !MULTI && !C::OVL && p.conv;  // (the overlapped order would need a deeper halo)
    float *halo = reinterpret_cast<float *>(smem + C::OFF_HALO);  // [2][CB][4]

    const float *zoh_iA = (EXT && !MULTI && p.zoh) ? iAv : nullptr;
    float *bcbuf0 = reinterpret_cast<float *>(smem + C::OFF_BC);
    uint8_t *obrows[CL];
#pragma unroll
    for (int c = 0; c < CL; ++c) obrows[c] = smem + C::OFF_OB + chs[c] * C::OBROW;
    const uint32_t bar0 = smem_u32(smem + C::OFF_BAR);
    const uint32_t smem0 = smem_u32(smem);
    const bool z_tiled = gate_in_prep;
    const uint32_t tx_bytes = (2u + (z_tiled ? 1u : 0u)) * C::CB * (uint32_t)C::ROWB +
                              (do_y ? 2u : 1u) * N * (uint32_t)C::ROWB;
    const uint64_t budget = g_wait_budget_ns;
    // VIEW tiles take P boxes per tensor a chunk: lane 0 of every warp issues
    // those of its tensors (each warp arrives on the stage's barrier with its
    // own bytes); other tiles, one box per tensor, all issued by thread 0
    const bool issuer = C::VIEW ? (lane == 0) : (tid == 0);

    if (tid == 0) {
        prefetch_tensormap(umap);
        prefetch_tensormap(&tm_dl);
        prefetch_tensormap(&tm_B);
        prefetch_tensormap(&tm_C);
        if (p.has_z) prefetch_tensormap(&tm_z);
#pragma unroll 1
        for (int s = 0; s < C::STAGES; ++s) mbar_init(bar0 + 8 * s, C::VIEW ? C::W : 1);
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
        // u/z tile of a reversed row order: positions L-(i+1)T .. L-1-iT (may
        // start below 0 on the last chunk; the copy fills zeros there)
        const int xu = (p.order == 2) ? (int)(p.L - (int64_t)(i + 1) * T) : x;
        if constexpr (C::VIEW) {
            // the chunk's tensors, in the order u, Delta, z (when tiled), B, C
            // (when read): warp w issues those of rank w, w + W, ...; box j
            // holds the rows r = j mod P, from view column j*L + first step
            // rounded down to a 16-byte boundary (a negative column reads
            // zeros; columns of a neighbouring row are masked by the prep)
            const int vs = p.vshift, P = 1 << vs, L32 = (int)p.L;
            const int ntens = 3 + (z_tiled ? 1 : 0) + (do_y ? 1 : 0);
            // rank -> tensor: 0 u, 1 Delta, 2 z, 3 B, 4 C
            auto tensor_of = [&](int r) { return r < 2 ? r : (z_tiled ? r : r + 1); };
            uint32_t bytes = 0;
            for (int r = warp; r < ntens; r += C::W) bytes += (tensor_of(r) < 3 ? C::CB : N) * C::ROWB;
            mbar_expect_tx(bar, bytes);
            for (int r = warp; r < ntens; r += C::W) {
                const int tsel = tensor_of(r);
                const CUtensorMap *map = tsel == 0 ? umap : tsel == 1 ? &tm_dl : tsel == 2 ? &tm_z
                                         : tsel == 3 ? &tm_B : &tm_C;
                const int vrow = (tsel == 0 || tsel == 2 ? row_tma : tsel == 1 ? dlrow_tma : bcrow_tma) >> vs;
                const uint32_t dst = st + (tsel == 0 ? C::OFF_U : tsel == 1 ? C::OFF_DL : tsel == 2 ? C::OFF_Z
                                           : tsel == 3 ? C::OFF_B : C::OFF_C);
                const int bs = C::box_stride(tsel < 3 ? C::CB : N, vs);
                int xj = (tsel == 0 || tsel == 2) ? xu : x;  // view column of box j's first step
#pragma unroll 1
                for (int j = 0; j < P; ++j, xj += L32)
                    tma_load_2d(dst + j * bs, map, xj & ~(C::VPC - 1), vrow, bar);
            }
            return;
        }
        mbar_expect_tx(bar, tx_bytes);
        tma_load_2d(st + C::OFF_U, umap, xu, row_tma, bar);
        tma_load_2d(st + C::OFF_DL, &tm_dl, x, dlrow_tma, bar);
        if (z_tiled) tma_load_2d(st + C::OFF_Z, &tm_z, xu, row_tma, bar);
        tma_load_2d(st + C::OFF_B, &tm_B, x, bcrow_tma, bar);
        if (do_y) tma_load_2d(st + C::OFF_C, &tm_C, x, bcrow_tma, bar);
    };
    if (issuer) {
#pragma unroll 1
        for (int i = 0; i < C::STAGES && i < nchunks; ++i) issue(i);
    }

    float sdt_acc = 0.f;
    MergeRegs<C> mr;
    if (MULTI) mr.init(p, warp, lane, cblk, row0);
    // Converts B/C and preps the steps of chunk i into buffer half (i & 1).
    auto prep_chunk = [&](int i) {
        const int s = i % C::STAGES;
        const uint8_t *st = smem + s * C::STAGE;
        const int64_t xc = t_begin + (int64_t)i * T;  // first step of the chunk
        if constexpr (C::VIEW)
            convert_bc_view<C>(st + C::OFF_B, st + C::OFF_C, bcbuf0 + (i & 1) * (C::BCBUF / 4), tid, do_y,
                               (int)p.L, p.vshift, (int)min((int64_t)T, t_end - xc));
        else
            convert_bc<C>(st + C::OFF_B, st + C::OFF_C, bcbuf0 + (i & 1) * (C::BCBUF / 4), tid, do_y);
        const int pb = C::OVL ? (i & 1) : 0;
        float4 *pdxrow = reinterpret_cast<float4 *>(smem + C::OFF_DX + pb * C::PREPBUF +
                                                    pch * C::DXROW);
        float4 *pgdrow = reinterpret_cast<float4 *>(smem + C::OFF_GD + pb * C::PREPBUF +
                                                    pch * C::GDROW);
        float uu[E], dd[E], zz[E];
        if constexpr (C::VIEW) {
            load_view_row<C, E>(st + C::OFF_DL, vroff, vmis_f + pt0, dd);
            if (p.order == 0) {
                load_view_row<C, E>(st + C::OFF_U, vroff, vmis_f + pt0, uu);
                if (z_tiled) load_view_row<C, E>(st + C::OFF_Z, vroff, vmis_f + pt0, zz);
            } else {
                float tmp[E];
                load_view_row<C, E>(st + C::OFF_U, vroff, vmis_r + T - pt0 - E, tmp);
#pragma unroll
                for (int e = 0; e < E; ++e) uu[e] = tmp[E - 1 - e];
            }
        } else {
        load_tile_row<IO, E>(st + C::OFF_DL, pch, pt0, dd);
        if (p.order == 0) {
            load_tile_row<IO, E>(st + C::OFF_U, pch, pt0, uu);
            if (z_tiled) load_tile_row<IO, E>(st + C::OFF_Z, pch, pt0, zz);
        } else {
            // reversed tile: step pt0+e sits at tile column T-1-(pt0+e)
            float tmp[E];
            load_tile_row<IO, E>(st + C::OFF_U, pch, T - pt0 - E, tmp);
#pragma unroll
            for (int e = 0; e < E; ++e) uu[e] = tmp[E - 1 - e];
            if (z_tiled) {
                load_tile_row<IO, E>(st + C::OFF_Z, pch, T - pt0 - E, tmp);
#pragma unroll
                for (int e = 0; e < E; ++e) zz[e] = tmp[E - 1 - e];
            }
        }
        }
        if (conv) {
            // raw inputs at columns pt0-3 .. pt0-1: this tile, or the previous
            // chunk's last three (the halo), or the history for the first chunk
            const float4 w4 = __ldg(reinterpret_cast<const float4 *>(p.conv_w) + pd);
            const float cw[4] = {w4.x, w4.y, w4.z, w4.w};
            const float cb = p.conv_b ? __ldg(p.conv_b + pd) : 0.f;
            float hx[3];
#pragma unroll
            for (int j = 0; j < 3; ++j) {
                const int col = pt0 - 3 + j;
                if (col >= 0) {
                    hx[j] = load_tile_elem<IO>(st + C::OFF_U, pch, col);
                } else if (i == 0) {
                    // before this launch's first step: the given history at the
                    // start of the sequence, else the previous L-chunk's inputs
                    const int hj = col + 3;
                    hx[j] = t_begin == 0
                                ? (p.conv_x0 ? __ldg(p.conv_x0 + prow * 3 + hj) : 0.f)
                                : IOT<IO>::load(reinterpret_cast<const IO *>(p.u_g) + prow * p.L +
                                                t_begin - 3 + hj);
                } else {
                    hx[j] = halo[((i & 1) * C::CB + pch) * 4 + col + 3];
                }
            }
            // keep this chunk's last three inputs for the next chunk
#pragma unroll
            for (int e = 0; e < E; ++e)
                if (pt0 + e >= T - 3) halo[((((i + 1) & 1) * C::CB) + pch) * 4 + pt0 + e - (T - 3)] = uu[e];
            float uc[E];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float x3 = e >= 3 ? uu[e - 3] : hx[e];
                const float x2 = e >= 2 ? uu[e - 2] : hx[e + 1];
                const float x1 = e >= 1 ? uu[e - 1] : hx[2];
                const float v = fmaf(cw[3], uu[e], fmaf(cw[2], x1, fmaf(cw[1], x2, fmaf(cw[0], x3, cb))));
                uc[e] = silu(v);
            }
#pragma unroll
            for (int e = 0; e < E; ++e) uu[e] = uc[e];
        }
        // steps of this chunk at or past the end of the L-chunk leave h unchanged
        const int lim = (int)min((int64_t)T, t_end - (t_begin + (int64_t)i * T)) - pt0;
        if (C::VIEW && t_end - xc < T) {
            // a VIEW tile holds the neighbouring row's values past the row's
            // ends (only in a chunk that runs past the end): zero them, so that
            // the terms of those steps are zero whatever the values were
#pragma unroll
            for (int e = 0; e < E; ++e)
                if (e >= lim) {
                    uu[e] = 0.f;
                    if (z_tiled) zz[e] = 0.f;
                }
        }
#pragma unroll
        for (int e = 0; e < E; e += 2) {
            float dl[2], xx[2], ga[2], du[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                float v = dd[e + k] + bd;
                if (p.softplus) v = softplus(v);
                if (e + k >= lim) v = 0.f;
                dl[k] = v;
                xx[k] = (EXT && !MULTI && p.zoh) ? uu[e + k] : v * uu[e + k];
                ga[k] = gate_in_prep ? silu(zz[e + k]) : 1.f;
                du[k] = Dd * uu[e + k] * ga[k];
                if (p.pass == 1) sdt_acc += v;
            }
            const int slot = swz_slot((pt0 + e) >> 1);
            pdxrow[slot] = make_float4(dl[0], dl[1], xx[0], xx[1]);
            if constexpr (C::DU_ONLY) reinterpret_cast<float2 *>(pgdrow)[slot] = make_float2(du[0], du[1]);
            else if (do_y) pgdrow[slot] = make_float4(ga[0], du[0], ga[1], du[1]);
        }
    };
    // Bounded wait for chunk i's tiles; on timeout the whole CTA drains its
    // copies and exits (returns true then).
    auto abandon = [&](int i, bool ok) -> bool {
        if (!__syncthreads_or(!ok)) return false;
        if (tid == 0) {
            report_timeout();
            // let every copy this CTA issued land before its smem goes away
#pragma unroll 1
            for (int k = i; k < nchunks && k < i + C::STAGES; ++k)
                if (!(k == 0 && skip_first))
                    (void)mbar_wait_bounded(bar0 + 8 * (k % C::STAGES), (k / C::STAGES) & 1,
                                            1000000000ull);
        }
        return true;
    };

    if (C::OVL && nchunks > 0) {
        const bool ok = mbar_wait_bounded(bar0, 0, budget);
        if (ok) prep_chunk(0);
        if (abandon(0, ok)) return;
        if (issuer && C::STAGES < nchunks) {
            fence_proxy_async_smem();
            issue(C::STAGES);
        }
    }
#pragma unroll 1
    for (int i = 0; i < nchunks; ++i) {
        const bool more = i + 1 < nchunks;
        bool ok = true;
        if constexpr (C::OVL) {
            if (more) {
                ok = mbar_wait_bounded(bar0 + 8 * ((i + 1) % C::STAGES), ((i + 1) / C::STAGES) & 1,
                                       budget);
                if (ok) prep_chunk(i + 1);
            }
        } else {
            // classic order: tiles of chunk i, prep, barrier, refill, scan
            ok = mbar_wait_bounded(bar0 + 8 * (i % C::STAGES), (i / C::STAGES) & 1, budget);
            if (ok) prep_chunk(i);
            if (abandon(i, ok)) return;
            if (issuer && i + C::STAGES < nchunks) {
                fence_proxy_async_smem();
                issue(i + C::STAGES);
            }
        }
        const int rb = C::OVL ? (i & 1) : 0;
        if (MULTI && do_y) load_partials<C>(p, mr, (int64_t)i * T);

        const float *bc = bcbuf0 + (i & 1) * (C::BCBUF / 4);
        const float4 *dxrows[CL];
        const float4 *gdrows[CL];
#pragma unroll
        for (int c = 0; c < CL; ++c) {
            dxrows[c] = reinterpret_cast<const float4 *>(smem + C::OFF_DX + rb * C::PREPBUF +
                                                         chs[c] * C::DXROW);
            gdrows[c] = reinterpret_cast<const float4 *>(smem + C::OFF_GD + rb * C::PREPBUF +
                                                         chs[c] * C::GDROW);
        }
        auto emit = [&](int c, float y, int t) {
            float v;
            if constexpr (C::DU_ONLY) {
                // D*u only (rows of GDROW bytes: two floats a step pair)
                v = y + reinterpret_cast<const float *>(gdrows[c])[2 * swz_slot(t >> 1) + (t & 1)];
            } else {
                const float2 ge = reinterpret_cast<const float2 *>(gdrows[c] + swz_slot(t >> 1))[t & 1];
                v = fmaf(y, ge.x, ge.y);
            }
            if (p.mode == OUT_STORE) reinterpret_cast<IO *>(obrows[c])[t] = IOT<IO>::from_f(v);
            else reinterpret_cast<float *>(obrows[c])[t] = v;
        };
        // valid steps of this chunk: fewer than T only in a chunk that runs
        // past the end of the sequence (or of the L-chunk)
        const int nvs = (int)min((int64_t)T, t_end - (t_begin + (int64_t)i * T));
        if constexpr (C::PIPE) {
            auto none = [](int, float, int) {};
            constexpr int BS = C::R >= 2 ? C::R : 2;  // steps per readout block
            if (C::VIEW && MULTI && nvs < T) {
                // only the readout blocks holding valid steps: the later steps
                // would leave h unchanged and their outputs are not stored (the
                // view-tiled direction pair only, whose 197-step rows would waste
                // 27 of 224 scanned steps; in the other kernels the extra path
                // costs their schedule more than it saves)
                const int nb = (nvs + BS - 1) / BS;
                if (do_y) scan_chunk_cl<C, true, true>(dxrows, bc, g, h, A2p, emit, nb);
                else scan_chunk_cl<C, false, true>(dxrows, bc, g, h, A2p, none, nb);
            } else if (EXT && zoh_iA) {
                if (do_y) scan_chunk_pipe<C, true, true>(dxrows, bc, g, h, A2p, emit, zoh_iA);
                else scan_chunk_pipe<C, false, true>(dxrows, bc, g, h, A2p, none, zoh_iA);
            } else {
                if (do_y) scan_chunk_pipe<C, true, false, DEFER>(dxrows, bc, g, h, A2p, emit);
                else scan_chunk_pipe<C, false, false, DEFER>(dxrows, bc, g, h, A2p, none);
            }
        } else {
            if (do_y) scan_chunk_cl<C, true>(dxrows, bc, g, h, A2p, emit);
            else scan_chunk_cl<C, false>(dxrows, bc, g, h, A2p, [](int, float, int) {});
        }
        __syncwarp();

        if (do_y && p.mode != OUT_STORE) {
            store_partials<C>(p, mr, smem, (int64_t)i * T);
            __syncwarp();
        } else if (C::VIEW && do_y) {
            // rows that do not start on 16-byte boundaries: one value per lane,
            // consecutive lanes on consecutive steps of a channel
#pragma unroll 1
            for (int k = lane; k < C::CHW * T; k += 32) {
                const int rr = k / T, e = k % T;
                const int chr = warp * C::CHW + rr;
                const int dgr = cblk * C::CB + chr;
                const int64_t t = t_begin + (int64_t)i * T + e;
                if (dgr < p.dpg && t < t_end)
                    reinterpret_cast<IO *>(p.out)[(row0 + dgr) * p.L + t] =
                        reinterpret_cast<const IO *>(smem + C::OFF_OB + chr * C::OBROW)[e];
            }
            __syncwarp();
        } else if (do_y) {
            constexpr int VPC = 16 / C::ES;
#pragma unroll 1
            for (int k = lane; k < C::CHW * 4; k += 32) {
                const int rr = k >> 2, qq = k & 3;
                const int chr = warp * C::CHW + rr;
                const int dgr = cblk * C::CB + chr;
                const int64_t t = t_begin + (int64_t)i * T + qq * VPC;
                if (dgr < p.dpg && t < t_end) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(smem + C::OFF_OB + chr * C::OBROW + qq * 16);
                    IO *dst = reinterpret_cast<IO *>(p.out) + (row0 + dgr) * p.L + t;
                    *reinterpret_cast<uint4 *>(dst) = v;
                }
            }
            __syncwarp();
        }
        if constexpr (C::OVL) {
            // chunk i+1's tiles are consumed and chunk i's rows are read: refill
            if (abandon(i + 1, ok)) return;
            if (issuer && more && i + 1 + C::STAGES < nchunks) {
                fence_proxy_async_smem();
                issue(i + 1 + C::STAGES);
            }
        }
    }

    if (p.pass == 1) {
        // sum of Delta' over this L-chunk: reduce over the channel's PT prep threads
#pragma unroll
        for (int m = 1; m < C::PT; m <<= 1) sdt_acc += __shfl_xor_sync(kFull, sdt_acc, m);
        if (pvalid && (tid % C::PT) == 0) p.sdt[(row0 + pdg) * p.J + jc] = sdt_acc;
    }
    const bool last_chunk = (jc == p.J - 1);
#pragma unroll
    for (int c = 0; c < CL; ++c) {
        if (!valid[c]) continue;
        if (p.last_state && (p.pass == 0 || (p.pass == 2 && last_chunk))) {
            // last_state [batch, K, dim, N]
            const int64_t ls = (((int64_t)b * p.K + p.k) * p.dim + (rows[c] - (int64_t)b * p.dim)) * N;
#pragma unroll
            for (int j = 0; j < NPT; ++j) p.last_state[ls + g * NPT + j] = h[c][j];
        }
        if (p.pass == 1) {
#pragma unroll
            for (int j = 0; j < NPT; ++j) p.hend[(rows[c] * p.J + jc) * N + g * NPT + j] = h[c][j];
        }
    }
}

// The scan kernel of every path but the direct single-direction one: the
// compiler's default register target; readouts combined block by block.
template <class C, bool MULTI, bool EXT = false>
__global__ void __launch_bounds__(C::THREADS)
k_scan1d(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
         const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
         const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_u2,
         const Scan1dParams p) {
    scan1d_body<C, MULTI, EXT, false>(tm_u, tm_dl, tm_z, tm_B, tm_C, tm_u2, p);
}

// The direct single-direction scan (one pass over the whole sequence, no
// options).  Its grid is one CTA per CB channels, a few per SM -- all the
// parallelism a scan has -- so warps are few and each must hide its own
// latencies: it may take as many registers as it wants (at least one CTA per
// SM), keeps the chunk's partial readouts in them and combines them after the
// chunk (DEFER).  On the chunked path, whose grids fill the SMs several times
// over, the same choice measured slower (a lower CTA residency), so that path
// keeps k_scan1d.
// (A VIEW configuration, whose shifted reads take more registers, is held to
// three CTAs per SM, as many as the plain one reaches unconstrained.)
template <class C>
__global__ void __launch_bounds__(C::THREADS, C::VIEW ? 3 : 1)
k_scan1d_direct(const __grid_constant__ CUtensorMap tm_u, const __grid_constant__ CUtensorMap tm_dl,
                const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_B,
                const __grid_constant__ CUtensorMap tm_C, const Scan1dParams p) {
    scan1d_body<C, false, false, true>(tm_u, tm_dl, tm_z, tm_B, tm_C, tm_u, p);
}

// Final merge of a four-direction call (SS2D) whose directions stored their
// terms y_k + D_k*u into four fp32 slices: the row orders by position
// (r0 forward, r1 reversed), the column orders by column-major index (c0, c1),
// i.e. each direction's steps in its pair's traversal.  out = (r0 + r1 +
// (c0 + c1) transposed back) gated by SiLU(z), in the I/O type.  Slices are
// [rows, H, W] (rows) and [rows, W, H] (columns).  One 32 x 32 tile of one row
// per block: the column tiles are read along their contiguous axis into shared
// memory and written out along the map's.
template <typename IO>
__global__ void __launch_bounds__(256) k_merge2(const float *__restrict__ r0, const float *__restrict__ r1,
                                                const float *__restrict__ c0, const float *__restrict__ c1,
                                                const IO *__restrict__ z, IO *__restrict__ out,
                                                int H, int W) {
    __shared__ float tile[32][33];
    const int64_t row = blockIdx.x;
    const int64_t L = (int64_t)H * W;
    const int cb = blockIdx.y * 32, rb = blockIdx.z * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int c = cb + ty + k, r = rb + tx;
        if (c < W && r < H) {
            const int64_t i = row * L + (int64_t)c * H + r;
            tile[ty + k][tx] = c0[i] + c1[i];
        }
    }
    __syncthreads();
    IO *o = out + row * L;
    const IO *zr = z ? z + row * L : nullptr;
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int r = rb + ty + k, c = cb + tx;
        if (c < W && r < H) {
            const int64_t pos = (int64_t)r * W + c;
            float v = r0[row * L + pos] + r1[row * L + pos] + tile[tx][ty + k];
            if (zr) v *= silu(IOT<IO>::load(zr + pos));
            o[pos] = IOT<IO>::from_f(v);
        }
    }
}

// k_merge2 for maps whose column slices fit in shared memory: one CTA (256
// threads) per row stages the sum of the two column slices as a whole
// column-major map with an odd column stride P >= H, so a warp reading one
// map row across consecutive columns hits 32 distinct banks, then sums every
// position.  Loads go four per thread at a time, for enough bytes in flight.
// Dynamic shared memory: W * P floats.
template <typename IO>
__global__ void __launch_bounds__(256) k_merge2_map(const float *__restrict__ r0, const float *__restrict__ r1,
                                                    const float *__restrict__ c0, const float *__restrict__ c1,
                                                    const IO *__restrict__ z, IO *__restrict__ out,
                                                    int H, int W, int P) {
    extern __shared__ float colmap[];  // [W][P]
    const int64_t row = blockIdx.x;
    const int L = H * W;
    const int t = threadIdx.x;
    constexpr int U = 4;
    {
        // column-major index i -> cell (r, c) = (i % H, i / H), stepped by 256
        const float *a0 = c0 + row * (int64_t)L, *a1 = c1 + row * (int64_t)L;
        int c = t / H, r = t - c * H;
        const int dc = 256 / H, dr = 256 - dc * H;
        for (int i0 = t; i0 < L; i0 += U * 256) {
            float v[U];
            int at[U];
#pragma unroll
            for (int j = 0; j < U; ++j) {
                const int i = i0 + j * 256;
                v[j] = i < L ? a0[i] + a1[i] : 0.f;
                at[j] = c * P + r;
                r += dr;
                c += dc;
                if (r >= H) {
                    r -= H;
                    ++c;
                }
            }
#pragma unroll
            for (int j = 0; j < U; ++j)
                if (i0 + j * 256 < L) colmap[at[j]] = v[j];
        }
    }
    __syncthreads();
    const float *b0 = r0 + row * (int64_t)L, *b1 = r1 + row * (int64_t)L;
    IO *o = out + row * (int64_t)L;
    const IO *zr = z ? z + row * (int64_t)L : nullptr;
    // map position -> cell (r, c) = (pos / W, pos % W), stepped by 256
    int r = t / W, c = t - r * W;
    const int dr = 256 / W, dc = 256 - dr * W;
    for (int p0 = t; p0 < L; p0 += U * 256) {
        float v[U], g[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int pos = p0 + j * 256;
            const bool in = pos < L;
            v[j] = in ? b0[pos] + b1[pos] + colmap[c * P + r] : 0.f;
            g[j] = (in && zr) ? IOT<IO>::load(zr + pos) : 0.f;
            c += dc;
            r += dr;
            if (c >= W) {
                c -= W;
                ++r;
            }
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int pos = p0 + j * 256;
            if (pos < L) o[pos] = IOT<IO>::from_f(zr ? v[j] * silu(g[j]) : v[j]);
        }
    }
}

// Four I/O values as one vector access (8 bytes for bf16, 16 for fp32).
template <typename IO> struct IO4;
template <> struct IO4<float> {
    static __device__ __forceinline__ float4 load(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    static __device__ __forceinline__ void store(float *p, float4 v) {
        *reinterpret_cast<float4 *>(p) = v;
    }
};
template <> struct IO4<__nv_bfloat16> {
    static __device__ __forceinline__ float4 load(const __nv_bfloat16 *p) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(p));
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, float4 v) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t *>(&lo);
        w.y = *reinterpret_cast<const uint32_t *>(&hi);
        *reinterpret_cast<uint2 *>(p) = w;
    }
};

// k_merge2_map with four consecutive values per access, for H and W multiples
// of 4 (a vector of the column slices then stays in one column, one of the row
// slices in one row) and z, out aligned to four values.  The same sums in the
// same order as k_merge2_map.  Dynamic shared memory: W * P floats.
template <typename IO>
__global__ void __launch_bounds__(256) k_merge2_map4(const float *__restrict__ r0, const float *__restrict__ r1,
                                                     const float *__restrict__ c0, const float *__restrict__ c1,
                                                     const IO *__restrict__ z, IO *__restrict__ out,
                                                     int H, int W, int P) {
    extern __shared__ float colmap[];  // [W][P]
    const int64_t row = blockIdx.x;
    const int L = H * W, nv = L / 4;
    const int t = threadIdx.x;
    constexpr int U = 2;
    {
        const float4 *a0 = reinterpret_cast<const float4 *>(c0 + row * (int64_t)L);
        const float4 *a1 = reinterpret_cast<const float4 *>(c1 + row * (int64_t)L);
        for (int i0 = t; i0 < nv; i0 += U * 256) {
            float4 x[U], y[U];
#pragma unroll
            for (int j = 0; j < U; ++j)
                if (i0 + j * 256 < nv) {
                    x[j] = a0[i0 + j * 256];
                    y[j] = a1[i0 + j * 256];
                }
#pragma unroll
            for (int j = 0; j < U; ++j)
                if (i0 + j * 256 < nv) {
                    const int i = 4 * (i0 + j * 256);
                    const int c = i / H, r = i - c * H;  // column-major index -> (r..r+3, c)
                    float *m = colmap + c * P + r;
                    m[0] = x[j].x + y[j].x;
                    m[1] = x[j].y + y[j].y;
                    m[2] = x[j].z + y[j].z;
                    m[3] = x[j].w + y[j].w;
                }
        }
    }
    __syncthreads();
    const float4 *b0 = reinterpret_cast<const float4 *>(r0 + row * (int64_t)L);
    const float4 *b1 = reinterpret_cast<const float4 *>(r1 + row * (int64_t)L);
    IO *o = out + row * (int64_t)L;
    const IO *zr = z ? z + row * (int64_t)L : nullptr;
    for (int p0 = t; p0 < nv; p0 += U * 256) {
        float4 x[U], y[U], g[U];
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (p0 + j * 256 < nv) {
                x[j] = b0[p0 + j * 256];
                y[j] = b1[p0 + j * 256];
                if (zr) g[j] = IO4<IO>::load(zr + 4 * (p0 + j * 256));
            }
#pragma unroll
        for (int j = 0; j < U; ++j)
            if (p0 + j * 256 < nv) {
                const int pos = 4 * (p0 + j * 256);
                const int r = pos / W, c = pos - r * W;  // map position -> (r, c..c+3)
                const float *m = colmap + c * P + r;
                float4 v = make_float4(x[j].x + y[j].x + m[0], x[j].y + y[j].y + m[P],
                                       x[j].z + y[j].z + m[2 * P], x[j].w + y[j].w + m[3 * P]);
                if (zr) {
                    v.x *= silu(g[j].x);
                    v.y *= silu(g[j].y);
                    v.z *= silu(g[j].z);
                    v.w *= silu(g[j].w);
                }
                IO4<IO>::store(o + pos, v);
            }
    }
}

// Final merge of a call whose directions stored their terms by scan step
// (OUT_STEP), for directions of any order: out[p] = (sum_k acc_k[step_k(p)]) *
// SiLU(z[p]) in the I/O type, where step_k inverts direction k's traversal.
// acc is [K][rows][L].  A thread owns one position: it inverts the K
// traversals once and then walks rows blockIdx.y, blockIdx.y + gridDim.y, ...
// (the traversals are the same for every row).
struct OrderSet {
    int K, H, W, win;
    int orders[8];
    int64_t pitch;  // row pitch (floats) of the accumulators: H*W, or more for view-tiled rows
};
template <typename IO>
__global__ void __launch_bounds__(256) k_merge_steps(const float *__restrict__ acc, int64_t rows,
                                                     const IO *__restrict__ z, IO *__restrict__ out,
                                                     const OrderSet os) {
    const int64_t L = (int64_t)os.H * os.W;
    const int pos = blockIdx.x * blockDim.x + threadIdx.x;
    if (pos >= L) return;
    const int r = pos / os.W, c = pos - r * os.W;
    uint32_t st[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) st[k] = k < os.K ? step_of(os.orders[k], r, c, os.H, os.W, os.win) : 0u;
    for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
        float y = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (k < os.K) y += acc[((int64_t)k * rows + row) * os.pitch + st[k]];
        const int64_t i = row * L + pos;
        if (z) y *= silu(IOT<IO>::load(z + i));
        out[i] = IOT<IO>::from_f(y);
    }
}

// Copy of u permuted into the step order of one traversal: out[row][s] =
// u[row][pos(s)].  A direction of that traversal (or of its reverse) then reads
// u as row-order tiles of the copy.  A thread owns one step: it finds the
// step's position once and walks rows blockIdx.y, blockIdx.y + gridDim.y, ...
// (the traversal is the same for every row).
template <typename IO>
__global__ void __launch_bounds__(256) k_permute_order(const IO *__restrict__ u, IO *__restrict__ out,
                                                       int64_t rows, int order, int H, int W, int win) {
    const int64_t L = (int64_t)H * W;
    const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= L) return;
    OrderWalk ow;
    ow.start(order, H, W, win, L, s);
    const int64_t pos = ow.pos_next();
    for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) out[row * L + s] = u[row * L + pos];
}

// Rows whose length is not a multiple of 16 bytes cannot be TMA tiles.  Such
// inputs are copied once per call into padded rows of pitch Lp (a multiple of
// 16 bytes) in the workspace; a job may also reverse its rows (the reversed
// direction of a bidirectional scan then reads u in its own step order).
// dst[r][c] = src[r][rev ? L-1-c : c] for c < L, zero for L <= c < Lp.
struct RepitchJob {
    const void *src;
    void *dst;
    int64_t rows;
    int rev;
};
struct RepitchJobs {
    RepitchJob job[6];
    int n;
    int64_t L, Lp;
};
// 128 bits of a 256-bit window (four 64-bit words, low first) starting at bit
// 8 * sb (sb a multiple of the element size, below 16).
__device__ __forceinline__ uint4 window_bits(const uint64_t (&q)[4], int sb) {
    const int j = sb >> 3, b = (sb & 7) * 8;
    const uint64_t a0 = j ? q[1] : q[0], a1 = j ? q[2] : q[1], a2 = j ? q[3] : q[2];
    const uint64_t lo = b ? (a0 >> b) | (a1 << (64 - b)) : a0;
    const uint64_t hi = b ? (a1 >> b) | (a2 << (64 - b)) : a1;
    return make_uint4((uint32_t)lo, (uint32_t)(lo >> 32), (uint32_t)hi, (uint32_t)(hi >> 32));
}

// One thread writes one 16-byte vector of a padded row (8 bf16 or 4 fp32);
// blockIdx.y selects the job.  The source span of the vector (unaligned in
// general) is read as the two aligned 16-byte vectors that cover it and
// shifted into place; vectors at the ends of the tensor, where that window
// would leave it, are read element by element.
template <typename IO>
__global__ void __launch_bounds__(256) k_repitch(const RepitchJobs jobs) {
    constexpr int ES = sizeof(IO), VPV = 16 / ES;
    const RepitchJob jb = jobs.job[blockIdx.y];
    const int64_t L = jobs.L;
    const int64_t vpr = jobs.Lp / VPV;  // vectors per padded row
    const int64_t nvec = jb.rows * vpr;
    const int64_t nel = jb.rows * L;    // source elements
    const IO *src = reinterpret_cast<const IO *>(jb.src);
    const uint4 *src4 = reinterpret_cast<const uint4 *>(jb.src);
    // two vectors per thread and iteration, so that four 16-byte loads are in flight
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    auto vector_at = [&](int64_t v) -> uint4 {
        const int64_t r = v / vpr;
        const int64_t c0 = (v - r * vpr) * VPV;
        const int nv = (int)min((int64_t)VPV, max((int64_t)0, L - c0));  // valid elements
        uint4 out = make_uint4(0, 0, 0, 0);
        if (nv > 0) {
            // source elements of the vector, in output order: e0 + e (forward) or
            // e0 + VPV-1 - e (reversed); e0 = first element of the window
            const int64_t e0 = jb.rev ? r * L + L - c0 - VPV : r * L + c0;
            const int64_t w0 = e0 >= 0 ? e0 / VPV : -1;
            if (w0 >= 0 && (w0 + 2) * VPV <= nel) {
                const uint4 va = src4[w0], vb = src4[w0 + 1];
                const uint64_t q[4] = {(uint64_t)va.x | ((uint64_t)va.y << 32),
                                       (uint64_t)va.z | ((uint64_t)va.w << 32),
                                       (uint64_t)vb.x | ((uint64_t)vb.y << 32),
                                       (uint64_t)vb.z | ((uint64_t)vb.w << 32)};
                out = window_bits(q, (int)(e0 - w0 * VPV) * ES);
                if (jb.rev) {  // reverse the element order
                    if constexpr (ES == 2)
                        out = make_uint4(__byte_perm(out.w, 0, 0x1032), __byte_perm(out.z, 0, 0x1032),
                                         __byte_perm(out.y, 0, 0x1032), __byte_perm(out.x, 0, 0x1032));
                    else
                        out = make_uint4(out.w, out.z, out.y, out.x);
                }
            } else {
                typename IOT<IO>::Raw w[VPV];
#pragma unroll
                for (int e = 0; e < VPV; ++e) {
                    const int64_t c = c0 + e;
                    w[e] = 0;
                    if (c < L) w[e] = IOT<IO>::load_raw(src + r * L + (jb.rev ? L - 1 - c : c));
                }
                if constexpr (ES == 2)
                    out = make_uint4((uint32_t)w[0] | ((uint32_t)w[1] << 16), (uint32_t)w[2] | ((uint32_t)w[3] << 16),
                                     (uint32_t)w[4] | ((uint32_t)w[5] << 16), (uint32_t)w[6] | ((uint32_t)w[7] << 16));
                else
                    out = make_uint4(__float_as_uint(w[0]), __float_as_uint(w[1]), __float_as_uint(w[2]),
                                     __float_as_uint(w[3]));
            }
            if (nv < VPV) {  // zero the columns past the row's end
                uint32_t o[4] = {out.x, out.y, out.z, out.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int lo_e = i * 4 / ES;  // first element held by word i
                    if (ES == 2) {
                        if (lo_e >= nv) o[i] = 0;
                        else if (lo_e + 1 >= nv) o[i] &= 0xffffu;
                    } else if (lo_e >= nv) {
                        o[i] = 0;
                    }
                }
                out = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        return out;
    };
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += 2 * stride) {
        const int64_t v2 = v + stride;
        const uint4 o1 = vector_at(v);
        const uint4 o2 = v2 < nvec ? vector_at(v2) : make_uint4(0, 0, 0, 0);
        reinterpret_cast<uint4 *>(jb.dst)[v] = o1;
        if (v2 < nvec) reinterpret_cast<uint4 *>(jb.dst)[v2] = o2;
    }
}

// Final merge of a bidirectional call over re-pitched rows: the forward and the
// reversed direction stored y_k + D_k*u by scan step into fp32 slices of pitch
// Lp (s0 by position, s1 by position L-1-step); out[r][p] = (s0[r][p] +
// s1[r][L-1-p]) * SiLU(z[r][p]) in the I/O type, rows of the caller's pitch L.
// A thread takes four consecutive positions of a row: one 16-byte load of s0,
// four of s1 (read backwards) and of z, four stores.
template <typename IO>
__global__ void __launch_bounds__(256) k_merge_bidir(const float *__restrict__ s0,
                                                     const float *__restrict__ s1,
                                                     const IO *__restrict__ z, IO *__restrict__ out,
                                                     int64_t rows, int64_t L, int64_t Lp, FastDiv dq) {
    const int64_t qpr = (L + 3) / 4;  // groups of four positions per row
    const int64_t n = rows * qpr;
    // group -> row by a multiply-shift when the group count fits 32 bits (dq
    // divides by qpr), a 64-bit division otherwise
    const bool narrow = n <= 0xffffffffll;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = narrow ? (int64_t)dq.div((uint32_t)i) : i / qpr;
        const int64_t p0 = (i - r * qpr) * 4;
        const float4 a = *reinterpret_cast<const float4 *>(s0 + r * Lp + p0);
        const float av[4] = {a.x, a.y, a.z, a.w};
        const float *b = s1 + r * Lp + (L - 1);
        // every load of the group is issued before the first use
        float bv[4], zv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const bool in = p0 + j < L;
            bv[j] = in ? b[-(p0 + j)] : 0.f;
            zv[j] = (in && z) ? IOT<IO>::load(z + r * L + p0 + j) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (p0 + j >= L) break;
            float y = av[j] + bv[j];
            if (z) y *= silu(zv[j]);
            out[r * L + p0 + j] = IOT<IO>::from_f(y);
        }
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
