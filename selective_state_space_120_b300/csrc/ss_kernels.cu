// Kernel instantiations and launchers of the selective-scan library (sm_103a).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ss_bwd.cuh"
#include "ss_chunks.h"
#include "ss_conv2d.cuh"
#include "ss_device.cuh"
#include "ss_internal.h"
#include "ss_multidir.cuh"
#include "ss_scan1d.cuh"
#include "ss_step.cuh"

namespace ssi {

namespace {

// ---------------------------------------------------------------- tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D map over a [rows, cols] row-major tensor with a row pitch of `pitch`
// elements (0: cols); boxes of [box_rows, box_cols] with 64-byte rows and the
// 64-byte swizzle.  Out-of-range boxes read zeros.
ss_status make_map(CUtensorMap *m, const void *base, int io, uint64_t cols, uint64_t rows,
                   uint32_t box_cols, uint32_t box_rows, uint64_t pitch = 0) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(SS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const uint64_t es = (io == SS_BF16) ? 2 : 4;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {(pitch ? pitch : cols) * es};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, io == SS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SS_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return SS_OK;
}

// View of a [rows, cols] row-major tensor whose rows are not 16-byte aligned
// as a [rows / P, P * cols] tensor (P * cols * element size a multiple of 16),
// boxes of [box_rows, box_cols] unswizzled (the VIEW tiles of the scan).
ss_status make_view_map(CUtensorMap *m, const void *base, int io, uint64_t cols, uint64_t rows, int P,
                        uint32_t box_cols, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(SS_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const uint64_t es = (io == SS_BF16) ? 2 : 4;
    cuuint64_t dims[2] = {(uint64_t)P * cols, rows / (uint64_t)P};
    cuuint64_t strides[1] = {(uint64_t)P * cols * es};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, io == SS_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SS_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", (int)r);
    return SS_OK;
}

ss_status check_launch(const char *what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SS_ERR_CUDA, "%s launch failed: %s", what, cudaGetErrorString(e));
    return SS_OK;
}

int num_sms() {
    int dev = 0, n = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 148;
    } else {
        cudaGetLastError();  // no device on this host: size for a B300 (148 SMs)
    }
    return n;
}

// ---------------------------------------------------------------- traversal copies
// Base traversal of an order: the step order of the copy of u its direction
// reads.  0 = u itself (row orders), 1 = column-major, 2 = windows, 3 = windows
// taken column-major; a reversed order reads its base's copy back to front.
int order_base(int o) {
    if (o == ORD_ROW || o == ORD_ROW_REV) return 0;
    if (o == ORD_COL || o == ORD_COL_REV) return 1;
    return (o == ORD_WIN || o == ORD_WIN_REV) ? 2 : 3;
}
bool order_reversed(int o) {
    return o == ORD_ROW_REV || o == ORD_COL_REV || o == ORD_WIN_REV || o == ORD_WIN_COL_REV;
}
constexpr int kBaseOrder[4] = {ORD_ROW, ORD_COL, ORD_WIN, ORD_WIN_COL};

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// Row length rounded up to a multiple of 16 bytes (the pitch of re-pitched copies).
int64_t padded_len(const ScanArgs &a) {
    const int64_t vpv = a.io == SS_BF16 ? 8 : 4;
    return (a.L + vpv - 1) / vpv * vpv;
}

// Workspace of a bidirectional call over rows that are not 16-byte aligned:
// the two directions' fp32 terms [2, rows, Lp], u forward and reversed [rows,
// Lp], Delta [2 rows, Lp], B and C [batch*2*G*N, Lp].
size_t bidir_padded_bytes(const ScanArgs &a) {
    const int64_t rows = a.batch * a.dim, Lp = padded_len(a);
    const size_t es = a.io == SS_BF16 ? 2 : 4;
    const int64_t bcrows = a.batch * 2 * a.G * a.N;
    return align256((size_t)2 * rows * Lp * sizeof(float)) + 2 * align256((size_t)rows * Lp * es) +
           align256((size_t)2 * rows * Lp * es) + 2 * align256((size_t)bcrows * Lp * es);
}

// Workspace of a call over directions of any order: the fp32 accumulators by
// step [K][rows][L], then one permuted copy of u per base traversal in use.
size_t steps_acc_bytes(const ScanArgs &a) {
    return align256((size_t)a.K * a.batch * a.dim * a.L * sizeof(float));
}
size_t steps_copy_bytes(const ScanArgs &a) {
    return align256((size_t)a.batch * a.dim * a.L * (a.io == SS_BF16 ? 2 : 4));
}
// slot[b] = index of base b's copy, or -1 when no direction reads it; returns
// the number of copies.
int steps_copy_slots(const ScanArgs &a, int slot[4]) {
    bool used[4] = {false, false, false, false};
    for (int k = 0; k < a.K; ++k) used[order_base(a.orders[k])] = true;
    int n = 0;
    slot[0] = -1;
    for (int b = 1; b < 4; ++b) slot[b] = used[b] ? n++ : -1;
    return n;
}

// Writes u permuted into the step order of `order` (a column or windowed base
// order) to `dst`: the column order by whole-plane shared-memory transposes
// (planes of at most 48 KB whose H is a multiple of a 16-byte vector) or 32 x
// 32 tiles, any order by one walk of the traversal per step.
ss_status permuted_copy(const ScanArgs &a, int order, void *dst) {
    const int64_t rows = a.batch * a.dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
    const bool tiles = order == ORD_COL && (a.H + 31) / 32 <= 65535 && (a.W + 31) / 32 <= 65535 &&
                       rows < (1ll << 31);
    const int es = a.io == SS_BF16 ? 2 : 4;
    const bool planes = order == ORD_COL && a.H % (16 / es) == 0 && a.L * es <= 48 * 1024 &&
                        rows < (1ll << 31) && reinterpret_cast<uintptr_t>(a.u) % 16 == 0 &&
                        reinterpret_cast<uintptr_t>(dst) % 16 == 0;
    if (planes) {
        const size_t sm = (size_t)a.L * es;
        if (a.io == SS_BF16)
            ssk::k_transpose_planes<__nv_bfloat16><<<(unsigned)rows, 256, sm, s>>>(
                reinterpret_cast<const __nv_bfloat16 *>(a.u), reinterpret_cast<__nv_bfloat16 *>(dst),
                (int)a.H, (int)a.W);
        else
            ssk::k_transpose_planes<float><<<(unsigned)rows, 256, sm, s>>>(
                reinterpret_cast<const float *>(a.u), reinterpret_cast<float *>(dst), (int)a.H, (int)a.W);
        return check_launch("map transpose");
    }
    if (tiles) {
        const dim3 tg((unsigned)rows, (unsigned)((a.H + 31) / 32), (unsigned)((a.W + 31) / 32));
        if (a.io == SS_BF16)
            ssk::k_transpose_maps<__nv_bfloat16><<<tg, 256, 0, s>>>(
                reinterpret_cast<const __nv_bfloat16 *>(a.u), reinterpret_cast<__nv_bfloat16 *>(dst),
                (int)a.H, (int)a.W);
        else
            ssk::k_transpose_maps<float><<<tg, 256, 0, s>>>(reinterpret_cast<const float *>(a.u),
                                                            reinterpret_cast<float *>(dst), (int)a.H,
                                                            (int)a.W);
        return check_launch("map transpose");
    }
    const unsigned bx = (unsigned)((a.L + 255) / 256);
    const int64_t want_y = std::max<int64_t>(1, (int64_t)num_sms() * 32 / bx);
    const dim3 grid(bx, (unsigned)std::min<int64_t>({rows, want_y, (int64_t)65535}));
    if (a.io == SS_BF16)
        ssk::k_permute_order<__nv_bfloat16><<<grid, 256, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16 *>(a.u), reinterpret_cast<__nv_bfloat16 *>(dst), rows,
            order, (int)a.H, (int)a.W, a.win);
    else
        ssk::k_permute_order<float><<<grid, 256, 0, s>>>(reinterpret_cast<const float *>(a.u),
                                                         reinterpret_cast<float *>(dst), rows, order,
                                                         (int)a.H, (int)a.W, a.win);
    return check_launch("order permute");
}

// ---------------------------------------------------------------- single direction
template <class C>
struct Scan1d {
    // One direction; a VIEW configuration (rows not 16-byte aligned, read in
    // place through views of 1 << vshift rows to a view row) takes the plain
    // kernel only.
    static ss_status run(const ScanArgs &a, int J, int vshift = 0) {
        using namespace ssk;
        const int io = a.io;
        const int64_t rows = a.batch * a.dim;
        const uint64_t bcrows = (uint64_t)a.batch * a.G * C::N;
        CUtensorMap mu, md, mz, mb, mc;
        ss_status st;
        if constexpr (C::VIEW) {
            const int P = 1 << vshift;
            const uint32_t bch = (uint32_t)(C::CB >> vshift), bbc = (uint32_t)(C::N >> vshift);
            if ((st = make_view_map(&mu, a.u, io, a.L, rows, P, C::BW, bch))) return st;
            if ((st = make_view_map(&md, a.delta, io, a.L, rows, P, C::BW, bch))) return st;
            if ((st = make_view_map(&mz, a.z ? a.z : a.u, io, a.L, rows, P, C::BW, bch))) return st;
            if ((st = make_view_map(&mb, a.B, io, a.L, bcrows, P, C::BW, bbc))) return st;
            if ((st = make_view_map(&mc, a.C, io, a.L, bcrows, P, C::BW, bbc))) return st;
        } else {
            if ((st = make_map(&mu, a.u, io, a.L, rows, C::T, C::CB))) return st;
            if ((st = make_map(&md, a.delta, io, a.L, rows, C::T, C::CB))) return st;
            if ((st = make_map(&mz, a.z ? a.z : a.u, io, a.L, rows, C::T, C::CB))) return st;
            if ((st = make_map(&mb, a.B, io, a.L, bcrows, C::T, C::N))) return st;
            if ((st = make_map(&mc, a.C, io, a.L, bcrows, C::T, C::N))) return st;
        }

        // the plain kernel unless the zero-order hold or the fused Conv1D is asked for
        auto kern = k_scan1d<C, false, false>;
        if constexpr (!C::VIEW) {
            if (a.zoh || a.conv) kern = k_scan1d<C, false, true>;
        }
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
        const bool plain = !a.zoh && !a.conv;

        Scan1dParams p{};
        p.dim = a.dim;
        p.L = a.L;
        p.pitch = a.L;
        p.vshift = vshift;
        p.G = a.G;
        p.dpg = (int)(a.dim / a.G);
        p.K = 1;
        p.k = 0;
        p.order = ORD_ROW;
        p.mode = OUT_STORE;
        p.u_g = a.u;
        p.z_g = a.z;
        p.A = a.A;
        p.D = a.D;
        p.bias = a.bias;
        p.softplus = a.softplus;
        p.has_z = a.z != nullptr;
        p.zoh = a.zoh;
        p.h0 = a.h0;
        p.conv = a.conv;
        p.conv_w = a.conv_w;
        p.conv_b = a.conv_b;
        p.conv_x0 = a.conv_x0;
        p.out = a.out;
        p.last_state = a.last_state;
        const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
        const unsigned bgs = (unsigned)(a.batch * a.G);
        cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
        const ChunkGeom geo = chunk_geom(a.L, J, (int64_t)cblocks * bgs,
                                         (int64_t)num_sms() * slots_per_sm(), C::T);
        J = geo.J;
        if (J <= 1) {
            p.Lc = a.L;
            p.J = 1;
            p.L0 = a.L;
            p.pass = 0;
            if (plain) {
                auto kd = k_scan1d_direct<C>;
                if (cudaFuncSetAttribute(kd, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
                    cudaSuccess)
                    return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
                kd<<<dim3(cblocks, bgs, 1), C::THREADS, C::SMEM, s>>>(mu, md, mz, mb, mc, p);
            } else {
                kern<<<dim3(cblocks, bgs, 1), C::THREADS, C::SMEM, s>>>(mu, md, mz, mb, mc, mu, p);
            }
            return check_launch("scan");
        }
        // chunked path: the L-chunks of `geo`
        float *ws = reinterpret_cast<float *>(a.ws);
        p.L0 = geo.L0;
        p.Lc = geo.Lm;
        p.J = J;
        p.hend = ws;
        p.carry = ws + rows * J * C::N;
        p.sdt = ws + 2 * rows * J * C::N;
        p.pass = 1;
        kern<<<dim3(cblocks, bgs, J - 1), C::THREADS, C::SMEM, s>>>(mu, md, mz, mb, mc, mu, p);
        if ((st = check_launch("scan chunk-local pass"))) return st;
        const int64_t nthr = rows * C::N;
        k_carry<<<(unsigned)((nthr + 255) / 256), 256, 0, s>>>(rows, a.dim, J, C::N, a.A, p.hend,
                                                            p.sdt, const_cast<float *>(p.carry));
        if ((st = check_launch("carry"))) return st;
        p.pass = 2;
        kern<<<dim3(cblocks, bgs, J - 1), C::THREADS, C::SMEM, s>>>(mu, md, mz, mb, mc, mu, p);
        return check_launch("scan fix-up pass");
    }
    // K directions (bidirectional or SS2D) as K launches over one fp32
    // accumulator by position: direction k reads its Delta_k, B_k, C_k rows in
    // scan order and u at the positions its order visits; the first launch
    // stores y_0 + D_0*u, the middle ones add, the last adds, gates and writes out.
    static ss_status run_dirs(const ScanArgs &a) {
        using namespace ssk;
        const int io = a.io;
        const int64_t rows = a.batch * a.dim;
        const int K = a.K;
        CUtensorMap mu, md, mz, mb, mc;
        ss_status st;
        if ((st = make_map(&mu, a.u, io, a.L, rows, C::T, C::CB))) return st;
        if ((st = make_map(&md, a.delta, io, a.L, (uint64_t)rows * K, C::T, C::CB))) return st;
        if ((st = make_map(&mz, a.z ? a.z : a.u, io, a.L, rows, C::T, C::CB))) return st;
        const uint64_t bcrows = (uint64_t)a.batch * K * a.G * C::N;
        if ((st = make_map(&mb, a.B, io, a.L, bcrows, C::T, C::N))) return st;
        if ((st = make_map(&mc, a.C, io, a.L, bcrows, C::T, C::N))) return st;
        auto kern = k_scan1d<C, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
        Scan1dParams p{};
        p.dim = a.dim;
        p.L = a.L;
        p.pitch = a.L;
        p.G = a.G;
        p.dpg = (int)(a.dim / a.G);
        p.Lc = a.L;
        p.J = 1;
        p.L0 = a.L;
        p.pass = 0;
        p.K = K;
        p.acc = reinterpret_cast<float *>(a.ws);
        p.u_g = a.u;
        p.z_g = a.z;
        p.A = a.A;
        p.D = a.D;
        p.bias = a.bias;
        p.softplus = a.softplus;
        p.has_z = a.z != nullptr;
        p.out = a.out;
        p.last_state = a.last_state;
        const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
        const unsigned bgs = (unsigned)(a.batch * a.G);
        cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
        float *acc0 = reinterpret_cast<float *>(a.ws);
        if (K != 4) {
            // directions in order over one accumulator: store, add, ..., add + gate + write
            for (int k = 0; k < K; ++k) {
                p.nz = 1;
                p.k0 = k;
                p.orders_z[0] = a.orders[k];
                p.modes_z[0] = (k == 0) ? OUT_ACC_FIRST : (k == K - 1) ? OUT_ACC_LAST : OUT_ACC_ADD;
                p.accs_z[0] = acc0;
                kern<<<dim3(cblocks, bgs, 1), C::THREADS, C::SMEM, s>>>(mu, md, mz, mb, mc, mu, p);
                if ((st = check_launch("direction scan"))) return st;
            }
            return SS_OK;
        }
        // SS2D: one launch of the four directions side by side (grid z), each
        // storing y_k + D_k*u into its own fp32 slice in its pair's traversal
        // (the row orders by position, the column orders by column-major index,
        // so every access is a contiguous 16-byte vector), then one merge.
        // The column directions read u as row-order tiles of the transposed map
        // (one transpose, instead of a gather per element): the odd slices of
        // the launch take that map, and their orders are presented as row
        // orders (column -> row, reversed column -> reversed row).
        const size_t map4 = (size_t)rows * a.L;
        float *sl[4] = {acc0, acc0 + map4, acc0 + 2 * map4, acc0 + 3 * map4};
        CUtensorMap mu2;
        void *uT = reinterpret_cast<uint8_t *>(a.ws) + 4 * map4 * sizeof(float);
        if ((st = permuted_copy(a, ORD_COL, uT))) return st;
        if ((st = make_map(&mu2, uT, io, a.L, rows, C::T, C::CB))) return st;
        p.nz = 4;
        p.k0 = 0;
        for (int d = 0; d < 4; ++d) {
            const int o = a.orders[d];
            p.orders_z[d] = (o == ORD_ROW || o == ORD_COL) ? ORD_ROW : ORD_ROW_REV;
            p.modes_z[d] = OUT_ACC_FIRST;
            p.accs_z[d] = sl[d];
        }
        kern<<<dim3(cblocks, bgs, 4), C::THREADS, C::SMEM, s>>>(mu, md, mz, mb, mc, mu2, p);
        if ((st = check_launch("four-direction scan"))) return st;
        using IO = typename C::IO;
        // slices: 0 row, 1 column, 2 reversed row, 3 reversed column
        // whole maps in shared memory when the column map fits (odd stride P)
        const int P = (a.H & 1) ? (int)a.H : (int)a.H + 1;
        const size_t msm = (size_t)a.W * P * sizeof(float);
        const uintptr_t al = 4 * sizeof(IO);
        if (msm <= 48 * 1024 && rows < (1ll << 31) && a.H % 4 == 0 && a.W % 4 == 0 &&
            reinterpret_cast<uintptr_t>(a.out) % al == 0 && reinterpret_cast<uintptr_t>(a.z) % al == 0) {
            k_merge2_map4<IO><<<(unsigned)rows, 256, msm, s>>>(sl[0], sl[2], sl[1], sl[3],
                                                               reinterpret_cast<const IO *>(a.z),
                                                               reinterpret_cast<IO *>(a.out), (int)a.H,
                                                               (int)a.W, P);
            return check_launch("merge");
        }
        if (msm <= 48 * 1024 && rows < (1ll << 31)) {
            k_merge2_map<IO><<<(unsigned)rows, 256, msm, s>>>(sl[0], sl[2], sl[1], sl[3],
                                                              reinterpret_cast<const IO *>(a.z),
                                                              reinterpret_cast<IO *>(a.out), (int)a.H,
                                                              (int)a.W, P);
            return check_launch("merge");
        }
        const dim3 mgrid((unsigned)rows, (unsigned)((a.W + 31) / 32), (unsigned)((a.H + 31) / 32));
        k_merge2<IO><<<mgrid, dim3(32, 8), 0, s>>>(sl[0], sl[2], sl[1], sl[3],
                                                  reinterpret_cast<const IO *>(a.z),
                                                  reinterpret_cast<IO *>(a.out), (int)a.H, (int)a.W);
        return check_launch("merge");
    }

    // Bidirectional call over rows that are not 16-byte aligned: the inputs are
    // re-pitched into the workspace (u twice, forward and reversed; Delta, B,
    // C) so that both directions read TMA tiles in their own step order; they
    // scan side by side, each storing y_k + D_k*u by scan step into an fp32
    // slice, and one more launch sums the slices by position and gates.
    static ss_status run_bidir_padded(const ScanArgs &a) {
        using namespace ssk;
        using IO = typename C::IO;
        const int io = a.io;
        const int64_t rows = a.batch * a.dim;
        const int64_t Lp = padded_len(a);
        const size_t es = io == SS_BF16 ? 2 : 4;
        cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
        uint8_t *ws = reinterpret_cast<uint8_t *>(a.ws);
        const int64_t bcrows = a.batch * 2 * a.G * C::N;
        float *s0 = reinterpret_cast<float *>(ws);
        float *s1 = s0 + rows * Lp;
        uint8_t *cp = ws + align256((size_t)2 * rows * Lp * sizeof(float));
        void *uf = cp;
        void *ur = cp + align256((size_t)rows * Lp * es);
        void *dlp = reinterpret_cast<uint8_t *>(ur) + align256((size_t)rows * Lp * es);
        void *bp = reinterpret_cast<uint8_t *>(dlp) + align256((size_t)2 * rows * Lp * es);
        void *cpp = reinterpret_cast<uint8_t *>(bp) + align256((size_t)bcrows * Lp * es);
        RepitchJobs jobs{};
        jobs.L = a.L;
        jobs.Lp = Lp;
        jobs.n = 5;
        jobs.job[0] = {a.u, uf, rows, 0};
        jobs.job[1] = {a.u, ur, rows, 1};
        jobs.job[2] = {a.delta, dlp, 2 * rows, 0};
        jobs.job[3] = {a.B, bp, bcrows, 0};
        jobs.job[4] = {a.C, cpp, bcrows, 0};
        ss_status st;
        {
            const int64_t vmax = 2 * rows * (Lp * (int64_t)es / 16);
            const unsigned bx = (unsigned)std::min<int64_t>((vmax + 255) / 256, (int64_t)num_sms() * 16);
            k_repitch<IO><<<dim3(bx, 5), 256, 0, s>>>(jobs);
            if ((st = check_launch("re-pitch"))) return st;
        }
        CUtensorMap mu, mur, md, mb, mc;
        if ((st = make_map(&mu, uf, io, a.L, rows, C::T, C::CB, Lp))) return st;
        if ((st = make_map(&mur, ur, io, a.L, rows, C::T, C::CB, Lp))) return st;
        if ((st = make_map(&md, dlp, io, a.L, (uint64_t)rows * 2, C::T, C::CB, Lp))) return st;
        if ((st = make_map(&mb, bp, io, a.L, (uint64_t)bcrows, C::T, C::N, Lp))) return st;
        if ((st = make_map(&mc, cpp, io, a.L, (uint64_t)bcrows, C::T, C::N, Lp))) return st;
        auto kern = k_scan1d<C, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
        Scan1dParams p{};
        p.dim = a.dim;
        p.L = a.L;
        p.pitch = Lp;
        p.G = a.G;
        p.dpg = (int)(a.dim / a.G);
        p.Lc = a.L;
        p.J = 1;
        p.L0 = a.L;
        p.pass = 0;
        p.K = 2;
        p.u_g = a.u;
        p.A = a.A;
        p.D = a.D;
        p.bias = a.bias;
        p.softplus = a.softplus;
        p.has_z = 0;
        p.out = a.out;
        p.last_state = a.last_state;
        p.nz = 2;
        p.k0 = 0;
        for (int d = 0; d < 2; ++d) {
            p.orders_z[d] = ORD_ROW;  // each over its own copy of u, in its step order
            p.modes_z[d] = OUT_STEP;
            p.accs_z[d] = d == 0 ? s0 : s1;
        }
        const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
        const unsigned bgs = (unsigned)(a.batch * a.G);
        kern<<<dim3(cblocks, bgs, 2), C::THREADS, C::SMEM, s>>>(mu, md, mu, mb, mc, mur, p);
        if ((st = check_launch("direction pair scan"))) return st;
        const int64_t groups = rows * ((a.L + 3) / 4);
        const unsigned mblocks = (unsigned)std::min<int64_t>((groups + 255) / 256, (int64_t)num_sms() * 32);
        k_merge_bidir<IO><<<mblocks, 256, 0, s>>>(s0, s1, reinterpret_cast<const IO *>(a.z),
                                                  reinterpret_cast<IO *>(a.out), rows, a.L, Lp,
                                                  FastDiv((uint32_t)((a.L + 3) / 4)));
        return check_launch("bidirectional merge");
    }

    // Bidirectional call over rows that are not 16-byte aligned, read in place
    // through VIEW tiles (C is a VIEW configuration; P = 1 << vshift rows per
    // view row): the two directions scan side by side, direction 1 reading u's
    // tiles back to front, each storing y_k + D_k*u by scan step into an fp32
    // slice of pitch Lp, and one more launch sums the slices by position and
    // gates -- the re-pitched path without its copies.
    static ss_status run_bidir_view(const ScanArgs &a, int vshift) {
        using namespace ssk;
        using IO = typename C::IO;
        static_assert(C::VIEW, "a VIEW configuration");
        const int io = a.io;
        const int P = 1 << vshift;
        const int64_t rows = a.batch * a.dim;
        const int64_t Lp = padded_len(a);
        cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
        float *s0 = reinterpret_cast<float *>(a.ws);
        float *s1 = s0 + rows * Lp;
        const int64_t bcrows = a.batch * 2 * a.G * C::N;
        ss_status st;
        CUtensorMap mu, md, mb, mc;
        if ((st = make_view_map(&mu, a.u, io, a.L, rows, P, C::BW, C::CB >> vshift))) return st;
        if ((st = make_view_map(&md, a.delta, io, a.L, (uint64_t)rows * 2, P, C::BW, C::CB >> vshift))) return st;
        if ((st = make_view_map(&mb, a.B, io, a.L, (uint64_t)bcrows, P, C::BW, C::N >> vshift))) return st;
        if ((st = make_view_map(&mc, a.C, io, a.L, (uint64_t)bcrows, P, C::BW, C::N >> vshift))) return st;
        auto kern = k_scan1d<C, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
        Scan1dParams p{};
        p.dim = a.dim;
        p.L = a.L;
        p.pitch = Lp;
        p.vshift = vshift;
        p.G = a.G;
        p.dpg = (int)(a.dim / a.G);
        p.Lc = a.L;
        p.J = 1;
        p.L0 = a.L;
        p.pass = 0;
        p.K = 2;
        p.u_g = a.u;
        p.A = a.A;
        p.D = a.D;
        p.bias = a.bias;
        p.softplus = a.softplus;
        p.has_z = 0;
        p.out = a.out;
        p.last_state = a.last_state;
        p.nz = 2;
        p.k0 = 0;
        p.orders_z[0] = ORD_ROW;
        p.orders_z[1] = ORD_ROW_REV;
        for (int d = 0; d < 2; ++d) {
            p.modes_z[d] = OUT_STEP;
            p.accs_z[d] = d == 0 ? s0 : s1;
        }
        const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
        const unsigned bgs = (unsigned)(a.batch * a.G);
        kern<<<dim3(cblocks, bgs, 2), C::THREADS, C::SMEM, s>>>(mu, md, mu, mb, mc, mu, p);
        if ((st = check_launch("direction pair scan"))) return st;
        const int64_t groups = rows * ((a.L + 3) / 4);
        const unsigned mblocks = (unsigned)std::min<int64_t>((groups + 255) / 256, (int64_t)num_sms() * 32);
        k_merge_bidir<IO><<<mblocks, 256, 0, s>>>(s0, s1, reinterpret_cast<const IO *>(a.z),
                                                  reinterpret_cast<IO *>(a.out), rows, a.L, Lp,
                                                  FastDiv((uint32_t)((a.L + 3) / 4)));
        return check_launch("bidirectional merge");
    }

    // SS2D over maps whose rows (H*W values) are not 16-byte aligned, read in
    // place through VIEW tiles (C is a VIEW configuration; P = 1 << vshift rows
    // per view row): the transposed copy of u for the column directions, one
    // launch of the four directions side by side (grid z; the odd slots read
    // the copy), each storing y_k + D_k*u by scan step into its own fp32 slice
    // of pitch Lp, then one merge by step of the four slices, in a fixed order.
    static ss_status run_ss2d_view(const ScanArgs &a, int vshift) {
        using namespace ssk;
        using IO = typename C::IO;
        static_assert(C::VIEW && !C::VIEWZ, "a direction-pair VIEW configuration");
        const int io = a.io;
        const int P = 1 << vshift;
        const int64_t rows = a.batch * a.dim;
        const int64_t Lp = padded_len(a);
        cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
        float *acc0 = reinterpret_cast<float *>(a.ws);
        void *uT = reinterpret_cast<uint8_t *>(a.ws) + align256((size_t)4 * rows * Lp * sizeof(float));
        ss_status st;
        if ((st = permuted_copy(a, ORD_COL, uT))) return st;
        const uint64_t bcrows = (uint64_t)a.batch * 4 * a.G * C::N;
        const uint32_t bch = (uint32_t)(C::CB >> vshift), bbc = (uint32_t)(C::N >> vshift);
        CUtensorMap mu, mu2, md, mb, mc;
        if ((st = make_view_map(&mu, a.u, io, a.L, rows, P, C::BW, bch))) return st;
        if ((st = make_view_map(&mu2, uT, io, a.L, rows, P, C::BW, bch))) return st;
        if ((st = make_view_map(&md, a.delta, io, a.L, (uint64_t)rows * 4, P, C::BW, bch))) return st;
        if ((st = make_view_map(&mb, a.B, io, a.L, bcrows, P, C::BW, bbc))) return st;
        if ((st = make_view_map(&mc, a.C, io, a.L, bcrows, P, C::BW, bbc))) return st;
        auto kern = k_scan1d<C, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
        Scan1dParams p{};
        p.dim = a.dim;
        p.L = a.L;
        p.pitch = Lp;
        p.vshift = vshift;
        p.G = a.G;
        p.dpg = (int)(a.dim / a.G);
        p.Lc = a.L;
        p.J = 1;
        p.L0 = a.L;
        p.pass = 0;
        p.K = 4;
        p.u_g = a.u;
        p.A = a.A;
        p.D = a.D;
        p.bias = a.bias;
        p.softplus = a.softplus;
        p.has_z = 0;
        p.out = a.out;
        p.last_state = a.last_state;
        p.nz = 4;
        p.k0 = 0;
        for (int d = 0; d < 4; ++d) {
            const int o = a.orders[d];
            p.orders_z[d] = (o == ORD_ROW || o == ORD_COL) ? ORD_ROW : ORD_ROW_REV;
            p.modes_z[d] = OUT_STEP;
            p.accs_z[d] = acc0 + (int64_t)d * rows * Lp;
        }
        const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
        const unsigned bgs = (unsigned)(a.batch * a.G);
        kern<<<dim3(cblocks, bgs, 4), C::THREADS, C::SMEM, s>>>(mu, md, mu, mb, mc, mu2, p);
        if ((st = check_launch("four-direction scan"))) return st;
        OrderSet os{};
        os.K = 4;
        os.H = (int)a.H;
        os.W = (int)a.W;
        os.win = 0;
        for (int k = 0; k < 4; ++k) os.orders[k] = a.orders[k];
        os.pitch = Lp;
        const unsigned bx = (unsigned)((a.L + 255) / 256);
        const int64_t want_y = std::max<int64_t>(1, (int64_t)num_sms() * 32 / bx);
        const unsigned by = (unsigned)std::min<int64_t>({rows, want_y, (int64_t)65535});
        k_merge_steps<IO><<<dim3(bx, by), 256, 0, s>>>(acc0, rows, reinterpret_cast<const IO *>(a.z),
                                                      reinterpret_cast<IO *>(a.out), os);
        return check_launch("merge by step");
    }

    // K directions of any order: each launch stores its direction's y_k + D_k*u
    // by scan step into its own fp32 accumulator; one merge inverts the
    // traversals and sums by position.
    static ss_status run_steps(const ScanArgs &a) {
        using namespace ssk;
        const int io = a.io;
        const int64_t rows = a.batch * a.dim;
        const int K = a.K;
        CUtensorMap mu, md, mz, mb, mc;
        ss_status st;
        if ((st = make_map(&mu, a.u, io, a.L, rows, C::T, C::CB))) return st;
        if ((st = make_map(&md, a.delta, io, a.L, (uint64_t)rows * K, C::T, C::CB))) return st;
        if ((st = make_map(&mz, a.z ? a.z : a.u, io, a.L, rows, C::T, C::CB))) return st;
        const uint64_t bcrows = (uint64_t)a.batch * K * a.G * C::N;
        if ((st = make_map(&mb, a.B, io, a.L, bcrows, C::T, C::N))) return st;
        if ((st = make_map(&mc, a.C, io, a.L, bcrows, C::T, C::N))) return st;
        // Directions read u as row-order tiles: of u itself (row orders), or of
        // a copy permuted into their base traversal's step order (made once per
        // call, after the accumulators), forward or back to front.
        CUtensorMap umaps[4];
        umaps[0] = mu;
        int slot[4];
        steps_copy_slots(a, slot);
        uint8_t *copies = reinterpret_cast<uint8_t *>(a.ws) + steps_acc_bytes(a);
        const size_t copyb = steps_copy_bytes(a);
        for (int b = 1; b < 4; ++b) {
            if (slot[b] < 0) continue;
            void *dst = copies + (size_t)slot[b] * copyb;
            if ((st = permuted_copy(a, kBaseOrder[b], dst))) return st;
            if ((st = make_map(&umaps[b], dst, io, a.L, rows, C::T, C::CB))) return st;
        }
        auto kern = k_scan1d<C, true>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
            return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
        Scan1dParams p{};
        p.dim = a.dim;
        p.L = a.L;
        p.pitch = a.L;
        p.G = a.G;
        p.dpg = (int)(a.dim / a.G);
        p.Lc = a.L;
        p.J = 1;
        p.L0 = a.L;
        p.pass = 0;
        p.K = K;
        p.u_g = a.u;
        p.z_g = a.z;
        p.A = a.A;
        p.D = a.D;
        p.bias = a.bias;
        p.softplus = a.softplus;
        p.has_z = a.z != nullptr;
        p.out = a.out;
        p.last_state = a.last_state;
        const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
        const unsigned bgs = (unsigned)(a.batch * a.G);
        cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
        float *acc0 = reinterpret_cast<float *>(a.ws);
        // directions two at a time, side by side (grid z), for twice the warps
        for (int k = 0; k < K; k += 2) {
            const int nz = (k + 1 < K) ? 2 : 1;
            p.nz = nz;
            p.k0 = k;
            const CUtensorMap *um[2];
            for (int d = 0; d < 2; ++d) {
                const int kk = (d < nz) ? k + d : k;
                p.orders_z[d] = order_reversed(a.orders[kk]) ? ORD_ROW_REV : ORD_ROW;
                p.modes_z[d] = OUT_STEP;
                p.accs_z[d] = acc0 + (int64_t)kk * rows * a.L;
                um[d] = &umaps[order_base(a.orders[kk])];
            }
            kern<<<dim3(cblocks, bgs, (unsigned)nz), C::THREADS, C::SMEM, s>>>(*um[0], md, mz, mb, mc,
                                                                              *um[1], p);
            if ((st = check_launch("direction scan"))) return st;
        }
        using IO = typename C::IO;
        OrderSet os{};
        os.K = K;
        os.H = (int)a.H;
        os.W = (int)a.W;
        os.win = a.win;
        for (int k = 0; k < K; ++k) os.orders[k] = a.orders[k];
        os.pitch = a.L;
        const unsigned bx = (unsigned)((a.L + 255) / 256);
        const int64_t want_y = std::max<int64_t>(1, (int64_t)num_sms() * 32 / bx);
        const unsigned by = (unsigned)std::min<int64_t>({rows, want_y, (int64_t)65535});
        k_merge_steps<IO><<<dim3(bx, by), 256, 0, s>>>(acc0, rows, reinterpret_cast<const IO *>(a.z),
                                                      reinterpret_cast<IO *>(a.out), os);
        return check_launch("merge by step");
    }

    // CTAs of the plain scan kernel resident on one SM (registers and shared
    // memory), the slots the chunked passes fill.
    static int slots_per_sm() {
        static int cached = 0;
        if (cached > 0) return cached;
        int nb = 0;
        auto kern = ssk::k_scan1d<C, false, false>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, C::THREADS, C::SMEM) !=
                cudaSuccess ||
            nb < 1) {
            cudaGetLastError();  // no device: one CTA per SM
            return 1;
        }
        cached = nb;
        return nb;
    }
};

// Configuration per (I/O type, N): NPT states per lane, W warps per CTA, a
// 3-stage TMA ring, CL channels per lane (CL > 1 reuses each B/C value read
// from shared memory for several channels).
template <typename IO, int N>
struct Pick1d;
template <typename IO> struct Pick1d<IO, 1> { using C = ssk::Cfg1<IO, 1, 1, 2, 3, 1, 1>; };
template <typename IO> struct Pick1d<IO, 2> { using C = ssk::Cfg1<IO, 2, 2, 2, 3, 1, 1>; };
template <typename IO> struct Pick1d<IO, 4> { using C = ssk::Cfg1<IO, 4, 4, 2, 3, 1, 1>; };
template <typename IO> struct Pick1d<IO, 8> { using C = ssk::Cfg1<IO, 8, 4, 4, 3, 1, 1>; };
template <typename IO> struct Pick1d<IO, 16> { using C = ssk::Cfg1<IO, 16, 4, 4, 3, 1, 1>; };
template <typename IO> struct Pick1d<IO, 32> { using C = ssk::Cfg1<IO, 32, 4, 4, 3, 1, 1>; };
template <typename IO> struct Pick1d<IO, 64> { using C = ssk::Cfg1<IO, 64, 8, 4, 3, 1, 1>; };

// L-chunks to use: 1 (direct) when the direct path gives every SM sub-partition
// at least two warps.  Otherwise, when one L-chunk's CTAs fill at most half the
// GPU's slots, enough middle chunks for about kMidWaves waves of the slots that
// the long first and last chunks leave free (chunk_geom); else enough chunks
// for about twelve warps per sub-partition (the chunked path rescans all but
// the first chunk, so it only pays off when the direct path would leave the
// sub-partitions short of warps).  On the B300 the 1 x 5120 x 131072 scan
// measured 5.52 ms at 12 equal chunks, 5.61 at 10, 5.62 at 8, 5.84 at 14 and
// 16, 6.04 at 4.
constexpr double kMidWaves = 6.0;

template <class C>
int choose_chunks(const ScanArgs &a) {
    const int64_t rows = a.batch * a.dim;
    const int64_t threads = rows * C::R / C::CL;
    const int64_t one_per_smsp = (int64_t)num_sms() * 4 * 32;
    if (threads >= 2 * one_per_smsp) return 1;
    int64_t J = (12 * one_per_smsp + threads - 1) / threads;
    const int64_t R = (a.dim / a.G + C::CB - 1) / C::CB * a.batch * a.G;
    const int64_t S = (int64_t)num_sms() * Scan1d<C>::slots_per_sm();
    if (2 * R <= S) J = 2 + (int64_t)std::ceil(kMidWaves * (double)(S - R) / (double)R);
    const int64_t maxJ = a.L / (4 * C::T);  // keep L-chunks at least 4 T-chunks long
    if (J > maxJ) J = maxJ;
    return J < 2 ? 1 : (int)J;
}

template <typename IO, int N>
int chunks_for(const ScanArgs &a) {
    using C = typename Pick1d<IO, N>::C;
    const int J = a.chunks > 0 ? a.chunks : choose_chunks<C>(a);
    const int64_t R = (a.dim / a.G + C::CB - 1) / C::CB * a.batch * a.G;
    return chunk_geom(a.L, J, R, (int64_t)num_sms() * Scan1d<C>::slots_per_sm(), C::T).J;
}

template <typename IO, int N>
ss_status dispatch1d(const ScanArgs &a) {
    using C = typename Pick1d<IO, N>::C;
    return Scan1d<C>::run(a, chunks_for<IO, N>(a));
}

template <typename IO, int N>
ss_status dispatch_dirs(const ScanArgs &a) {
    using C = typename Pick1d<IO, N>::C;
    return Scan1d<C>::run_dirs(a);
}

template <typename IO, int N>
ss_status dispatch_bidir_padded(const ScanArgs &a) {
    using C = typename Pick1d<IO, N>::C;
    return Scan1d<C>::run_bidir_padded(a);
}

// The VIEW configuration of a (I/O type, N) configuration: a 2-stage ring, and
// twice the warps when a CTA has at most 32 channels.  A VIEW chunk takes P
// boxes per tensor and the copy engine's time goes by boxes, so more channels
// per box pays: on the Vision Mamba shape 328 us a call with 8 warps of 64
// channels, 338 with 4 warps, 350 with 16 (a third ring stage: no faster).
template <class C>
using ViewCfg = ssk::Cfg1<typename C::IO, C::N, C::NPT, (C::CB <= 32 ? 2 * C::W : C::W), 2, C::CL,
                          C::PIPE ? 1 : 0, 0, 1>;
// two CTAs of 8 warps per SM (by shared memory) for the Vision Mamba shape's configuration
static_assert(ViewCfg<Pick1d<__nv_bfloat16, 16>::C>::SMEM + 1024 <= 228 * 1024 / 2,
              "VIEW tiles of N = 16 fit two CTAs per SM");

template <typename IO, int N>
ss_status dispatch_bidir_view(const ScanArgs &a, int vshift) {
    using C = ViewCfg<typename Pick1d<IO, N>::C>;
    return a.K == 4 ? Scan1d<C>::run_ss2d_view(a, vshift) : Scan1d<C>::run_bidir_view(a, vshift);
}

template <typename IO>
ss_status dispatch_bidir_view_n(const ScanArgs &a, int vshift) {
    switch (a.N) {
    case 2: return dispatch_bidir_view<IO, 2>(a, vshift);
    case 4: return dispatch_bidir_view<IO, 4>(a, vshift);
    case 8: return dispatch_bidir_view<IO, 8>(a, vshift);
    case 16: return dispatch_bidir_view<IO, 16>(a, vshift);
    case 32: return dispatch_bidir_view<IO, 32>(a, vshift);
    case 64: return dispatch_bidir_view<IO, 64>(a, vshift);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d cannot be read through VIEW tiles", a.N);
    }
}

template <typename IO>
ss_status dispatch_bidir_padded_n(const ScanArgs &a) {
    switch (a.N) {
    case 1: return dispatch_bidir_padded<IO, 1>(a);
    case 2: return dispatch_bidir_padded<IO, 2>(a);
    case 4: return dispatch_bidir_padded<IO, 4>(a);
    case 8: return dispatch_bidir_padded<IO, 8>(a);
    case 16: return dispatch_bidir_padded<IO, 16>(a);
    case 32: return dispatch_bidir_padded<IO, 32>(a);
    case 64: return dispatch_bidir_padded<IO, 64>(a);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not one of 1,2,4,8,16,32,64", a.N);
    }
}

template <typename IO, int N>
ss_status dispatch_steps(const ScanArgs &a) {
    using C = typename Pick1d<IO, N>::C;
    return Scan1d<C>::run_steps(a);
}

template <typename IO>
ss_status dispatch_steps_n(const ScanArgs &a) {
    switch (a.N) {
    case 1: return dispatch_steps<IO, 1>(a);
    case 2: return dispatch_steps<IO, 2>(a);
    case 4: return dispatch_steps<IO, 4>(a);
    case 8: return dispatch_steps<IO, 8>(a);
    case 16: return dispatch_steps<IO, 16>(a);
    case 32: return dispatch_steps<IO, 32>(a);
    case 64: return dispatch_steps<IO, 64>(a);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not one of 1,2,4,8,16,32,64", a.N);
    }
}

template <typename IO, int N>
size_t ws1d(const ScanArgs &a) {
    const int J = chunks_for<IO, N>(a);
    if (J <= 1) return 0;
    const int64_t rows = a.batch * a.dim;
    return (size_t)rows * J * (2 * N + 1) * sizeof(float);
}

// The single-direction VIEW configuration of a (I/O type, N) configuration: a
// z tile and the gate in the prep, a 2-stage ring, the warps of the aligned
// configuration (the direct path's few CTAs per SM need its registers).
template <class C>
using ViewCfgZ = ssk::Cfg1<typename C::IO, C::N, C::NPT, C::W, 2, C::CL, C::PIPE ? 1 : 0, 0, 2>;

// One direction over rows read through views: chunked when the caller's
// workspace holds the chunked path's, else in one pass.
template <typename IO, int N>
ss_status dispatch1d_view(const ScanArgs &a, int vshift) {
    using C = ViewCfgZ<typename Pick1d<IO, N>::C>;
    int J = chunks_for<IO, N>(a);
    if (J > 1 && (!a.ws || a.ws_bytes < ws1d<IO, N>(a))) J = 1;
    return Scan1d<C>::run(a, J, vshift);
}

template <typename IO>
ss_status dispatch1d_view_n(const ScanArgs &a, int vshift) {
    switch (a.N) {
    case 2: return dispatch1d_view<IO, 2>(a, vshift);
    case 4: return dispatch1d_view<IO, 4>(a, vshift);
    case 8: return dispatch1d_view<IO, 8>(a, vshift);
    case 16: return dispatch1d_view<IO, 16>(a, vshift);
    case 32: return dispatch1d_view<IO, 32>(a, vshift);
    case 64: return dispatch1d_view<IO, 64>(a, vshift);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d cannot be read through VIEW tiles", a.N);
    }
}


// ---------------------------------------------------------------- multi direction
template <class C>
ss_status run_multi(const ScanArgs &a) {
    using namespace ssk;
    const int64_t smem = C::smem_bytes(a.L);
    int dev = 0, maxsm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&maxsm, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (smem > maxsm)
        return fail(SS_ERR_UNSUPPORTED,
                    "sequence of %lld positions needs %lld bytes of shared memory (limit %d)",
                    (long long)a.L, (long long)smem, maxsm);
    auto kern = k_multidir<C>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return fail(SS_ERR_CUDA, "cannot reserve %lld bytes of shared memory", (long long)smem);
    MultiParams p{};
    p.dim = a.dim;
    p.L = a.L;
    p.H = (int)a.H;
    p.W = (int)a.W;
    p.G = a.G;
    p.dpg = (int)(a.dim / a.G);
    for (int k = 0; k < 4; ++k) p.orders[k] = a.orders[k];
    p.divH = FastDiv((uint32_t)a.H);
    p.u = a.u;
    p.delta = a.delta;
    p.B = a.B;
    p.C = a.C;
    p.z = a.z;
    p.A = a.A;
    p.D = a.D;
    p.bias = a.bias;
    p.softplus = a.softplus;
    p.out = a.out;
    p.zoh = a.zoh;
    p.h0 = a.h0;
    p.last_state = a.last_state;
    const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
    kern<<<dim3(cblocks, (unsigned)(a.batch * a.G), 1), C::THREADS, (size_t)smem, s>>>(p);
    return check_launch("multi-direction scan");
}

// NPT states per lane (at most 8 lanes per channel); WPD warps per direction.
template <typename IO, int N, int K>
struct PickM;
template <typename IO, int K> struct PickM<IO, 1, K> { using C = ssk::CfgM<IO, 1, 1, K, 1>; };
template <typename IO, int K> struct PickM<IO, 2, K> { using C = ssk::CfgM<IO, 2, 1, K, (K == 4 ? 1 : 4)>; };
template <typename IO, int K> struct PickM<IO, 4, K> { using C = ssk::CfgM<IO, 4, 2, K, (K == 4 ? 1 : 4)>; };
template <typename IO, int K> struct PickM<IO, 8, K> { using C = ssk::CfgM<IO, 8, 2, K, (K == 4 ? 1 : 2)>; };
template <typename IO, int K> struct PickM<IO, 16, K> { using C = ssk::CfgM<IO, 16, 2, K, (K == 4 ? 1 : 4), 16>; };
template <typename IO, int K> struct PickM<IO, 32, K> { using C = ssk::CfgM<IO, 32, 4, K, (K == 4 ? 1 : 2)>; };
template <typename IO, int K> struct PickM<IO, 64, K> { using C = ssk::CfgM<IO, 64, 8, K, (K == 4 ? 1 : 2)>; };

template <typename IO, int K>
ss_status dispatch_multi_n(const ScanArgs &a) {
    switch (a.N) {
    case 1: return run_multi<typename PickM<IO, 1, K>::C>(a);
    case 2: return run_multi<typename PickM<IO, 2, K>::C>(a);
    case 4: return run_multi<typename PickM<IO, 4, K>::C>(a);
    case 8: return run_multi<typename PickM<IO, 8, K>::C>(a);
    case 16: return run_multi<typename PickM<IO, 16, K>::C>(a);
    case 32: return run_multi<typename PickM<IO, 32, K>::C>(a);
    case 64: return run_multi<typename PickM<IO, 64, K>::C>(a);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not supported on this path", a.N);
    }
}

template <typename IO>
ss_status dispatch_multi(const ScanArgs &a) {
    switch (a.K) {
    case 1: return dispatch_multi_n<IO, 1>(a);
    case 2: return dispatch_multi_n<IO, 2>(a);
    case 4: return dispatch_multi_n<IO, 4>(a);
    default: return fail(SS_ERR_INVALID_ARG, "directions must be 1, 2 or 4");
    }
}

template <typename IO>
ss_status dispatch1d_n(const ScanArgs &a) {
    switch (a.N) {
    case 1: return dispatch1d<IO, 1>(a);
    case 2: return dispatch1d<IO, 2>(a);
    case 4: return dispatch1d<IO, 4>(a);
    case 8: return dispatch1d<IO, 8>(a);
    case 16: return dispatch1d<IO, 16>(a);
    case 32: return dispatch1d<IO, 32>(a);
    case 64: return dispatch1d<IO, 64>(a);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not one of 1,2,4,8,16,32,64", a.N);
    }
}

template <typename IO>
ss_status dispatch_dirs_n(const ScanArgs &a) {
    switch (a.N) {
    case 1: return dispatch_dirs<IO, 1>(a);
    case 2: return dispatch_dirs<IO, 2>(a);
    case 4: return dispatch_dirs<IO, 4>(a);
    case 8: return dispatch_dirs<IO, 8>(a);
    case 16: return dispatch_dirs<IO, 16>(a);
    case 32: return dispatch_dirs<IO, 32>(a);
    case 64: return dispatch_dirs<IO, 64>(a);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not one of 1,2,4,8,16,32,64", a.N);
    }
}

template <typename IO>
size_t ws1d_n(const ScanArgs &a) {
    switch (a.N) {
    case 1: return ws1d<IO, 1>(a);
    case 2: return ws1d<IO, 2>(a);
    case 4: return ws1d<IO, 4>(a);
    case 8: return ws1d<IO, 8>(a);
    case 16: return ws1d<IO, 16>(a);
    case 32: return ws1d<IO, 32>(a);
    case 64: return ws1d<IO, 64>(a);
    default: return 0;
    }
}

}  // namespace

// The TMA path needs 16-byte aligned rows: seqlen * element size % 16 == 0.
bool scan1d_uses_tma(const ScanArgs &a) {
    const int64_t es = (a.io == SS_BF16) ? 2 : 4;
    return (a.L * es) % 16 == 0 && a.batch * a.dim < (1ll << 31) &&
           a.batch * a.G * a.N < (1ll << 31) && a.L < (1ll << 31);
}

// log2 of the rows folded into one view row for a call over rows that are not
// 16-byte aligned, or -1: P = (16 / element size) / gcd(L, 16 / element size)
// must divide the channels per group and N (so that every box holds whole rows
// of one channel block or one B/C tile), and the view's sizes fit its map.
int view_fold_shift(const ScanArgs &a) {
    const int64_t vpc = a.io == SS_BF16 ? 8 : 4;  // values per 16 bytes (a power of two)
    int64_t g = 1;
    while (g < vpc && a.L % (2 * g) == 0) g *= 2;  // gcd(L, vpc)
    const int64_t P = vpc / g;
    const int64_t dpg = a.dim / a.G;
    if (P < 2 || dpg % P != 0 || a.N % P != 0) return -1;
    if (P * a.L >= (1ll << 31) || (int64_t)a.K * a.batch * a.dim >= (1ll << 31) ||
        (int64_t)a.K * a.batch * a.G * a.N >= (1ll << 31))
        return -1;
    return P == 2 ? 1 : P == 4 ? 2 : 3;
}

// One direction over rows that are not 16-byte aligned, without the zero-order
// hold or the fused Conv1D: read through views (else the on-chip kernel).
int scan1d_view_shift(const ScanArgs &a) {
    if (scan1d_uses_tma(a) || a.zoh || a.conv || a.N < 2) return -1;
    return view_fold_shift(a);
}

size_t scan1d_workspace_bytes(const ScanArgs &a) {
    // rows read through views may take the chunked path too (their workspace
    // is optional: without it they run in one pass)
    if (!scan1d_uses_tma(a) && scan1d_view_shift(a) < 0) return 0;
    return a.io == SS_BF16 ? ws1d_n<__nv_bfloat16>(a) : ws1d_n<float>(a);
}

ss_status launch_scan1d(const ScanArgs &a) {
    if (!scan1d_uses_tma(a)) {
        const int vshift = scan1d_view_shift(a);
        if (vshift > 0)
            return a.io == SS_BF16 ? dispatch1d_view_n<__nv_bfloat16>(a, vshift)
                                   : dispatch1d_view_n<float>(a, vshift);
        ScanArgs m = a;
        m.K = 1;
        m.H = 1;
        m.W = a.L;
        m.orders[0] = ORD_ROW;
        return a.io == SS_BF16 ? dispatch_multi<__nv_bfloat16>(m) : dispatch_multi<float>(m);
    }
    return a.io == SS_BF16 ? dispatch1d_n<__nv_bfloat16>(a) : dispatch1d_n<float>(a);
}

// Bidirectional calls over rows that are not 16-byte aligned re-pitch their
// inputs when the row counts fit the TMA maps (else they merge on chip).
bool bidir_padded_ok(const ScanArgs &a) {
    if (a.K != 2 || scan1d_uses_tma(a)) return false;
    const int64_t rows = a.batch * a.dim;
    return 2 * rows < (1ll << 31) && a.batch * 2 * a.G * a.N < (1ll << 31) && a.L < (1ll << 30);
}

// log2 of the rows folded into one view row for a bidirectional call read in
// place through VIEW tiles, or -1 when the call cannot take that path: its rows
// are 16-byte aligned, or P does not divide the channels per group or N (so
// that every box holds whole rows of one channel block or one B/C tile).
int bidir_view_shift(const ScanArgs &a) {
    if (!bidir_padded_ok(a)) return -1;
    return view_fold_shift(a);
}
// Workspace of the VIEW path: the two directions' fp32 slices [2, rows, Lp].
size_t bidir_view_bytes(const ScanArgs &a) {
    return align256((size_t)2 * a.batch * a.dim * padded_len(a) * sizeof(float));
}

// SS2D over maps whose rows are not 16-byte aligned, read through VIEW tiles
// (else the on-chip kernel): log2 of the rows to a view row, or -1.
int ss2d_view_shift(const ScanArgs &a) {
    if (a.K != 4 || scan1d_uses_tma(a)) return -1;
    for (int k = 0; k < 4; ++k)
        if (a.orders[k] > ORD_COL_REV) return -1;
    return view_fold_shift(a);
}
// Workspace of that path: four fp32 slices [rows, Lp] and the transposed copy of u.
size_t ss2d_view_bytes(const ScanArgs &a) {
    const int64_t rows = a.batch * a.dim;
    return align256((size_t)4 * rows * padded_len(a) * sizeof(float)) +
           align256((size_t)rows * a.L * (a.io == SS_BF16 ? 2 : 4));
}

size_t multidir_workspace_bytes(const ScanArgs &a) {
    if (bidir_padded_ok(a)) return bidir_padded_bytes(a);
    if (ss2d_view_shift(a) > 0) return ss2d_view_bytes(a);  // optional: else on chip
    if (!scan1d_uses_tma(a)) return 0;  // rows not 16-byte aligned: on-chip merge path
    // one fp32 accumulator; SS2D scans its four directions side by side into
    // four fp32 slices, and reads u of its column directions from a transposed
    // copy (sized as an fp32 map, for either dtype)
    const size_t map = (size_t)a.batch * a.dim * a.L * sizeof(float);
    return a.K == 4 ? 5 * map : map;
}

size_t steps_workspace_bytes(const ScanArgs &a) {
    int slot[4];
    return steps_acc_bytes(a) + (size_t)steps_copy_slots(a, slot) * steps_copy_bytes(a);
}

ss_status launch_steps(const ScanArgs &a) {
    return a.io == SS_BF16 ? dispatch_steps_n<__nv_bfloat16>(a) : dispatch_steps_n<float>(a);
}

ss_status launch_multidir(const ScanArgs &a) {
    if (bidir_padded_ok(a)) {
        // rows read in place through VIEW tiles, or re-pitched, when the caller
        // gave the workspace; else on chip
        const int vshift = bidir_view_shift(a);
        if (vshift > 0 && a.ws && a.ws_bytes >= bidir_view_bytes(a))
            return a.io == SS_BF16 ? dispatch_bidir_view_n<__nv_bfloat16>(a, vshift)
                                   : dispatch_bidir_view_n<float>(a, vshift);
        if (a.ws && a.ws_bytes >= bidir_padded_bytes(a))
            return a.io == SS_BF16 ? dispatch_bidir_padded_n<__nv_bfloat16>(a)
                                   : dispatch_bidir_padded_n<float>(a);
        return a.io == SS_BF16 ? dispatch_multi<__nv_bfloat16>(a) : dispatch_multi<float>(a);
    }
    if (!scan1d_uses_tma(a)) {
        // SS2D over unaligned rows: view tiles when the caller gave the
        // workspace, else on chip
        const int vshift = ss2d_view_shift(a);
        if (vshift > 0 && a.ws && a.ws_bytes >= ss2d_view_bytes(a))
            return a.io == SS_BF16 ? dispatch_bidir_view_n<__nv_bfloat16>(a, vshift)
                                   : dispatch_bidir_view_n<float>(a, vshift);
        return a.io == SS_BF16 ? dispatch_multi<__nv_bfloat16>(a) : dispatch_multi<float>(a);
    }
    if (multidir_workspace_bytes(a) > 0)
        return a.io == SS_BF16 ? dispatch_dirs_n<__nv_bfloat16>(a) : dispatch_dirs_n<float>(a);
    return a.io == SS_BF16 ? dispatch_multi<__nv_bfloat16>(a) : dispatch_multi<float>(a);
}

namespace {
template <typename IO>
ss_status launch_step_io(const ScanArgs &a, float *state) {
    ssk::StepParams p{};
    p.rows = a.batch * a.dim;
    p.dim = a.dim;
    p.G = a.G;
    p.dpg = (int)(a.dim / a.G);
    p.x = a.u;
    p.delta = a.delta;
    p.B = a.B;
    p.C = a.C;
    p.z = a.z;
    p.A = a.A;
    p.D = a.D;
    p.bias = a.bias;
    p.softplus = a.softplus;
    p.zoh = a.zoh;
    p.state = state;
    p.out = a.out;
    const unsigned blocks = (unsigned)((p.rows + 127) / 128);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(a.stream);
    switch (a.N) {
    case 1: ssk::k_step<IO, 1><<<blocks, 128, 0, s>>>(p); break;
    case 2: ssk::k_step<IO, 2><<<blocks, 128, 0, s>>>(p); break;
    case 4: ssk::k_step<IO, 4><<<blocks, 128, 0, s>>>(p); break;
    case 8: ssk::k_step<IO, 8><<<blocks, 128, 0, s>>>(p); break;
    case 16: ssk::k_step<IO, 16><<<blocks, 128, 0, s>>>(p); break;
    case 32: ssk::k_step<IO, 32><<<blocks, 128, 0, s>>>(p); break;
    case 64: ssk::k_step<IO, 64><<<blocks, 128, 0, s>>>(p); break;
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not one of 1,2,4,8,16,32,64", a.N);
    }
    return check_launch("state update");
}
}  // namespace

ss_status launch_step(const ScanArgs &a, float *state) {
    return a.io == SS_BF16 ? launch_step_io<__nv_bfloat16>(a, state) : launch_step_io<float>(a, state);
}

// ---------------------------------------------------------------- backward
namespace {
// Checkpoint workspace: every configuration checkpoints every 8 or 16 steps; the
// workspace is sized for 8.
constexpr int kBwdMinBlock = 8;

// MULTI: directions ks[0..nz) of a multi-direction call, side by side (ckpt and
// du_acc from the caller), reading u, z, dout from the maps given here (the
// call's own tensors, or copies permuted into the directions' step order), in
// the row order or its reverse (`ords`); otherwise the single direction with its
// checkpoints in a.ws.
struct DirLaunch {
    int nz = 1;
    int ks[2] = {0, 0}, ords[2] = {0, 0};
    const void *u = nullptr, *z = nullptr, *dout = nullptr;
};

template <class C, bool MULTI = false, bool EXT = false>
ss_status run_scan_bwd(const BwdArgs &a, const DirLaunch &dl = DirLaunch(), float *ckpt = nullptr,
                       float *du_acc = nullptr) {
    const int nz = MULTI ? dl.nz : 1;
    using namespace ssk;
    static_assert(C::TS >= kBwdMinBlock, "checkpoint interval");
    const ScanArgs &f = a.f;
    const int io = f.io;
    const int64_t rows = f.batch * f.dim;
    const int K = MULTI ? f.K : 1;
    const uint64_t bcrows = (uint64_t)f.batch * K * f.G * C::N;
    CUtensorMap mu, md, mz, mdy, mb, mc;
    ss_status st;
    const void *tu = MULTI ? dl.u : f.u, *tz = MULTI ? dl.z : f.z, *tdy = MULTI ? dl.dout : a.dout;
    if ((st = make_map(&mu, tu, io, f.L, rows, C::T, C::CB))) return st;
    if ((st = make_map(&md, f.delta, io, f.L, (uint64_t)rows * K, C::T, C::CB))) return st;
    if ((st = make_map(&mz, tz ? tz : tu, io, f.L, rows, C::T, C::CB))) return st;
    if ((st = make_map(&mdy, tdy, io, f.L, rows, C::T, C::CB))) return st;
    if ((st = make_map(&mb, f.B, io, f.L, bcrows, C::T, C::N))) return st;
    if ((st = make_map(&mc, f.C, io, f.L, bcrows, C::T, C::N))) return st;
    auto kern = k_scan_bwd<C, MULTI, EXT>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess)
        return fail(SS_ERR_CUDA, "cannot reserve %d bytes of shared memory", C::SMEM);
    BwdParams p{};
    p.K = K;
    for (int j = 0; j < 2; ++j) {
        const int jj = j < nz ? j : 0;
        p.k_z[j] = MULTI ? dl.ks[jj] : 0;
        p.order_z[j] = MULTI ? dl.ords[jj] : 0;
    }
    p.du_acc = du_acc;
    p.du_zstride = rows * f.L;
    p.dim = f.dim;
    p.L = f.L;
    p.G = f.G;
    p.dpg = (int)(f.dim / f.G);
    p.nblk = (int)((f.L + C::TS - 1) / C::TS);
    p.ck_zstride = rows * p.nblk * C::N;
    p.A = f.A;
    p.D = f.D;
    p.bias = f.bias;
    p.softplus = f.softplus;
    p.has_z = f.z != nullptr;
    p.ckpt = MULTI ? ckpt : reinterpret_cast<float *>(a.ws);
    p.du = a.du;
    p.ddelta = a.ddelta;
    p.dz = a.dz;
    p.dA = a.dA;
    p.dB = a.dB;
    p.dC = a.dC;
    p.dD = a.dD;
    p.dbias = a.dbias;
    p.zoh = f.zoh;
    p.h0 = f.h0;
    p.dh0 = a.dh0;
    if (!MULTI) {
        p.du_acc = a.du_f32;  // nullable: du in the I/O type otherwise
        p.du_zstride = 0;
    }
    const unsigned cblocks = (unsigned)((p.dpg + C::CB - 1) / C::CB);
    const unsigned bgs = (unsigned)(f.batch * f.G);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(f.stream);
    kern<<<dim3(cblocks, bgs, (unsigned)nz), C::THREADS, C::SMEM, s>>>(mu, md, mz, mdy, mb, mc, p);
    return check_launch("scan backward");
}

template <typename IO, bool MULTI = false, bool EXT = false>
ss_status dispatch_bwd(const BwdArgs &a, const DirLaunch &dl = DirLaunch(), float *ckpt = nullptr,
                       float *du_acc = nullptr) {
    using namespace ssk;
    // CfgB<IO, N, warps per CTA, channels per lane, states per lane, steps per
    // block, CTAs per SM for the register budget>
    // float32 I/O has twice the prep registers: a budget of two CTAs per SM
    constexpr int MB = sizeof(IO) == 2 ? 3 : 2;
    switch (a.f.N) {
    case 1: return run_scan_bwd<CfgB<IO, 1, 2, 1, 4, 16, 2>, MULTI, EXT>(a, dl, ckpt, du_acc);
    case 2: return run_scan_bwd<CfgB<IO, 2, 2, 1, 4, 16, 2>, MULTI, EXT>(a, dl, ckpt, du_acc);
    case 4: return run_scan_bwd<CfgB<IO, 4, 2, 1, 4, 16, 2>, MULTI, EXT>(a, dl, ckpt, du_acc);
    case 8: return run_scan_bwd<CfgB<IO, 8, 2, 1, 4, 16, MB>, MULTI, EXT>(a, dl, ckpt, du_acc);
    case 16: return run_scan_bwd<CfgB<IO, 16, 4, 1, 4, 16, MB>, MULTI, EXT>(a, dl, ckpt, du_acc);
    case 32: return run_scan_bwd<CfgB<IO, 32, 4, 1, 4, 16, MB>, MULTI, EXT>(a, dl, ckpt, du_acc);
    case 64: return run_scan_bwd<CfgB<IO, 64, 4, 1, 4, 16, 2>, MULTI, EXT>(a, dl, ckpt, du_acc);
    default: return fail(SS_ERR_UNSUPPORTED, "dstate %d is not one of 1,2,4,8,16,32,64", a.f.N);
    }
}

ss_status zero_async(void *p, size_t bytes, cudaStream_t s) {
    if (!p || bytes == 0) return SS_OK;
    const cudaError_t e = cudaMemsetAsync(p, 0, bytes, s);
    if (e != cudaSuccess) return fail(SS_ERR_CUDA, "cudaMemsetAsync failed: %s", cudaGetErrorString(e));
    return SS_OK;
}
}  // namespace

size_t scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t L, int N, bool conv) {
    if (batch <= 0 || dim <= 0 || L <= 0 || N <= 0) return 0;
    const size_t ck = (size_t)batch * dim * ((L + kBwdMinBlock - 1) / kBwdMinBlock) * N * sizeof(float);
    if (!conv) return ck;
    return align256(ck) + 2 * align256((size_t)batch * dim * L * sizeof(float));
}

namespace {
template <typename IO>
ss_status bwd_with_options(const BwdArgs &a) {
    using namespace ssk;
    const ScanArgs &f = a.f;
    const bool ext = f.zoh || f.h0;
    if (!f.conv) return ext ? dispatch_bwd<IO, false, true>(a) : dispatch_bwd<IO>(a);
    // the fused Conv1D: recompute its output u, run the scan's backward pass on
    // it into a du buffer, then turn du into the gradients of x, w, b and x0
    cudaStream_t s = reinterpret_cast<cudaStream_t>(f.stream);
    const int64_t rows = f.batch * f.dim;
    uint8_t *ws = reinterpret_cast<uint8_t *>(a.ws);
    const size_t ck = align256((size_t)rows * ((f.L + kBwdMinBlock - 1) / kBwdMinBlock) * f.N *
                               sizeof(float));
    void *um = ws + ck;
    void *dum = ws + ck + align256((size_t)rows * f.L * sizeof(float));
    ConvSiluParams cp{};
    cp.rows = rows;
    cp.dim = f.dim;
    cp.L = f.L;
    cp.x = f.u;
    cp.w = f.conv_w;
    cp.bias = f.conv_b;
    cp.x0 = f.conv_x0;
    cp.u = um;
    cp.du = reinterpret_cast<const float *>(dum);
    cp.dx = a.du;
    cp.dw = a.dconv_w;
    cp.dbias = a.dconv_b;
    cp.dx0 = a.dconv_x0;
    const int64_t n = rows * f.L;
    k_conv_silu_fwd<IO><<<(unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)num_sms() * 32), 256, 0, s>>>(cp);
    ss_status st = check_launch("conv1d forward");
    if (st) return st;
    BwdArgs b = a;
    b.f.u = um;
    b.du = dum;  // (unused: du goes to du_f32)
    b.du_f32 = reinterpret_cast<float *>(dum);
    st = dispatch_bwd<IO, false, true>(b);  // (the option instantiation writes du in fp32)
    if (st) return st;
    if ((st = zero_async(a.dconv_w, (size_t)f.dim * 4 * sizeof(float), s))) return st;
    if ((st = zero_async(a.dconv_b, (size_t)f.dim * sizeof(float), s))) return st;
    const dim3 grid((unsigned)((f.L + CONV_TS - 1) / CONV_TS), (unsigned)rows);
    k_conv_silu_bwd<IO><<<grid, CONV_TS, 0, s>>>(cp);
    return check_launch("conv1d backward");
}
}  // namespace

ss_status launch_scan_bwd(const BwdArgs &a, bool empty) {
    const ScanArgs &f = a.f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(f.stream);
    // outputs that are sums (over batch, time or channels) start from zero
    const size_t bc = (size_t)f.batch * f.G * f.N * f.L * sizeof(float);
    ss_status st;
    if ((st = zero_async(a.dA, (size_t)f.dim * f.N * sizeof(float), s))) return st;
    if ((st = zero_async(a.dB, bc, s))) return st;
    if ((st = zero_async(a.dC, bc, s))) return st;
    if ((st = zero_async(a.dD, (size_t)f.dim * sizeof(float), s))) return st;
    if ((st = zero_async(a.dbias, (size_t)f.dim * sizeof(float), s))) return st;
    if (empty) {
        // gradients of the options' tensors over an empty sequence
        if ((st = zero_async(a.dconv_w, (size_t)f.dim * 4 * sizeof(float), s))) return st;
        if ((st = zero_async(a.dconv_b, (size_t)f.dim * sizeof(float), s))) return st;
        if (f.L == 0 && a.dh0) {
            // no step: dh0 is zero (the state is not used)
            if ((st = zero_async(a.dh0, (size_t)f.batch * f.dim * f.N * sizeof(float), s))) return st;
        }
        if (f.L == 0 && a.dconv_x0)
            if ((st = zero_async(a.dconv_x0, (size_t)f.batch * f.dim * 3 * sizeof(float), s))) return st;
        return SS_OK;
    }
    return f.io == SS_BF16 ? bwd_with_options<__nv_bfloat16>(a) : bwd_with_options<float>(a);
}

ss_status launch_dwconv3x3(int64_t batch, int64_t dim, int64_t H, int64_t W, int io, const void *x,
                           const float *w, const float *bias, void *u, ss_stream_t stream) {
    using namespace ssk;
    const int64_t planes = batch * dim;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (W <= DWC_BAND_MAXW) {
        // bands of up to ~24 KB of fp32 rows (the whole plane when it fits)
        const int RB = (int)std::max<int64_t>(1, std::min<int64_t>(H, 6144 / (W + 2) - 2));
        const size_t smem = (size_t)(RB + 2) * (W + 2) * sizeof(float);
        const dim3 grid((unsigned)std::min<int64_t>(planes, (int64_t)num_sms() * 64),
                        (unsigned)((H + RB - 1) / RB));
        if (io == SS_BF16)
            k_dwconv3x3_silu_band<__nv_bfloat16><<<grid, DWC_THREADS, smem, s>>>(
                reinterpret_cast<const __nv_bfloat16 *>(x), w, bias,
                reinterpret_cast<__nv_bfloat16 *>(u), planes, (int)dim, (int)H, (int)W, RB);
        else
            k_dwconv3x3_silu_band<float><<<grid, DWC_THREADS, smem, s>>>(
                reinterpret_cast<const float *>(x), w, bias, reinterpret_cast<float *>(u), planes,
                (int)dim, (int)H, (int)W, RB);
        return check_launch("dwconv3x3");
    }
    const dim3 grid((unsigned)((W + DWC_TW - 1) / DWC_TW), (unsigned)((H + DWC_TH - 1) / DWC_TH),
                    (unsigned)std::min<int64_t>(planes, 65535));
    if (io == SS_BF16)
        k_dwconv3x3_silu<__nv_bfloat16><<<grid, DWC_THREADS, 0, s>>>(
            reinterpret_cast<const __nv_bfloat16 *>(x), w, bias, reinterpret_cast<__nv_bfloat16 *>(u),
            planes, (int)dim, (int)H, (int)W);
    else
        k_dwconv3x3_silu<float><<<grid, DWC_THREADS, 0, s>>>(reinterpret_cast<const float *>(x), w, bias,
                                                             reinterpret_cast<float *>(u), planes,
                                                             (int)dim, (int)H, (int)W);
    return check_launch("dwconv3x3");
}

size_t multi_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t L, int N, int K) {
    if (batch <= 0 || dim <= 0 || L <= 0 || N <= 0 || K <= 0) return 0;
    const size_t rows = (size_t)batch * dim;
    // the pre-gate output sum, the directions' du by step (first the forward
    // pass's accumulators), three map slots for the copies of u, dout and z in a
    // base traversal's step order (first the forward pass's copies of u), and two
    // checkpoint buffers (directions run two per launch)
    return align256(rows * L * 4) + align256((size_t)K * rows * L * 4) + 3 * align256(rows * L * 4) +
           align256(2 * rows * ((L + kBwdMinBlock - 1) / kBwdMinBlock) * N * sizeof(float));
}

ss_status launch_multi_bwd(const BwdArgs &a, bool empty) {
    using namespace ssk;
    const ScanArgs &f = a.f;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(f.stream);
    const int K = f.K;
    const size_t bc = (size_t)f.batch * K * f.G * f.N * f.L * sizeof(float);
    ss_status st;
    if ((st = zero_async(a.dA, (size_t)K * f.dim * f.N * sizeof(float), s))) return st;
    if ((st = zero_async(a.dB, bc, s))) return st;
    if ((st = zero_async(a.dC, bc, s))) return st;
    if ((st = zero_async(a.dD, (size_t)K * f.dim * sizeof(float), s))) return st;
    if ((st = zero_async(a.dbias, (size_t)K * f.dim * sizeof(float), s))) return st;
    if (empty) return SS_OK;
    const int64_t rows = f.batch * f.dim;
    uint8_t *ws = reinterpret_cast<uint8_t *>(a.ws);
    void *sbuf = ws;                                                   // pre-gate output sum
    float *duacc = reinterpret_cast<float *>(ws + align256((size_t)rows * f.L * 4));
    uint8_t *tmaps = reinterpret_cast<uint8_t *>(duacc) + align256((size_t)K * rows * f.L * 4);
    const size_t mapb = align256((size_t)rows * f.L * 4);
    float *ckpt = reinterpret_cast<float *>(tmaps + 3 * mapb);
    void *uT = tmaps, *dyT = tmaps + mapb, *zT = f.z ? (void *)(tmaps + 2 * mapb) : nullptr;
    if (f.z) {
        // dz needs the sum of all directions' outputs before the gate (its
        // accumulators and copies of u are followed by the transposed maps'
        // space, which is written only after it)
        ScanArgs fa = f;
        fa.z = nullptr;
        fa.out = sbuf;
        fa.last_state = nullptr;
        fa.ws = duacc;
        fa.ws_bytes = align256((size_t)K * rows * f.L * 4) + 3 * mapb;
        if ((st = launch_steps(fa))) return st;
    }
    // Every direction reads u, dout and z as row-order tiles, forward or back to
    // front: the call's own maps for the row orders, else copies permuted into
    // its base traversal's step order.  The bases take turns in the three maps'
    // space (stream order keeps a base's copies until its launches are done);
    // within a base, directions run two per launch (grid z), each with its own
    // checkpoints.
    for (int base = 0; base < 4; ++base) {
        int ks[8], n = 0;
        for (int k = 0; k < K; ++k)
            if (order_base(f.orders[k]) == base) ks[n++] = k;
        if (n == 0) continue;
        const void *tu = f.u, *tdy = a.dout, *tz = f.z;
        if (base != 0) {
            ScanArgs pa = f;
            const void *srcs[3] = {f.u, a.dout, f.z};
            void *dsts[3] = {uT, dyT, zT};
            for (int j = 0; j < 3; ++j) {
                if (!srcs[j]) continue;
                pa.u = srcs[j];
                if ((st = permuted_copy(pa, kBaseOrder[base], dsts[j]))) return st;
            }
            tu = uT;
            tdy = dyT;
            tz = zT;
        }
        for (int j = 0; j < n; j += 2) {
            DirLaunch dl;
            dl.nz = j + 1 < n ? 2 : 1;
            for (int q = 0; q < dl.nz; ++q) {
                dl.ks[q] = ks[j + q];
                dl.ords[q] = order_reversed(f.orders[ks[j + q]]) ? ORD_ROW_REV : ORD_ROW;
            }
            dl.u = tu;
            dl.dout = tdy;
            dl.z = tz;
            st = f.io == SS_BF16 ? dispatch_bwd<__nv_bfloat16, true>(a, dl, ckpt, duacc)
                                 : dispatch_bwd<float, true>(a, dl, ckpt, duacc);
            if (st) return st;
        }
    }
    BwdOrderSet os{};
    os.K = K;
    os.H = (int)f.H;
    os.W = (int)f.W;
    os.win = f.win;
    for (int k = 0; k < K; ++k) os.orders[k] = f.orders[k];
    const unsigned bx = (unsigned)((f.L + 255) / 256);
    const int64_t want_y = std::max<int64_t>(1, (int64_t)num_sms() * 32 / bx);
    const unsigned by = (unsigned)std::min<int64_t>({rows, want_y, (int64_t)65535});
    if (f.io == SS_BF16) {
        using IO = __nv_bfloat16;
        k_merge_bwd<IO><<<dim3(bx, by), 256, 0, s>>>(
            duacc, rows, os, reinterpret_cast<const IO *>(a.dout), reinterpret_cast<const IO *>(f.z),
            reinterpret_cast<const IO *>(sbuf), reinterpret_cast<IO *>(a.du), reinterpret_cast<IO *>(a.dz));
    } else {
        k_merge_bwd<float><<<dim3(bx, by), 256, 0, s>>>(
            duacc, rows, os, reinterpret_cast<const float *>(a.dout), reinterpret_cast<const float *>(f.z),
            reinterpret_cast<const float *>(sbuf), reinterpret_cast<float *>(a.du),
            reinterpret_cast<float *>(a.dz));
    }
    return check_launch("backward merge");
}

ss_status read_device_status(ss_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned int v = 0, zero = 0;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, ssk::g_status, sizeof(v));
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(ssk::g_status, &zero, sizeof(zero));
    if (e != cudaSuccess) return fail(SS_ERR_CUDA, "device status read failed: %s", cudaGetErrorString(e));
    if (v & 1u) return fail(SS_ERR_TIMEOUT, "a kernel abandoned a bounded wait (timeout)");
    return SS_OK;
}

// Scratch of ss_selective_scan_fwd_noalloc: fixed-size static device memory,
// present on every device that loads the library, shared by all its calls.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SS_NOALLOC_SCRATCH_BYTES];

// In host code g_noalloc_scratch names a host-side shadow, not device memory:
// the device address comes from cudaGetSymbolAddress, with the device current.
// It is looked up on every call (it allocates nothing and is cheap), so a
// context that was torn down and created again, which may place the array at a
// new address, never sees a stale pointer.
ss_status noalloc_scratch(void **ptr) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
        return fail(SS_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed: %s",
                    cudaGetErrorString(e));
    *ptr = p;
    return SS_OK;
}

ss_status set_debug_flags(unsigned int flags) {
    const cudaError_t e = cudaMemcpyToSymbol(ssk::g_debug_flags, &flags, sizeof(flags));
    if (e != cudaSuccess) return fail(SS_ERR_CUDA, "cannot set the debug flags: %s", cudaGetErrorString(e));
    return SS_OK;
}

ss_status set_wait_budget(unsigned long long ns) {
    const cudaError_t e = cudaMemcpyToSymbol(ssk::g_wait_budget_ns, &ns, sizeof(ns));
    if (e != cudaSuccess) return fail(SS_ERR_CUDA, "cannot set the wait budget: %s", cudaGetErrorString(e));
    return SS_OK;
}

}  // namespace ssi
