// C ABI of the selective-scan library: argument validation and dispatch.
// The arithmetic is in the kernels (ss_kernels.cu); nothing here touches tensor
// data, so every check below runs before any work is enqueued.
#include <algorithm>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <initializer_list>

#include "ss_internal.h"
#include "ssscan.h"

namespace ssi {

namespace {
thread_local char g_msg[512] = "no error";

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Byte range [p, p + n) for overlap checks.
struct Span {
    const char *p;
    int64_t n;
};
bool overlaps(Span a, Span b) {
    if (!a.p || !b.p || a.n <= 0 || b.n <= 0) return false;
    return a.p < b.p + b.n && b.p < a.p + a.n;
}

bool valid_dstate(int n) {
    return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64;
}

// Common checks of all three calls.  Returns SS_OK and sets *empty when there
// is nothing to compute.
ss_status check_common(const char *fn, int64_t batch, int64_t dim, int64_t L, int dstate,
                       int ngroups, int io, int K, const void *u, const void *delta,
                       const float *A, const void *B, const void *C, const float *D,
                       const void *z, const float *bias, const void *out,
                       const float *last_state, bool *empty) {
    *empty = false;
    if (batch < 0 || dim < 0 || L < 0)
        return fail(SS_ERR_INVALID_ARG, "%s: negative size (batch=%lld dim=%lld seqlen=%lld)", fn,
                    (long long)batch, (long long)dim, (long long)L);
    if (io != SS_F32 && io != SS_BF16)
        return fail(SS_ERR_UNSUPPORTED, "%s: unknown I/O dtype %d", fn, io);
    if (!valid_dstate(dstate))
        return fail(SS_ERR_UNSUPPORTED, "%s: dstate %d is not one of 1,2,4,8,16,32,64", fn, dstate);
    if (ngroups < 1) return fail(SS_ERR_INVALID_ARG, "%s: ngroups must be >= 1", fn);
    if (dim > 0 && dim % ngroups != 0)
        return fail(SS_ERR_INVALID_ARG, "%s: dim %lld is not a multiple of ngroups %d", fn,
                    (long long)dim, ngroups);
    if (batch == 0 || dim == 0 || L == 0) {
        *empty = true;
        return SS_OK;
    }
    if (!u || !delta || !A || !B || !C || !out)
        return fail(SS_ERR_INVALID_ARG, "%s: u, delta, A, B, C and out are required", fn);
    const void *ptrs[] = {u, delta, A, B, C, D, z, bias, out, last_state};
    for (const void *p : ptrs)
        if (p && !aligned16(p))
            return fail(SS_ERR_ALIGNMENT, "%s: tensor at %p is not 16-byte aligned", fn, p);
    if (batch * dim >= (1ll << 31) || L >= (1ll << 31) || batch * ngroups * dstate >= (1ll << 31) ||
        batch * K * dim >= (1ll << 31) || dim / ngroups >= (1ll << 30))
        return fail(SS_ERR_UNSUPPORTED, "%s: shape exceeds the 2^31 row/position limits", fn);
    if (batch * ngroups > 65535)
        return fail(SS_ERR_UNSUPPORTED, "%s: batch * ngroups %lld exceeds the 65535 grid rows", fn,
                    (long long)(batch * ngroups));
    const int64_t es = io == SS_BF16 ? 2 : 4;
    const int64_t nel = batch * dim * L;
    const Span so{static_cast<const char *>(out), nel * es};
    const Span ins[] = {{static_cast<const char *>(u), nel * es},
                        {static_cast<const char *>(delta), nel * K * es},
                        {static_cast<const char *>(B), batch * K * ngroups * dstate * L * es},
                        {static_cast<const char *>(C), batch * K * ngroups * dstate * L * es},
                        {static_cast<const char *>(z), z ? nel * es : 0},
                        {reinterpret_cast<const char *>(last_state),
                         last_state ? batch * K * dim * dstate * 4 : 0}};
    for (const Span &s : ins)
        if (overlaps(so, s)) return fail(SS_ERR_INVALID_ARG, "%s: out overlaps an input or last_state", fn);
    return SS_OK;
}

// Options of the single-direction calls: reserved fields zero, known flags, a
// 16-byte aligned initial state that does not overlap the output.
ss_status check_options(const char *fn, const ss_scan_options *o, int64_t batch, int64_t dim,
                        int dstate, const void *out, int io, int64_t L) {
    if (!o) return SS_OK;
    for (int r : o->reserved)
        if (r != 0) return fail(SS_ERR_INVALID_ARG, "%s: reserved option fields must be zero", fn);
    if (o->chunks < 0) return fail(SS_ERR_INVALID_ARG, "%s: options.chunks < 0", fn);
    if (o->flags & ~(SS_SCAN_ZOH | SS_SCAN_CONV_SILU))
        return fail(SS_ERR_INVALID_ARG, "%s: unknown option flags 0x%x", fn, o->flags);
    if (o->flags & SS_SCAN_CONV_SILU) {
        if (!o->conv_w) return fail(SS_ERR_INVALID_ARG, "%s: SS_SCAN_CONV_SILU needs conv_w", fn);
        for (const void *q : {(const void *)o->conv_w, (const void *)o->conv_b, (const void *)o->conv_x0})
            if (q && !aligned16(q)) return fail(SS_ERR_ALIGNMENT, "%s: a conv tensor is not 16-byte aligned", fn);
        const int64_t es = io == SS_BF16 ? 2 : 4;
        if ((L * es) % 16 != 0)
            return fail(SS_ERR_UNSUPPORTED, "%s: the fused Conv1D needs 16-byte aligned rows", fn);
    } else if (o->conv_w || o->conv_b || o->conv_x0) {
        return fail(SS_ERR_INVALID_ARG, "%s: conv tensors given without SS_SCAN_CONV_SILU", fn);
    }
    if (o->h0) {
        if (!aligned16(o->h0)) return fail(SS_ERR_ALIGNMENT, "%s: options.h0 is not 16-byte aligned", fn);
        const int64_t es = io == SS_BF16 ? 2 : 4;
        const Span so{static_cast<const char *>(out), batch * dim * L * es};
        const Span sh{reinterpret_cast<const char *>(o->h0), batch * dim * dstate * 4};
        if (overlaps(so, sh)) return fail(SS_ERR_INVALID_ARG, "%s: out overlaps options.h0", fn);
    }
    return SS_OK;
}

// The merge accumulator of the multi-direction calls must not overlap any tensor.
ss_status check_ws_overlap(const char *fn, const ScanArgs &a) {
    if (!a.ws || a.ws_bytes == 0) return SS_OK;
    const int64_t es = a.io == SS_BF16 ? 2 : 4;
    const int64_t nel = a.batch * a.dim * a.L;
    const Span w{static_cast<const char *>(a.ws), (int64_t)a.ws_bytes};
    const Span all[] = {{static_cast<const char *>(a.out), nel * es},
                        {static_cast<const char *>(a.u), nel * es},
                        {static_cast<const char *>(a.delta), nel * a.K * es},
                        {static_cast<const char *>(a.B), a.batch * a.K * a.G * a.N * a.L * es},
                        {static_cast<const char *>(a.C), a.batch * a.K * a.G * a.N * a.L * es},
                        {static_cast<const char *>(a.z), a.z ? nel * es : 0},
                        {reinterpret_cast<const char *>(a.last_state),
                         a.last_state ? a.batch * a.K * a.dim * a.N * 4 : 0}};
    for (const Span &t : all)
        if (overlaps(w, t)) return fail(SS_ERR_INVALID_ARG, "%s: workspace overlaps a tensor", fn);
    return SS_OK;
}

ss_status check_workspace(const char *fn, size_t need, const void *ws, size_t have) {
    if (need == 0) return SS_OK;
    if (!ws || have < need)
        return fail(SS_ERR_WORKSPACE, "%s: needs %zu bytes of workspace, got %zu%s", fn, need, have,
                    ws ? "" : " (null)");
    if (!aligned16(ws)) return fail(SS_ERR_ALIGNMENT, "%s: workspace is not 16-byte aligned", fn);
    return SS_OK;
}

ScanArgs scan_args(int64_t batch, int64_t dim, int64_t L, int dstate, int ngroups, int io,
                   const void *u, const void *delta, const float *A, const void *B, const void *C,
                   const float *D, const void *z, const float *bias, int softplus, void *out,
                   float *last_state, void *ws, size_t ws_bytes, ss_stream_t stream) {
    ScanArgs a;
    a.batch = batch;
    a.dim = dim;
    a.L = L;
    a.H = 1;
    a.W = L;
    a.N = dstate;
    a.G = ngroups;
    a.io = io;
    a.u = u;
    a.delta = delta;
    a.A = A;
    a.B = B;
    a.C = C;
    a.D = D;
    a.z = z;
    a.bias = bias;
    a.softplus = softplus ? 1 : 0;
    a.out = out;
    a.last_state = last_state;
    a.ws = ws;
    a.ws_bytes = ws_bytes;
    a.stream = stream;
    return a;
}

size_t ws_scan1d_any_dtype(int64_t batch, int64_t dim, int64_t L, int dstate, int chunks) {
    if (batch <= 0 || dim <= 0 || L <= 0 || !valid_dstate(dstate)) return 0;
    size_t best = 0;
    for (int io : {SS_F32, SS_BF16}) {
        ScanArgs a;
        a.batch = batch;
        a.dim = dim;
        a.L = L;
        a.W = L;
        a.N = dstate;
        a.io = io;
        a.chunks = chunks;
        const size_t w = scan1d_workspace_bytes(a);
        if (w > best) best = w;
    }
    return best;
}

size_t ws_multidir_any_dtype(int64_t batch, int64_t dim, int64_t L, int dstate, int K) {
    if (batch <= 0 || dim <= 0 || L <= 0 || !valid_dstate(dstate)) return 0;
    size_t best = 0;
    for (int io : {SS_F32, SS_BF16}) {
        ScanArgs a;
        a.batch = batch;
        a.dim = dim;
        a.L = L;
        a.W = L;
        a.N = dstate;
        a.io = io;
        a.K = K;
        const size_t w = multidir_workspace_bytes(a);
        if (w > best) best = w;
    }
    return best;
}

// Backward pass: required gradient pointers, alignment, and that no output
// overlaps an input, another output or the workspace.
ss_status check_bwd(const char *fn, int64_t batch, int64_t dim, int64_t L, int N, int G, int io,
                    const void *u, const void *delta, const float *A, const void *B,
                    const void *C, const float *D, const void *z, const float *bias,
                    const void *dout, const void *du, const void *ddelta, const float *dA,
                    const float *dB, const float *dC, const float *dD, const void *dz,
                    const float *dbias, const void *ws, size_t ws_bytes, int K = 1) {
    if (!dout || !du || !ddelta || !dA || !dB || !dC)
        return fail(SS_ERR_INVALID_ARG, "%s: dout, du, ddelta, dA, dB and dC are required", fn);
    if (z && !dz) return fail(SS_ERR_INVALID_ARG, "%s: dz is required when z is given", fn);
    if (!z && dz) return fail(SS_ERR_INVALID_ARG, "%s: dz given without z", fn);
    for (const void *q : {dout, du, ddelta, (const void *)dA, (const void *)dB, (const void *)dC,
                          (const void *)dD, dz, (const void *)dbias})
        if (q && !aligned16(q))
            return fail(SS_ERR_ALIGNMENT, "%s: tensor at %p is not 16-byte aligned", fn, q);
    const int64_t es = io == SS_BF16 ? 2 : 4;
    if ((L * es) % 16 != 0)
        return fail(SS_ERR_UNSUPPORTED,
                    "%s: rows must be 16-byte aligned (seqlen * element size %% 16 == 0)", fn);
    const int64_t nel = batch * dim * L;
    const int64_t nbc = batch * K * G * N * L;
    const int64_t kd = (int64_t)K * dim;
    const Span outs[] = {{static_cast<const char *>(du), nel * es},
                         {static_cast<const char *>(ddelta), nel * K * es},
                         {static_cast<const char *>(dz), dz ? nel * es : 0},
                         {reinterpret_cast<const char *>(dA), kd * N * 4},
                         {reinterpret_cast<const char *>(dB), nbc * 4},
                         {reinterpret_cast<const char *>(dC), nbc * 4},
                         {reinterpret_cast<const char *>(dD), dD ? kd * 4 : 0},
                         {reinterpret_cast<const char *>(dbias), dbias ? kd * 4 : 0},
                         {static_cast<const char *>(ws), ws ? (int64_t)ws_bytes : 0}};
    const Span ins[] = {{static_cast<const char *>(u), nel * es},
                        {static_cast<const char *>(delta), nel * K * es},
                        {reinterpret_cast<const char *>(A), kd * N * 4},
                        {static_cast<const char *>(B), nbc * es},
                        {static_cast<const char *>(C), nbc * es},
                        {reinterpret_cast<const char *>(D), D ? kd * 4 : 0},
                        {static_cast<const char *>(z), z ? nel * es : 0},
                        {reinterpret_cast<const char *>(bias), bias ? kd * 4 : 0},
                        {static_cast<const char *>(dout), nel * es}};
    const int nout = sizeof(outs) / sizeof(outs[0]);
    for (int i = 0; i < nout; ++i) {
        for (const Span &t : ins)
            if (overlaps(outs[i], t))
                return fail(SS_ERR_INVALID_ARG, "%s: a gradient output or the workspace overlaps an input", fn);
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(outs[i], outs[j]))
                return fail(SS_ERR_INVALID_ARG, "%s: two gradient outputs (or the workspace) overlap", fn);
    }
    return SS_OK;
}

}  // namespace

ss_status fail(ss_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
    va_end(ap);
    return st;
}

}  // namespace ssi

using namespace ssi;

extern "C" {

ss_status ss_selective_scan_fwd_opts(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                     int ngroups, ss_dtype io, const void *u, const void *delta,
                                     const float *A, const void *B, const void *C, const float *D,
                                     const void *z, const float *delta_bias, int delta_softplus,
                                     void *out, float *last_state, void *workspace,
                                     size_t workspace_bytes, const ss_scan_options *options,
                                     ss_stream_t stream) {
    static const char *fn = "ss_selective_scan_fwd";
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, seqlen, dstate, ngroups, io, 1, u, delta, A, B, C,
                                D, z, delta_bias, out, last_state, &empty);
    if (st != SS_OK || empty) return st;
    int chunks = 0;
    if ((st = check_options(fn, options, batch, dim, dstate, out, io, seqlen))) return st;
    if (options) chunks = options->chunks;
    ScanArgs a = scan_args(batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z,
                           delta_bias, delta_softplus, out, last_state, workspace,
                           workspace_bytes, stream);
    a.chunks = chunks;
    if (options) {
        a.h0 = options->h0;
        a.zoh = (options->flags & SS_SCAN_ZOH) ? 1 : 0;
        a.conv = (options->flags & SS_SCAN_CONV_SILU) ? 1 : 0;
        a.conv_w = options->conv_w;
        a.conv_b = options->conv_b;
        a.conv_x0 = options->conv_x0;
    }
    // Rows that are not 16-byte aligned: a workspace is optional -- with one of
    // at least the reported size the view-tiled scan may take the chunked
    // path, otherwise it runs in one pass.
    if (!scan1d_uses_tma(a)) {
        if (workspace && !aligned16(workspace))
            return fail(SS_ERR_ALIGNMENT, "%s: workspace is not 16-byte aligned", fn);
    } else if ((st = check_workspace(fn, scan1d_workspace_bytes(a), workspace, workspace_bytes))) {
        return st;
    }
    if ((st = check_ws_overlap(fn, a))) return st;
    return launch_scan1d(a);
}

ss_status ss_selective_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                int ngroups, ss_dtype io, const void *u, const void *delta,
                                const float *A, const void *B, const void *C, const float *D,
                                const void *z, const float *delta_bias, int delta_softplus,
                                void *out, float *last_state, void *workspace,
                                size_t workspace_bytes, ss_stream_t stream) {
    return ss_selective_scan_fwd_opts(batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C,
                                      D, z, delta_bias, delta_softplus, out, last_state,
                                      workspace, workspace_bytes, nullptr, stream);
}

ss_status ss_selective_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                        int ngroups, ss_dtype io, const void *u,
                                        const void *delta, const float *A, const void *B,
                                        const void *C, const float *D, const void *z,
                                        const float *delta_bias, int delta_softplus, void *out,
                                        float *last_state, const ss_scan_options *options,
                                        ss_stream_t stream) {
    static const char *fn = "ss_selective_scan_fwd_noalloc";
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, seqlen, dstate, ngroups, io, 1, u, delta, A, B, C,
                                D, z, delta_bias, out, last_state, &empty);
    if (st != SS_OK || empty) return st;
    int chunks = 0;
    if ((st = check_options(fn, options, batch, dim, dstate, out, io, seqlen))) return st;
    if (options) chunks = options->chunks;
    ScanArgs a = scan_args(batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z,
                           delta_bias, delta_softplus, out, last_state, nullptr, 0, stream);
    a.chunks = chunks;
    if (options) {
        a.h0 = options->h0;
        a.zoh = (options->flags & SS_SCAN_ZOH) ? 1 : 0;
        a.conv = (options->flags & SS_SCAN_CONV_SILU) ? 1 : 0;
        a.conv_w = options->conv_w;
        a.conv_b = options->conv_b;
        a.conv_x0 = options->conv_x0;
    }
    // rows that are not 16-byte aligned run in one pass here (their workspace
    // is optional)
    const size_t need = scan1d_uses_tma(a) ? scan1d_workspace_bytes(a) : 0;
    if (need > SS_NOALLOC_SCRATCH_BYTES)
        return fail(SS_ERR_UNSUPPORTED,
                    "%s: this shape needs %zu bytes of scratch, more than the fixed %zu bytes "
                    "the library holds; request fewer chunks, or call ss_selective_scan_fwd "
                    "with a workspace",
                    fn, need, (size_t)SS_NOALLOC_SCRATCH_BYTES);
    if (need > 0) {
        void *scratch = nullptr;
        if ((st = noalloc_scratch(&scratch))) return st;
        a.ws = scratch;
        a.ws_bytes = SS_NOALLOC_SCRATCH_BYTES;
    }
    return launch_scan1d(a);
}

ss_status ss_bidir_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int dstate, int ngroups,
                            ss_dtype io, const void *u, const void *delta, const float *A,
                            const void *B, const void *C, const float *D, const void *z,
                            const float *delta_bias, int delta_softplus, void *out,
                            float *last_state, void *workspace, size_t workspace_bytes,
                            ss_stream_t stream) {
    static const char *fn = "ss_bidir_scan_fwd";
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, seqlen, dstate, ngroups, io, 2, u, delta, A, B, C,
                                D, z, delta_bias, out, last_state, &empty);
    if (st != SS_OK || empty) return st;
    ScanArgs a = scan_args(batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z,
                           delta_bias, delta_softplus, out, last_state, workspace,
                           workspace_bytes, stream);
    a.K = 2;
    a.orders[0] = ORD_ROW;
    a.orders[1] = ORD_ROW_REV;
    // Rows that are not 16-byte aligned: a workspace is optional -- with one of
    // at least the re-pitched path's size (which grows with ngroups) the inputs
    // are re-pitched into it, otherwise the call merges on chip.
    if (!scan1d_uses_tma(a)) {
        if (workspace && !aligned16(workspace))
            return fail(SS_ERR_ALIGNMENT, "%s: workspace is not 16-byte aligned", fn);
    } else if ((st = check_workspace(fn, multidir_workspace_bytes(a), workspace, workspace_bytes))) {
        return st;
    }
    if ((st = check_ws_overlap(fn, a))) return st;
    return launch_multidir(a);
}

ss_status ss_cross_scan2d_fwd(int64_t batch, int64_t dim, int64_t H, int64_t W, int dstate,
                              int ngroups, ss_dtype io, const void *u, const void *delta,
                              const float *A, const void *B, const void *C, const float *D,
                              const float *delta_bias, int delta_softplus, const void *z,
                              void *out, float *last_state, void *workspace,
                              size_t workspace_bytes, ss_stream_t stream) {
    static const char *fn = "ss_cross_scan2d_fwd";
    if (H < 0 || W < 0) return fail(SS_ERR_INVALID_ARG, "%s: negative map size", fn);
    if (H >= (1ll << 31) || W >= (1ll << 31) || (H > 0 && W > (INT64_MAX / H)))
        return fail(SS_ERR_UNSUPPORTED, "%s: map too large", fn);
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, H * W, dstate, ngroups, io, 4, u, delta, A, B, C,
                                D, z, delta_bias, out, last_state, &empty);
    if (st != SS_OK || empty) return st;
    ScanArgs a = scan_args(batch, dim, H * W, dstate, ngroups, io, u, delta, A, B, C, D, z,
                           delta_bias, delta_softplus, out, last_state, workspace,
                           workspace_bytes, stream);
    a.K = 4;
    a.H = H;
    a.W = W;
    a.orders[0] = ORD_ROW;
    a.orders[1] = ORD_COL;
    a.orders[2] = ORD_ROW_REV;
    a.orders[3] = ORD_COL_REV;
    // Maps whose rows are not 16-byte aligned: a workspace is optional -- with
    // one of at least the reported size the call reads the rows through view
    // tiles, otherwise it merges on chip.
    if (!scan1d_uses_tma(a)) {
        if (workspace && !aligned16(workspace))
            return fail(SS_ERR_ALIGNMENT, "%s: workspace is not 16-byte aligned", fn);
    } else if ((st = check_workspace(fn, multidir_workspace_bytes(a), workspace, workspace_bytes))) {
        return st;
    }
    if ((st = check_ws_overlap(fn, a))) return st;
    return launch_multidir(a);
}

ss_status ss_selective_state_update(int64_t batch, int64_t dim, int dstate, int ngroups,
                                    ss_dtype io, const void *x, const void *delta,
                                    const float *A, const void *B, const void *C,
                                    const float *D, const void *z, const float *delta_bias,
                                    int delta_softplus, unsigned int flags, float *state,
                                    void *out, ss_stream_t stream) {
    static const char *fn = "ss_selective_state_update";
    bool empty = false;
    if (flags & ~SS_SCAN_ZOH) return fail(SS_ERR_INVALID_ARG, "%s: unknown flags 0x%x", fn, flags);
    ss_status st = check_common(fn, batch, dim, 1, dstate, ngroups, io, 1, x, delta, A, B, C, D, z,
                                delta_bias, out, state, &empty);
    if (st != SS_OK || empty) return st;
    if (!state) return fail(SS_ERR_INVALID_ARG, "%s: state is required", fn);
    if (!aligned16(state)) return fail(SS_ERR_ALIGNMENT, "%s: state is not 16-byte aligned", fn);
    ScanArgs a = scan_args(batch, dim, 1, dstate, ngroups, io, x, delta, A, B, C, D, z, delta_bias,
                           delta_softplus, out, nullptr, nullptr, 0, stream);
    a.zoh = (flags & SS_SCAN_ZOH) ? 1 : 0;
    return launch_step(a, state);
}

ss_status ss_multi_scan_fwd(int64_t batch, int64_t dim, int64_t H, int64_t W, int ndirs,
                            const int *orders, int window, int dstate, int ngroups, ss_dtype io,
                            const void *u, const void *delta, const float *A, const void *B,
                            const void *C, const float *D, const float *delta_bias,
                            int delta_softplus, const void *z, void *out, float *last_state,
                            void *workspace, size_t workspace_bytes, ss_stream_t stream) {
    static const char *fn = "ss_multi_scan_fwd";
    if (H < 0 || W < 0) return fail(SS_ERR_INVALID_ARG, "%s: negative map size", fn);
    if (H >= (1ll << 31) || W >= (1ll << 31) || (H > 0 && W > (INT64_MAX / H)))
        return fail(SS_ERR_UNSUPPORTED, "%s: map too large", fn);
    if (ndirs < 1 || ndirs > 8)
        return fail(SS_ERR_INVALID_ARG, "%s: ndirs %d is not in 1..8", fn, ndirs);
    if (!orders) return fail(SS_ERR_INVALID_ARG, "%s: orders is required", fn);
    bool windowed = false;
    for (int k = 0; k < ndirs; ++k) {
        if (orders[k] < SS_DIR_ROW || orders[k] > SS_DIR_WIN_COL_REV)
            return fail(SS_ERR_INVALID_ARG, "%s: orders[%d] = %d is not an SS_DIR_* code", fn, k,
                        orders[k]);
        windowed = windowed || orders[k] >= SS_DIR_WIN;
    }
    if (windowed && window < 1)
        return fail(SS_ERR_INVALID_ARG, "%s: a windowed order needs window >= 1", fn);
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, H * W, dstate, ngroups, io, ndirs, u, delta, A, B,
                                C, D, z, delta_bias, out, last_state, &empty);
    if (st != SS_OK || empty) return st;
    const int64_t es = io == SS_BF16 ? 2 : 4;
    if ((H * W * es) % 16 != 0)
        return fail(SS_ERR_UNSUPPORTED,
                    "%s: rows must be 16-byte aligned (H * W * element size %% 16 == 0)", fn);
    ScanArgs a = scan_args(batch, dim, H * W, dstate, ngroups, io, u, delta, A, B, C, D, z,
                           delta_bias, delta_softplus, out, last_state, workspace,
                           workspace_bytes, stream);
    a.K = ndirs;
    a.H = H;
    a.W = W;
    for (int k = 0; k < ndirs; ++k) a.orders[k] = orders[k];
    // a window at least as large as the map is one window: the same traversal
    const int64_t big = H > W ? H : W;
    a.win = windowed ? (int)(window < big ? window : big) : 1;
    if ((st = check_workspace(fn, steps_workspace_bytes(a), workspace, workspace_bytes))) return st;
    if ((st = check_ws_overlap(fn, a))) return st;
    return launch_steps(a);
}

ss_status ss_multi_scan_bwd(int64_t batch, int64_t dim, int64_t H, int64_t W, int ndirs,
                            const int *orders, int window, int dstate, int ngroups, ss_dtype io,
                            const void *u, const void *delta, const float *A, const void *B,
                            const void *C, const float *D, const float *delta_bias,
                            int delta_softplus, const void *z, const void *dout, void *du,
                            void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz,
                            float *ddelta_bias, void *workspace, size_t workspace_bytes,
                            ss_stream_t stream) {
    static const char *fn = "ss_multi_scan_bwd";
    if (H < 0 || W < 0) return fail(SS_ERR_INVALID_ARG, "%s: negative map size", fn);
    if (H >= (1ll << 31) || W >= (1ll << 31) || (H > 0 && W > (INT64_MAX / H)))
        return fail(SS_ERR_UNSUPPORTED, "%s: map too large", fn);
    if (ndirs < 1 || ndirs > 8)
        return fail(SS_ERR_INVALID_ARG, "%s: ndirs %d is not in 1..8", fn, ndirs);
    if (!orders) return fail(SS_ERR_INVALID_ARG, "%s: orders is required", fn);
    bool windowed = false;
    for (int k = 0; k < ndirs; ++k) {
        if (orders[k] < SS_DIR_ROW || orders[k] > SS_DIR_WIN_COL_REV)
            return fail(SS_ERR_INVALID_ARG, "%s: orders[%d] = %d is not an SS_DIR_* code", fn, k,
                        orders[k]);
        windowed = windowed || orders[k] >= SS_DIR_WIN;
    }
    if (windowed && window < 1)
        return fail(SS_ERR_INVALID_ARG, "%s: a windowed order needs window >= 1", fn);
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, H * W, dstate, ngroups, io, ndirs, u, delta, A, B,
                                C, D, z, delta_bias, du, nullptr, &empty);
    if (st != SS_OK) return st;
    BwdArgs a;
    a.f = scan_args(batch, dim, H * W, dstate, ngroups, io, u, delta, A, B, C, D, z, delta_bias,
                    delta_softplus, nullptr, nullptr, nullptr, 0, stream);
    a.f.K = ndirs;
    a.f.H = H;
    a.f.W = W;
    for (int k = 0; k < ndirs; ++k) a.f.orders[k] = orders[k];
    const int64_t big = H > W ? H : W;
    a.f.win = windowed ? (int)(window < big ? window : big) : 1;
    a.dout = dout;
    a.du = du;
    a.ddelta = ddelta;
    a.dz = dz;
    a.dA = dA;
    a.dB = dB;
    a.dC = dC;
    a.dD = dD;
    a.dbias = ddelta_bias;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    if (empty) return launch_multi_bwd(a, true);
    if ((st = check_bwd(fn, batch, dim, H * W, dstate, ngroups, io, u, delta, A, B, C, D, z,
                        delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, workspace,
                        workspace_bytes, ndirs)))
        return st;
    if ((st = check_workspace(fn, multi_bwd_workspace_bytes(batch, dim, H * W, dstate, ndirs),
                              workspace, workspace_bytes)))
        return st;
    return launch_multi_bwd(a, false);
}

size_t ss_multi_scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t H, int64_t W,
                                         int dstate, int ndirs) {
    if (H <= 0 || W <= 0 || ndirs < 1 || ndirs > 8 || !valid_dstate(dstate)) return 0;
    return multi_bwd_workspace_bytes(batch, dim, H * W, dstate, ndirs);
}

ss_status ss_dwconv3x3_silu_fwd(int64_t batch, int64_t dim, int64_t H, int64_t W, ss_dtype io,
                                const void *x, const float *w, const float *bias, void *u,
                                ss_stream_t stream) {
    static const char *fn = "ss_dwconv3x3_silu_fwd";
    if (batch < 0 || dim < 0 || H < 0 || W < 0)
        return fail(SS_ERR_INVALID_ARG, "%s: negative size", fn);
    if (io != SS_F32 && io != SS_BF16) return fail(SS_ERR_UNSUPPORTED, "%s: unknown I/O dtype %d", fn, io);
    if (batch == 0 || dim == 0 || H == 0 || W == 0) return SS_OK;
    if (H >= (1ll << 31) || W >= (1ll << 31) || H * W >= (1ll << 31) || batch * dim >= (1ll << 40))
        return fail(SS_ERR_UNSUPPORTED, "%s: map too large", fn);
    if (!x || !w || !u) return fail(SS_ERR_INVALID_ARG, "%s: x, w and u are required", fn);
    for (const void *q : {x, (const void *)w, (const void *)bias, (const void *)u})
        if (q && !aligned16(q)) return fail(SS_ERR_ALIGNMENT, "%s: tensor at %p is not 16-byte aligned", fn, q);
    const int64_t es = io == SS_BF16 ? 2 : 4;
    const int64_t n = batch * dim * H * W * es;
    if (overlaps({static_cast<const char *>(u), n}, {static_cast<const char *>(x), n}))
        return fail(SS_ERR_INVALID_ARG, "%s: u overlaps x", fn);
    return launch_dwconv3x3(batch, dim, H, W, io, x, w, bias, u, stream);
}

size_t ss_multi_scan_workspace_bytes(int64_t batch, int64_t dim, int64_t H, int64_t W, int ndirs) {
    if (batch <= 0 || dim <= 0 || H <= 0 || W <= 0 || ndirs < 1 || ndirs > 8) return 0;
    // the fp32 accumulators by step, then up to three copies of u permuted into
    // the column and windowed traversals (sized for float32 I/O, which covers
    // every order list and I/O type)
    auto a256 = [](size_t n) { return (n + 255) & ~size_t(255); };
    const size_t map = (size_t)batch * dim * H * W * sizeof(float);
    return a256((size_t)ndirs * map) + (size_t)std::min(ndirs, 3) * a256(map);
}

ss_status ss_selective_scan_bwd(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                int ngroups, ss_dtype io, const void *u, const void *delta,
                                const float *A, const void *B, const void *C, const float *D,
                                const void *z, const float *delta_bias, int delta_softplus,
                                const void *dout, void *du, void *ddelta, float *dA, float *dB,
                                float *dC, float *dD, void *dz, float *ddelta_bias,
                                void *workspace, size_t workspace_bytes, ss_stream_t stream) {
    static const char *fn = "ss_selective_scan_bwd";
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, seqlen, dstate, ngroups, io, 1, u, delta, A, B, C,
                                D, z, delta_bias, du, nullptr, &empty);
    if (st != SS_OK) return st;
    BwdArgs a;
    a.f = scan_args(batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z, delta_bias,
                    delta_softplus, nullptr, nullptr, nullptr, 0, stream);
    a.dout = dout;
    a.du = du;
    a.ddelta = ddelta;
    a.dz = dz;
    a.dA = dA;
    a.dB = dB;
    a.dC = dC;
    a.dD = dD;
    a.dbias = ddelta_bias;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    if (empty) return launch_scan_bwd(a, true);  // the gradient of an empty sum is zero
    if ((st = check_bwd(fn, batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z,
                        delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, workspace,
                        workspace_bytes)))
        return st;
    if ((st = check_workspace(fn, scan_bwd_workspace_bytes(batch, dim, seqlen, dstate), workspace,
                              workspace_bytes)))
        return st;
    return launch_scan_bwd(a, false);
}

ss_status ss_selective_scan_bwd_opts(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                     int ngroups, ss_dtype io, const void *u, const void *delta,
                                     const float *A, const void *B, const void *C, const float *D,
                                     const void *z, const float *delta_bias, int delta_softplus,
                                     const void *dout, void *du, void *ddelta, float *dA, float *dB,
                                     float *dC, float *dD, void *dz, float *ddelta_bias,
                                     const ss_scan_options *options, const ss_scan_bwd_extras *extras,
                                     void *workspace, size_t workspace_bytes, ss_stream_t stream) {
    static const char *fn = "ss_selective_scan_bwd_opts";
    bool empty = false;
    ss_status st = check_common(fn, batch, dim, seqlen, dstate, ngroups, io, 1, u, delta, A, B, C,
                                D, z, delta_bias, du, nullptr, &empty);
    if (st != SS_OK) return st;
    if ((st = check_options(fn, options, batch, dim, dstate, du, io, seqlen))) return st;
    if (options && options->chunks != 0)
        return fail(SS_ERR_INVALID_ARG, "%s: options.chunks has no meaning here (must be 0)", fn);
    const bool conv = options && (options->flags & SS_SCAN_CONV_SILU);
    ss_scan_bwd_extras ex{};
    if (extras) ex = *extras;
    for (int r : ex.reserved)
        if (r != 0) return fail(SS_ERR_INVALID_ARG, "%s: reserved extras fields must be zero", fn);
    if (conv && !ex.dconv_w)
        return fail(SS_ERR_INVALID_ARG, "%s: SS_SCAN_CONV_SILU needs extras.dconv_w", fn);
    if (!conv && (ex.dconv_w || ex.dconv_b || ex.dconv_x0))
        return fail(SS_ERR_INVALID_ARG, "%s: conv gradients given without SS_SCAN_CONV_SILU", fn);
    if (conv && ((ex.dconv_b && !options->conv_b) || (ex.dconv_x0 && !options->conv_x0)))
        return fail(SS_ERR_INVALID_ARG, "%s: a conv gradient is given without its tensor", fn);
    if (ex.dh0 && !(options && options->h0))
        return fail(SS_ERR_INVALID_ARG, "%s: extras.dh0 given without options.h0", fn);
    for (const void *q : {(const void *)ex.dh0, (const void *)ex.dconv_w, (const void *)ex.dconv_b,
                          (const void *)ex.dconv_x0})
        if (q && !aligned16(q))
            return fail(SS_ERR_ALIGNMENT, "%s: an extras tensor is not 16-byte aligned", fn);
    BwdArgs a;
    a.f = scan_args(batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z, delta_bias,
                    delta_softplus, nullptr, nullptr, nullptr, 0, stream);
    if (options) {
        a.f.h0 = options->h0;
        a.f.zoh = (options->flags & SS_SCAN_ZOH) ? 1 : 0;
        a.f.conv = conv ? 1 : 0;
        a.f.conv_w = options->conv_w;
        a.f.conv_b = options->conv_b;
        a.f.conv_x0 = options->conv_x0;
    }
    a.dout = dout;
    a.du = du;
    a.ddelta = ddelta;
    a.dz = dz;
    a.dA = dA;
    a.dB = dB;
    a.dC = dC;
    a.dD = dD;
    a.dbias = ddelta_bias;
    a.dh0 = ex.dh0;
    a.dconv_w = ex.dconv_w;
    a.dconv_b = ex.dconv_b;
    a.dconv_x0 = ex.dconv_x0;
    a.ws = workspace;
    a.ws_bytes = workspace_bytes;
    if (empty) return launch_scan_bwd(a, true);  // the gradient of an empty sum is zero
    if ((st = check_bwd(fn, batch, dim, seqlen, dstate, ngroups, io, u, delta, A, B, C, D, z,
                        delta_bias, dout, du, ddelta, dA, dB, dC, dD, dz, ddelta_bias, workspace,
                        workspace_bytes)))
        return st;
    if ((st = check_workspace(fn, scan_bwd_workspace_bytes(batch, dim, seqlen, dstate, conv),
                              workspace, workspace_bytes)))
        return st;
    return launch_scan_bwd(a, false);
}

size_t ss_workspace_bytes_opts(int kind, int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                               const ss_scan_options *options) {
    if (kind == SS_KIND_BIDIR || kind == SS_KIND_CROSS2D)
        return ws_multidir_any_dtype(batch, dim, seqlen, dstate, kind == SS_KIND_BIDIR ? 2 : 4);
    if (kind == SS_KIND_SCAN_BWD)
        return valid_dstate(dstate)
                   ? scan_bwd_workspace_bytes(batch, dim, seqlen, dstate,
                                              options && (options->flags & SS_SCAN_CONV_SILU))
                   : 0;
    if (kind != SS_KIND_SCAN) return 0;
    return ws_scan1d_any_dtype(batch, dim, seqlen, dstate, options ? options->chunks : 0);
}

size_t ss_workspace_bytes(int kind, int64_t batch, int64_t dim, int64_t seqlen, int dstate) {
    return ss_workspace_bytes_opts(kind, batch, dim, seqlen, dstate, nullptr);
}

ss_status ss_get_device_status(ss_stream_t stream) { return read_device_status(stream); }

ss_status ss_debug_set_wait_budget_ns(uint64_t ns) {
    return set_wait_budget(ns ? (unsigned long long)ns : 1000000000ull);
}

ss_status ss_debug_set_flags(uint32_t flags) {
    if (flags & ~uint32_t(SS_DEBUG_SKIP_FIRST_COPY))
        return fail(SS_ERR_INVALID_ARG, "ss_debug_set_flags: unknown flag bits 0x%x", flags);
    return set_debug_flags(flags);
}

const char *ss_last_error_string(void) { return g_msg; }

const char *ss_version(void) { return "ssscan 0.1 (sm_103a)"; }

}  // extern "C"
