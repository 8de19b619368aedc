// Host-side interface between the C ABI layer (ss_api.cpp) and the kernel
// translation unit (ss_kernels.cu).  Not part of the public API.
#pragma once

#include <cstddef>
#include <cstdint>

#include "ssscan.h"

namespace ssi {

// One call's arguments after validation.  Sequences are H x W maps; a plain
// sequence is H = 1, W = L.  orders[k] is the traversal of direction k.
struct ScanArgs {
    int64_t batch = 0, dim = 0, L = 0, H = 1, W = 0;
    int N = 0, G = 1, K = 1;
    int io = SS_BF16;
    const void *u = nullptr, *delta = nullptr, *B = nullptr, *C = nullptr, *z = nullptr;
    const float *A = nullptr, *D = nullptr, *bias = nullptr;
    int softplus = 1;
    void *out = nullptr;
    float *last_state = nullptr;
    void *ws = nullptr;
    size_t ws_bytes = 0;
    int orders[8] = {0, 1, 2, 3, 4, 5, 6, 7};
    int win = 0;  // window size of the windowed orders
    int chunks = 0;  // single direction: 0 automatic, 1 direct, >= 2 chunked with that many L-chunks
    const float *h0 = nullptr;  // single direction: initial state [batch, dim, N] (nullable)
    int zoh = 0;                // single direction: zero-order-hold input matrix
    // single direction: fused Conv1D(k=4) + SiLU in front of the scan
    int conv = 0;
    const float *conv_w = nullptr, *conv_b = nullptr, *conv_x0 = nullptr;
    ss_stream_t stream = nullptr;
};

// Directions of any order (including the windowed ones), each stored by scan
// step, then merged by position.
size_t steps_workspace_bytes(const ScanArgs &a);
ss_status launch_steps(const ScanArgs &a);

// Backward pass of one direction: the forward call's inputs in `f` (its out,
// last_state and workspace fields unused), the upstream gradient and the
// gradient outputs.
struct BwdArgs {
    ScanArgs f;
    const void *dout = nullptr;
    void *du = nullptr, *ddelta = nullptr, *dz = nullptr;  // I/O type
    float *dA = nullptr, *dB = nullptr, *dC = nullptr;     // fp32
    float *dD = nullptr, *dbias = nullptr;                 // fp32, nullable
    // single direction with options (f.zoh, f.h0, f.conv): the gradient of h0
    // and, with the fused Conv1D (du is then the gradient of its input x), of
    // its weights, bias and history
    float *dh0 = nullptr;
    float *dconv_w = nullptr, *dconv_b = nullptr, *dconv_x0 = nullptr;
    float *du_f32 = nullptr;  // internal: du in fp32 [batch*dim, L] instead of du (Conv1D path)
    void *ws = nullptr;
    size_t ws_bytes = 0;
};

// Workspace of a multi-direction backward pass: the pre-gate output sum s
// [rows, L] (I/O type), the directions' du by scan step [K, rows, L] fp32 (also
// the forward pass's accumulators before that), the state checkpoints.
size_t multi_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t L, int N, int K);
// Backward pass of directions of any order (f.K, f.orders, f.H, f.W, f.win).
ss_status launch_multi_bwd(const BwdArgs &a, bool empty);

// Direction traversal codes used by the kernels (match SS_DIR_*).
enum { ORD_ROW = 0, ORD_COL = 1, ORD_ROW_REV = 2, ORD_COL_REV = 3, ORD_WIN = 4, ORD_WIN_COL = 5,
       ORD_WIN_REV = 6, ORD_WIN_COL_REV = 7 };

// Sets the thread-local error message and returns `st`.
ss_status fail(ss_status st, const char *fmt, ...);

// True when the single-direction call runs the TMA path (16-byte aligned rows).
bool scan1d_uses_tma(const ScanArgs &a);
// Workspace the single-direction path needs for this call (0 when it runs direct).
size_t scan1d_workspace_bytes(const ScanArgs &a);

// Workspace the bidirectional / SS2D call needs (0 when it merges on chip).
size_t multidir_workspace_bytes(const ScanArgs &a);

ss_status launch_scan1d(const ScanArgs &a);
// One recurrence step (seqlen 1) updating `state` [batch*dim, N] in place.
ss_status launch_step(const ScanArgs &a, float *state);
ss_status launch_multidir(const ScanArgs &a);
// Checkpoint workspace of the backward pass: 16-step state checkpoints, fp32;
// with the fused Conv1D also the recomputed u and the scan's du (sized for
// either dtype).
size_t scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t L, int N, bool conv = false);
// Zeroes the summed gradient outputs, then runs the backward kernel (nothing
// but the zeroing when `empty`).
ss_status launch_scan_bwd(const BwdArgs &a, bool empty);
// Depthwise 3 x 3 convolution + SiLU over [batch, dim, H, W] maps.
ss_status launch_dwconv3x3(int64_t batch, int64_t dim, int64_t H, int64_t W, int io, const void *x,
                           const float *w, const float *bias, void *u, ss_stream_t stream);
ss_status read_device_status(ss_stream_t stream);
ss_status set_wait_budget(unsigned long long ns);
ss_status set_debug_flags(unsigned int flags);
// Device address of the fixed scratch array of ss_selective_scan_fwd_noalloc on
// the current device (looked up on every call).
ss_status noalloc_scratch(void **ptr);

}  // namespace ssi
