/*
 * ssscan.h -- C ABI of the B300 selective-scan library (libssscan.so).
 *
 * The library computes the forward pass of the selective state-space scan of
 * Mamba (S6) and its two vision variants, on an NVIDIA B300 (sm_103a):
 *
 *   ss_selective_scan_fwd  one direction over a sequence
 *   ss_bidir_scan_fwd      Vision Mamba's bidirectional scan (forward + reversed, summed)
 *   ss_cross_scan2d_fwd    VMamba's SS2D: four traversal orders of an H x W map, merged by sum
 *
 * Sources (page title, section):
 *   "Mamba Series from Selective State Spaces to Visual State Space Models",
 *     "mathematical form of the selective SSM": Abar = exp(Delta*A); input matrix
 *     (Euler form used here) Bbar = Delta*B; Delta = softplus(W_Delta x + b_Delta);
 *     block diagram "Mamba Block (1D)": output gated by SiLU(z);
 *     "key code" (cross_scan_fwd, SS2Dv0.forwardv0): the four orders (row-major,
 *     column-major, and the reverse of each), selective_scan(xs, dts, As, Bs, Cs,
 *     Ds, delta_bias, delta_softplus), and the merge (flip back, transpose back, sum).
 *   "From LSTM to Mamba: why bidirectional state-space models suit visual sequences",
 *     section 3.1: a forward scan plus a scan of the reversed sequence with its own
 *     parameters.
 *
 * Per (batch b, direction k, channel d) the scan takes steps s = 0..L-1, step s
 * visiting position p = pi_k(s), starting from h = 0:
 *     dt    = Delta_k[d,s] + delta_bias_k[d];  dt = softplus(dt) if delta_softplus
 *     h_n   = exp(dt * A_k[d,n]) * h_n + dt * B_k[g,n,s] * u[d,p]          n < dstate
 *     y_k(p) = sum_n C_k[g,n,s] * h_n + D_k[d] * u[d,p]
 *     out[d,p] = (sum_k y_k(p)) * (z ? z*sigmoid(z) : 1)     (z[d,p])
 * Channel d uses group g = d / (dim / ngroups).  u, z and out are indexed by
 * POSITION p (token order, or the H x W map in row-major order).  Each
 * direction's Delta_k, B_k and C_k are indexed by its own SCAN STEP s, the
 * layout in which the key code computes them (by projecting the already
 * reordered sequences).  The caller's u stays in position order; internally
 * the column and windowed orders read a copy of u permuted into their step
 * order, made in the workspace.
 *
 * Layouts: every tensor is dense and C-contiguous (last index fastest).
 *   dtype ss_dtype io:  u, delta, B, C, z, out          (SS_F32 or SS_BF16)
 *   float32 always:     A, D, delta_bias, last_state
 * Rounding: internal arithmetic is float32; out is rounded to the I/O type
 * (round-to-nearest-even).
 *
 * Ownership and synchronisation: the caller owns every buffer.  All tensor
 * pointers are DEVICE pointers.  The library never allocates device memory and
 * never synchronises the stream (except ss_get_device_status); work is enqueued
 * on `stream` and the call returns.  Kernel faults surface on the caller's next
 * synchronisation.  Each call validates its arguments before launching
 * anything; on error nothing is launched.
 *
 * Errors: every function returns ss_status; ss_last_error_string() gives a
 * thread-local message for the last failing call on the calling thread.
 */
#ifndef SSSCAN_H
#define SSSCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle type as cudaStream_t (struct CUstream_st*); NULL = legacy default stream. */
typedef struct CUstream_st *ss_stream_t;

typedef int ss_status;
#define SS_OK 0
#define SS_ERR_INVALID_ARG 1  /* null required pointer, negative size, dim % ngroups != 0, aliasing */
#define SS_ERR_UNSUPPORTED 2  /* dstate not in {1,2,4,8,16,32,64}, unknown dtype, shape beyond limits */
#define SS_ERR_ALIGNMENT 3    /* a tensor base pointer is not 16-byte aligned */
#define SS_ERR_WORKSPACE 4    /* workspace missing or smaller than ss_workspace_bytes() */
#define SS_ERR_CUDA 5         /* a CUDA runtime/driver call failed (launch, tensor-map encode) */
#define SS_ERR_TIMEOUT 6      /* a kernel gave up a bounded wait (reported by ss_get_device_status) */

typedef enum { SS_F32 = 0, SS_BF16 = 1 } ss_dtype;

/* Direction order codes of ss_cross_scan2d_fwd, in the order its tensors stack them. */
#define SS_DIR_ROW 0     /* row-major: position t                          */
#define SS_DIR_COL 1     /* column-major: position (t % H) * W + t / H     */
#define SS_DIR_ROW_REV 2 /* reversed row-major                             */
#define SS_DIR_COL_REV 3 /* reversed column-major                          */
/* Windowed orders of ss_multi_scan_fwd ("LocalMamba: Visual State Space Model with
 * Windowed Selective Scan": the map is scanned window by window).  The map is cut
 * into window x window windows -- those of the last band of rows and of the last
 * column cut short when the window does not divide H or W. */
#define SS_DIR_WIN 4         /* windows row-major, each window row-major       */
#define SS_DIR_WIN_COL 5     /* windows column-major, each window column-major */
#define SS_DIR_WIN_REV 6     /* reversed SS_DIR_WIN                            */
#define SS_DIR_WIN_COL_REV 7 /* reversed SS_DIR_WIN_COL                        */

/* Kinds for ss_workspace_bytes. */
#define SS_KIND_SCAN 0
#define SS_KIND_BIDIR 1
#define SS_KIND_CROSS2D 2
#define SS_KIND_SCAN_BWD 3 /* ss_selective_scan_bwd */

/*
 * ss_selective_scan_fwd -- one forward direction (Mamba S6 selective scan).
 *
 *   u          [batch, dim, seqlen]            io
 *   delta      [batch, dim, seqlen]            io    (raw Delta, before bias/softplus)
 *   A          [dim, dstate]                   float (already negative: A = -exp(A_log))
 *   B, C       [batch, ngroups, dstate, seqlen] io
 *   D          [dim]                           float, nullable (no skip term)
 *   z          [batch, dim, seqlen]            io, nullable (no gate)
 *   delta_bias [dim]                           float, nullable (zero)
 *   delta_softplus                             0 or 1
 *   out        [batch, dim, seqlen]            io, must not overlap any input
 *   last_state [batch, dim, dstate]            float, nullable; the state after the last step
 *   workspace  device scratch of at least ss_workspace_bytes(SS_KIND_SCAN, ...) bytes;
 *              may be NULL when that is 0.  Contents on entry are ignored.
 *
 * Empty inputs (batch, dim or seqlen = 0) return SS_OK without touching memory.
 * Long sequences with little batch*dim parallelism run a chunked path (per-chunk
 * local states, a carry pass, a fix-up pass) that uses the workspace.  Only the
 * middle L-chunks are scanned twice, so when one chunk's CTAs fill at most half
 * of the GPU the first and last chunks are made longer than the others, by as
 * much as keeps every SM busy in both passes.
 * Rows that are not 16-byte aligned (seqlen * element size % 16 != 0) are read
 * in place through a view whose rows hold P of theirs (P = (16 / element size)
 * / gcd(seqlen, 16 / element size)) when P divides dim / ngroups and dstate; for
 * them the workspace is optional: given one of the reported size they may take
 * the chunked path, without it they run in one pass.  Other unaligned rows run
 * an on-chip kernel that needs no workspace.
 */
ss_status ss_selective_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                int ngroups, ss_dtype io, const void *u, const void *delta,
                                const float *A, const void *B, const void *C, const float *D,
                                const void *z, const float *delta_bias, int delta_softplus,
                                void *out, float *last_state, void *workspace,
                                size_t workspace_bytes, ss_stream_t stream);

/* Options of ss_selective_scan_fwd_opts.  Zero-initialise, then set fields. */
typedef struct ss_scan_options {
    /* Sequence split.  0: automatic; 1: one pass over the whole sequence;
     * n >= 2: the chunked long-sequence path with at most n L-chunks (each
     * starting on a multiple of the kernel's step tile, the first and last
     * possibly longer than the others; fewer if the sequence is short). */
    int chunks;
    /* Bit flags, SS_SCAN_* (0 for the default Euler step from a zero state). */
    unsigned int flags;
    /* Initial state [batch, dim, dstate] float32 (device, 16-byte aligned), or
     * NULL for h = 0.  With last_state this continues a sequence across calls:
     * scanning L1 steps, then L2 steps from the first call's last_state, equals
     * one scan of L1 + L2 steps (the recurrent form the reading notes give for
     * inference). */
    const float *h0;
    /* With SS_SCAN_CONV_SILU: the Mamba block's input branch is fused in front
     * of the scan, and `u` is its input x.  The scan then runs on
     *     u[t] = SiLU(conv_b[d] + sum_{j<4} conv_w[d, j] * x[t - 3 + j])
     * (causal depthwise Conv1D of width 4, "Mamba Block (1D)" diagram), which
     * is also the u of the D*u skip term.  conv_w [dim, 4] float32 (required),
     * conv_b [dim] float32 (NULL: 0), conv_x0 [batch, dim, 3] float32: the
     * three inputs before the sequence, oldest first (NULL: zeros) -- with h0
     * this continues a sequence.  Rows must be 16-byte aligned (seqlen *
     * element size % 16 == 0), else SS_ERR_UNSUPPORTED. */
    const float *conv_w;
    const float *conv_b;
    const float *conv_x0;
    int reserved[6]; /* must be zero */
} ss_scan_options;

/* Zero-order-hold input matrix: Bbar = (Delta*A)^-1 (exp(Delta*A) - 1) * Delta*B
 * ("Mamba Series ...", mathematical form of the selective SSM) instead of the
 * default Euler Bbar = Delta*B.  For A = 0 it is Delta*B. */
#define SS_SCAN_ZOH 1u
/* Fuse the causal Conv1D(k=4) + SiLU input branch in front of the scan. */
#define SS_SCAN_CONV_SILU 2u

/* ss_selective_scan_fwd with options (NULL options = automatic). */
ss_status ss_selective_scan_fwd_opts(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                     int ngroups, ss_dtype io, const void *u, const void *delta,
                                     const float *A, const void *B, const void *C,
                                     const float *D, const void *z, const float *delta_bias,
                                     int delta_softplus, void *out, float *last_state,
                                     void *workspace, size_t workspace_bytes,
                                     const ss_scan_options *options, ss_stream_t stream);

/*
 * ss_bidir_scan_fwd -- Vision Mamba bidirectional scan: direction 0 visits
 * positions 0..L-1, direction 1 visits L-1..0, each with its own parameters;
 * the two outputs are summed and then gated once by SiLU(z).
 *
 *   u          [batch, dim, seqlen]               io
 *   delta      [batch, 2, dim, seqlen]            io (direction 1 in reversed order:
 *                                                   its step s is token L-1-s)
 *   A          [2*dim, dstate]                    float
 *   B, C       [batch, 2, ngroups, dstate, seqlen] io (scan order, as delta)
 *   D, delta_bias [2*dim]                         float, nullable
 *   z          [batch, dim, seqlen]               io, nullable
 *   out        [batch, dim, seqlen]               io
 *   last_state [batch, 2, dim, dstate]            float, nullable (direction 1: state after position 0)
 *   workspace  ss_workspace_bytes(SS_KIND_BIDIR, ...) bytes of device scratch, 16-byte
 *              aligned, not overlapping any tensor; NULL when that is 0.
 * When rows are 16-byte aligned (seqlen * element size % 16 == 0) the two
 * directions run as two TMA-staged scans that merge through the workspace, an
 * fp32 [batch, dim, seqlen] accumulator (first direction stores, second adds,
 * gates and writes out: deterministic).
 * Otherwise the workspace is optional.  With P = (16 / element size) /
 * gcd(seqlen, 16 / element size), the number of rows whose lengths add up to a
 * 16-byte multiple: when P divides dim / ngroups and dstate, and the workspace
 * holds two fp32 slices of [batch, dim, Lp] (Lp = seqlen rounded up to a
 * 16-byte multiple), both directions run side by side as TMA scans reading the
 * tensors in place through a view whose rows hold P of theirs, each storing
 * its terms into one slice, and one more launch merges the slices by position.
 * Otherwise, given at least the size the query reports (which assumes
 * ngroups = 1: the copied B and C grow with ngroups), the call first copies u
 * (forward and reversed), delta, B and C into rows of pitch Lp in the
 * workspace and scans those.  Without a workspace (NULL), or with a smaller
 * one, the call merges on chip.  The size the query reports always covers the
 * two slices.
 */
ss_status ss_bidir_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int dstate, int ngroups,
                            ss_dtype io, const void *u, const void *delta, const float *A,
                            const void *B, const void *C, const float *D, const void *z,
                            const float *delta_bias, int delta_softplus, void *out,
                            float *last_state, void *workspace, size_t workspace_bytes,
                            ss_stream_t stream);

/*
 * ss_cross_scan2d_fwd -- VMamba SS2D cross-scan: four selective scans, one per
 * traversal order, and the cross-merge that sums them by position.
 *
 *   u          [batch, dim, H, W]                 io
 *   delta      [batch, 4, dim, H*W]               io (direction k = SS_DIR_*, in its scan order)
 *   A          [4*dim, dstate]                    float
 *   B, C       [batch, 4, ngroups, dstate, H*W]   io (scan order of each direction)
 *   D, delta_bias [4*dim]                         float, nullable
 *   z          [batch, dim, H, W]                 io, nullable (VMamba gates after a norm,
 *                                                  so its SS2D passes NULL)
 *   out        [batch, dim, H, W]                 io: sum over the four directions
 *   last_state [batch, 4, dim, dstate]            float, nullable
 *   workspace  ss_workspace_bytes(SS_KIND_CROSS2D, batch, dim, H*W, dstate) bytes,
 *              16-byte aligned, not overlapping any tensor; NULL when that is 0.
 * When rows are 16-byte aligned (H*W * element size % 16 == 0) the four
 * directions run side by side in one launch of TMA-staged scans, each storing
 * its terms into its own fp32 [batch, dim, H*W] slice of the workspace (the
 * row orders by position, the column orders by column-major index); one more
 * launch sums the four slices by position (a fixed order: deterministic) and
 * gates.  The column directions read u as row-order tiles of a transposed copy
 * of u that the call makes in the workspace first.
 * Otherwise the workspace is optional.  With P = (16 / element size) /
 * gcd(H*W, 16 / element size): when P divides dim / ngroups and dstate, and a
 * workspace of the reported size is given, the four directions run side by
 * side as TMA scans reading the maps in place through a view whose rows hold P
 * of theirs (the column directions over the transposed copy of u), each storing
 * its terms by scan step into its own fp32 slice of rows padded to 16 bytes,
 * and one more launch sums them by position.  Otherwise the whole map of a
 * channel is merged in shared memory: H*W is then limited by the per-block
 * shared-memory size (SS_ERR_UNSUPPORTED beyond it).
 */
ss_status ss_cross_scan2d_fwd(int64_t batch, int64_t dim, int64_t H, int64_t W, int dstate,
                              int ngroups, ss_dtype io, const void *u, const void *delta,
                              const float *A, const void *B, const void *C, const float *D,
                              const float *delta_bias, int delta_softplus, const void *z,
                              void *out, float *last_state, void *workspace,
                              size_t workspace_bytes, ss_stream_t stream);

/*
 * ss_selective_scan_fwd_noalloc -- ss_selective_scan_fwd_opts for callers that
 * cannot allocate device memory.  (Library addition: the pages have no
 * counterpart; it computes exactly what ss_selective_scan_fwd_opts computes.)
 *
 * Who needs it: code that runs where device allocation is not allowed or not
 * affordable -- a plug-in executed inside another engine's enqueue step, where
 * the host engine owns all device memory; a real-time loop in which a
 * cudaMalloc/cudaFree (which may synchronise the device) would break its
 * latency budget; a caller without access to any allocator at all.  Such a
 * caller cannot supply the workspace that the long-sequence chunked path of
 * ss_selective_scan_fwd needs.
 *
 * Instead of a workspace, this call uses one fixed scratch array of
 * SS_NOALLOC_SCRATCH_BYTES bytes that the library holds as static device memory
 * on every GPU that loads it, until the process exits.  It calls no cudaMalloc,
 * no cudaFree and no allocating library routine.  Arguments, layouts, options
 * and results are those of ss_selective_scan_fwd_opts, without the workspace.
 *
 * - Each call looks up the array's device address on the current device
 *   (cudaGetSymbolAddress, which allocates nothing).  The first call on a
 *   device may also load the library's kernels there: make that first call
 *   before any stream capture on the device.
 * - Calls whose chunked path would need more than SS_NOALLOC_SCRATCH_BYTES
 *   (see ss_workspace_bytes_opts) return SS_ERR_UNSUPPORTED before launching
 *   anything; pass fewer chunks or use ss_selective_scan_fwd with a workspace.
 * - Every call on a device shares the one array, which keeps the last call's
 *   contents; the chunked path writes every scratch word before reading it, so
 *   nothing needs clearing between calls.  Calls that can overlap on the GPU
 *   (different streams without ordering, or several host threads) race on the
 *   array and produce undefined results: order them on one stream.
 */
#define SS_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
ss_status ss_selective_scan_fwd_noalloc(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                        int ngroups, ss_dtype io, const void *u,
                                        const void *delta, const float *A, const void *B,
                                        const void *C, const float *D, const void *z,
                                        const float *delta_bias, int delta_softplus, void *out,
                                        float *last_state, const ss_scan_options *options,
                                        ss_stream_t stream);

/*
 * ss_selective_state_update -- one step of the recurrence, for token-by-token
 * inference (the recurrent mode of the reading notes and of the review's
 * "selective SSM" form): with h the running state,
 *     dt = Delta[b,d] + delta_bias[d];  dt = softplus(dt) if delta_softplus
 *     h[b,d,n] = exp(dt * A[d,n]) * h[b,d,n] + dt * B[b,g,n] * x[b,d]    (Euler)
 *     out[b,d] = (sum_n C[b,g,n] * h[b,d,n] + D[d] * x[b,d]) * SiLU(z[b,d])
 * It equals ss_selective_scan_fwd over one step with h0 = state and
 * last_state = state.
 *
 *   x, delta, z  [batch, dim]          io (z nullable)
 *   A            [dim, dstate]         float
 *   B, C         [batch, ngroups, dstate] io
 *   D, delta_bias [dim]                float, nullable
 *   state        [batch, dim, dstate]  float, read and overwritten in place
 *   out          [batch, dim]          io
 * flags: 0 or SS_SCAN_ZOH.  All pointers device, 16-byte aligned; out must
 * not overlap the inputs or the state.  Asynchronous on `stream`.
 */
ss_status ss_selective_state_update(int64_t batch, int64_t dim, int dstate, int ngroups,
                                    ss_dtype io, const void *x, const void *delta,
                                    const float *A, const void *B, const void *C,
                                    const float *D, const void *z, const float *delta_bias,
                                    int delta_softplus, unsigned int flags, float *state,
                                    void *out, ss_stream_t stream);

/*
 * ss_multi_scan_fwd -- ndirs (1..8) directions of any traversal over an H x W map,
 * summed by position and gated: the SS2D computation for an arbitrary list of
 * orders.  Direction k visits the map in the order orders[k] (an SS_DIR_* code;
 * `window` is the window size of the windowed ones, ignored otherwise).  Besides
 * SS2D's four orders and LocalMamba's windowed scans this covers the spatio-
 * temporal scans of a video of T frames of h x w pixels (VideoMamba), taken as a
 * map of H = T rows and W = h*w columns: SS_DIR_ROW is the spatial-first scan
 * (frame by frame) and SS_DIR_COL the temporal-first one (pixel by pixel through
 * the frames), with their reverses.
 *
 *   u, z, out   [batch, dim, H, W]          io (z nullable: no gate)
 *   delta       [batch, ndirs, dim, H*W]    io, in each direction's scan order
 *   A           [ndirs*dim, dstate]         float
 *   B, C        [batch, ndirs, ngroups, dstate, H*W]  io, in each direction's scan order
 *   D, delta_bias [ndirs*dim]               float, nullable
 *   last_state  [batch, ndirs, dim, dstate] float, nullable
 *   orders      host array of ndirs SS_DIR_* codes
 *   workspace   ss_multi_scan_workspace_bytes(batch, dim, H, W, ndirs) bytes,
 *               16-byte aligned, contents ignored: the fp32 accumulators by step
 *               (ndirs*batch*dim*H*W*4 bytes, rounded up to 256), then room for
 *               up to min(ndirs, 3) copies of u (batch*dim*H*W*4 bytes each,
 *               rounded up to 256)
 * out = (sum_k y_k + D_k*u) * SiLU(z).  Rows must be 16-byte aligned (H*W *
 * element size % 16 == 0), else SS_ERR_UNSUPPORTED.  Every direction reads u
 * as row-order tiles, forward or back to front: of u itself (the row orders),
 * or of a copy of u permuted into its base traversal's step order (column-major,
 * windows, windows column-major), made once per call in the workspace.
 * Directions run two per launch of the scan kernel, each storing its terms by
 * scan step into its own fp32 slice of the workspace; one more launch sums them
 * by position.
 */
ss_status ss_multi_scan_fwd(int64_t batch, int64_t dim, int64_t H, int64_t W, int ndirs,
                            const int *orders, int window, int dstate, int ngroups, ss_dtype io,
                            const void *u, const void *delta, const float *A, const void *B,
                            const void *C, const float *D, const float *delta_bias,
                            int delta_softplus, const void *z, void *out, float *last_state,
                            void *workspace, size_t workspace_bytes, ss_stream_t stream);

/*
 * ss_multi_scan_bwd -- gradients of ss_multi_scan_fwd (Euler input matrix, zero
 * initial states) for an upstream gradient `dout` [batch, dim, H, W] of out.
 * Direction k's gradients are those of the single-direction scan of its inputs
 * taken in its order (ss_selective_scan_bwd), with dout and z read at the
 * positions it visits; du sums the directions back by position, and dz uses the
 * sum of all directions' outputs before the gate.  Inputs as ss_multi_scan_fwd.
 * Outputs, overwritten (the summed ones zeroed on `stream` first, then fp32
 * atomic adds):
 *   du, dz      [batch, dim, H, W]              io (dz iff z given, else NULL)
 *   ddelta      [batch, ndirs, dim, H*W]        io, each direction in its scan order
 *   dA          [ndirs*dim, dstate]             float
 *   dB, dC      [batch, ndirs, ngroups, dstate, H*W] float, in each direction's scan order
 *   dD, ddelta_bias [ndirs*dim]                 float, nullable
 * workspace: ss_multi_scan_bwd_workspace_bytes(batch, dim, H, W, dstate, ndirs)
 * bytes, 16-byte aligned.  Rows must be 16-byte aligned (H*W * element size % 16
 * == 0), else SS_ERR_UNSUPPORTED.  No output may overlap an input, another output
 * or the workspace.  With a gate, one forward pass without it computes the
 * output sum dz needs.  Then, per base traversal of the order list (row-major,
 * column-major, windows, windows column-major), u, dout and z are copied into
 * that traversal's step order (no copy for the row orders) and its directions
 * run two per launch of the backward kernel, reading the copies as row-order
 * tiles, forward or back to front; one more launch sums du by position.
 */
ss_status ss_multi_scan_bwd(int64_t batch, int64_t dim, int64_t H, int64_t W, int ndirs,
                            const int *orders, int window, int dstate, int ngroups, ss_dtype io,
                            const void *u, const void *delta, const float *A, const void *B,
                            const void *C, const float *D, const float *delta_bias,
                            int delta_softplus, const void *z, const void *dout, void *du,
                            void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz,
                            float *ddelta_bias, void *workspace, size_t workspace_bytes,
                            ss_stream_t stream);

/* Workspace of ss_multi_scan_bwd (0 for an invalid shape). */
size_t ss_multi_scan_bwd_workspace_bytes(int64_t batch, int64_t dim, int64_t H, int64_t W,
                                         int dstate, int ndirs);

/*
 * ss_dwconv3x3_silu_fwd -- the input branch of VMamba's SS2D block ("Mamba Series
 * ...", VSS block structure and SS2Dv0.forwardv0: DWConv 3x3 -> SiLU -> SS2D):
 *     u[b,d,r,c] = SiLU(bias[d] + sum_{i,j=-1..1} w[d,i+1,j+1] * x[b,d,r+i,c+j])
 * with zero padding of one cell (cross-correlation, as a conv2d layer computes it).
 *   x, u [batch, dim, H, W] io; w [dim, 3, 3] float; bias [dim] float, nullable.
 * Device pointers, 16-byte aligned; u must not overlap x.  Empty shapes return
 * SS_OK.  Asynchronous on `stream`.  It is a separate pass, not fused into the
 * scan: in the SS2D block the x_proj projection that makes Delta, B, C reads u,
 * so u is in memory before the scan starts anyway.
 */
ss_status ss_dwconv3x3_silu_fwd(int64_t batch, int64_t dim, int64_t H, int64_t W, ss_dtype io,
                                const void *x, const float *w, const float *bias, void *u,
                                ss_stream_t stream);

/* Workspace of ss_multi_scan_fwd (0 for an empty or invalid shape). */
size_t ss_multi_scan_workspace_bytes(int64_t batch, int64_t dim, int64_t H, int64_t W, int ndirs);

/*
 * ss_selective_scan_bwd -- gradients of ss_selective_scan_fwd (Euler input
 * matrix, zero initial state, no options; ss_selective_scan_bwd_opts below
 * takes the options) for an upstream gradient `dout` of
 * out.  The forward call computes ("Mamba Series from Selective State Spaces
 * to Visual State Space Models": mathematical form of the selective SSM, and
 * the Mamba Block (1D) diagram)
 *     Delta'_t = softplus(delta_t + delta_bias)   (delta_t + delta_bias without the flag)
 *     h_t = exp(Delta'_t A) h_{t-1} + Delta'_t B_t u_t,   h_{-1} = 0
 *     out_t = (C_t . h_t + D u_t) * SiLU(z_t)
 * and this call writes its derivatives:
 *   du, ddelta   [batch, dim, seqlen]             io     (ddelta is w.r.t. the raw delta)
 *   dz           [batch, dim, seqlen]             io     required iff z is given, else NULL
 *   dA           [dim, dstate]                    float  summed over batch and time
 *   dB, dC       [batch, ngroups, dstate, seqlen] float  summed over the group's channels
 *   dD           [dim]                            float  nullable; summed over batch and time
 *   ddelta_bias  [dim]                            float  nullable; summed over batch and time
 * The inputs u ... delta_softplus are the forward call's (same layouts and
 * rules), and dout [batch, dim, seqlen] is io.  The forward call keeps no
 * intermediate states; this call recomputes them, holding a checkpoint every 8
 * or 16 steps in `workspace`: at least ss_workspace_bytes(SS_KIND_SCAN_BWD, batch,
 * dim, seqlen, dstate) = batch*dim*ceil(seqlen/8)*dstate*4 bytes, 16-byte
 * aligned, contents ignored.  Rows must be 16-byte aligned (seqlen * element
 * size % 16 == 0), else SS_ERR_UNSUPPORTED.  All pointers are device pointers,
 * 16-byte aligned; no output may overlap an input, another output or the
 * workspace.  Outputs are overwritten: the summed ones are zeroed on `stream`
 * first, then accumulated with fp32 atomic adds, so their last bits may differ
 * between calls.  With batch, dim or seqlen = 0 the summed outputs are zeroed
 * and nothing else is touched.  Asynchronous on `stream`.
 */
ss_status ss_selective_scan_bwd(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                int ngroups, ss_dtype io, const void *u, const void *delta,
                                const float *A, const void *B, const void *C, const float *D,
                                const void *z, const float *delta_bias, int delta_softplus,
                                const void *dout, void *du, void *ddelta, float *dA, float *dB,
                                float *dC, float *dD, void *dz, float *ddelta_bias,
                                void *workspace, size_t workspace_bytes, ss_stream_t stream);

/*
 * ss_selective_scan_bwd_opts -- gradients of ss_selective_scan_fwd_opts: the
 * backward pass of a single-direction scan run with options.  The arguments
 * up to ddelta_bias are those of ss_selective_scan_bwd; `options` are the
 * forward call's (chunks must be 0), and the options' tensors get their
 * gradients in `extras`:
 *   SS_SCAN_ZOH        the zero-order-hold input matrix Bbar = (exp(Delta'A) - 1)/A * B
 *                      ("Mamba Series ...", mathematical form of the selective
 *                      SSM): dDelta' gains exp(Delta'A) B u in place of B u,
 *                      du and dB use (exp(Delta'A) - 1)/A in place of Delta', and
 *                      dA gains the derivative of that factor.
 *   options.h0         the initial state; extras.dh0 [batch, dim, dstate] float
 *                      (nullable) receives Abar_0 (.) dh_0, its gradient.
 *   SS_SCAN_CONV_SILU  the fused Conv1D + SiLU: `u` is its input x, `du`
 *                      receives the gradient with respect to x, and
 *                      extras.dconv_w [dim, 4] (required), dconv_b [dim] and
 *                      dconv_x0 [batch, dim, 3] (nullable; each only with its
 *                      tensor in the options) the gradients of the weights, bias
 *                      and history.  The convolution runs as passes of its own
 *                      around the scan's backward kernel: its output u is
 *                      recomputed into the workspace in the I/O type (so for
 *                      bf16 I/O the backward pass sees u rounded to bf16, where
 *                      the fused forward kept it in float32) and the scan's du
 *                      goes to the workspace in float32 before the
 *                      convolution's gradients are formed.
 * dA, dB, dC, dD, ddelta_bias, dconv_w and dconv_b are sums: zeroed on
 * `stream`, then accumulated with fp32 atomic adds.  Workspace: at least
 * ss_workspace_bytes_opts(SS_KIND_SCAN_BWD, batch, dim, seqlen, dstate,
 * options) bytes.  Every extras tensor is a device pointer, 16-byte aligned.
 */
typedef struct ss_scan_bwd_extras {
    float *dh0;      /* [batch, dim, dstate], nullable */
    float *dconv_w;  /* [dim, 4] */
    float *dconv_b;  /* [dim], nullable */
    float *dconv_x0; /* [batch, dim, 3], nullable */
    int reserved[8]; /* must be zero */
} ss_scan_bwd_extras;
ss_status ss_selective_scan_bwd_opts(int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                                     int ngroups, ss_dtype io, const void *u, const void *delta,
                                     const float *A, const void *B, const void *C, const float *D,
                                     const void *z, const float *delta_bias, int delta_softplus,
                                     const void *dout, void *du, void *ddelta, float *dA, float *dB,
                                     float *dC, float *dD, void *dz, float *ddelta_bias,
                                     const ss_scan_options *options, const ss_scan_bwd_extras *extras,
                                     void *workspace, size_t workspace_bytes, ss_stream_t stream);

/* Workspace bytes a call of the given kind and shape needs (0 if none), for
 * either I/O dtype (the larger of the two).  For SS_KIND_CROSS2D pass
 * seqlen = H*W.  Host computation only.  A call given a non-NULL workspace of
 * at least this size never fails for lack of one. */
size_t ss_workspace_bytes(int kind, int64_t batch, int64_t dim, int64_t seqlen, int dstate);

/* Same for ss_selective_scan_fwd_opts with the given options. */
size_t ss_workspace_bytes_opts(int kind, int64_t batch, int64_t dim, int64_t seqlen, int dstate,
                               const ss_scan_options *options);

/* Reads and clears the library's device error word for the current device after
 * synchronising `stream` (this call does synchronise).  Returns SS_OK, or
 * SS_ERR_TIMEOUT if a kernel abandoned a bounded wait since the last call, or
 * SS_ERR_CUDA if the synchronisation itself failed. */
ss_status ss_get_device_status(ss_stream_t stream);

/* Thread-local message describing the last error returned on this thread. */
const char *ss_last_error_string(void);

/* Version string of the library build. */
const char *ss_version(void);

/* Diagnostics: sets the time budget, in nanoseconds, of every bounded wait in
 * the kernels on the current device (default 1 s; 0 restores the default).
 * A wait that runs out records SS_ERR_TIMEOUT for ss_get_device_status, lets
 * the copies it issued land, and ends its CTA; outputs of that call are then
 * undefined.  Used to test the timeout path. */
ss_status ss_debug_set_wait_budget_ns(uint64_t ns);

/* Diagnostics: flags of the current device (0 = normal operation).
 * SS_DEBUG_SKIP_FIRST_COPY: in every launch of the single-direction TMA scan,
 * the first thread block never issues the copies of its first tile, so its
 * bounded wait for that tile runs out: the call then reports SS_ERR_TIMEOUT
 * through ss_get_device_status and the outputs of that call are undefined.
 * This is how the timeout path is tested without faulting or hanging the GPU.
 * Returns SS_ERR_INVALID_ARG for unknown bits. */
#define SS_DEBUG_SKIP_FIRST_COPY 1u
ss_status ss_debug_set_flags(uint32_t flags);

#ifdef __cplusplus
}
#endif

#endif /* SSSCAN_H */
