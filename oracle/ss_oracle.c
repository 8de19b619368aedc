/*
 * ss_oracle.c -- float64 CPU oracle for the selective state-space scan.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check and the CPU-baseline leg of the benchmark may load this file's
 * library.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (sources, by page title and section):
 *   - "Mamba Series from Selective State Spaces to Visual State Space Models",
 *     section "选择性 SSM 的数学形式" (the mathematical form of the selective SSM):
 *       discretisation  Abar = exp(Delta*A),
 *                       Bbar = (Delta*A)^-1 (exp(Delta*A) - I) * Delta*B   (zero-order hold),
 *       selection       Delta = softplus(W_Delta x + b_Delta), B = W_B x, C = W_C x.
 *     The simplified (Euler) input matrix Bbar = Delta*B is the default; the
 *     zero-order-hold form is selected by a flag.
 *   - same page, block diagram "Mamba Block (1D)": the scan output is multiplied
 *     by SiLU of the gate branch z.
 *   - same page, "关键代码" (key code), SS2D forward: four traversal orders of an
 *     H x W map (row-major, column-major, and the reverse of each), one scan per
 *     order, outputs mapped back to H x W and summed; softplus is applied to
 *     Delta + delta_bias, and a skip term D*u is part of each scan.  There the
 *     per-direction Delta, B and C are projections of the already reordered
 *     sequences xs, so each direction receives them in its own scan order;
 *     only the input x (u here) is gathered from the map.
 *   - "从LSTM到Mamba：为什么说双向状态空间模型是处理视觉序列的'潜力股'？",
 *     section 3.1: bidirectional scan = a forward scan plus a scan of the reversed
 *     sequence with its own parameters.  The two outputs are SUMMED here (not
 *     concatenated), with the backward output flipped back to token order.
 *
 * Recurrence, per (batch b, direction k, channel d), over scan steps s = 0..L-1
 * visiting positions p = pi_k(s):
 *     dt      = Delta_k[d, s] + bias_k[d];   dt = softplus(dt) if requested
 *     h_n     = exp(dt*A_k[d,n]) * h_n + Bbar_{k,n}(s) * u[d, p]      (n = 0..N-1)
 *     y_k(p)  = sum_n C_k[g, n, s] * h_n + D_k[d] * u[d, p]
 * with h = 0 (or a caller-given h0) before the first step, then
 *     out[d, p] = (sum_k y_k(p)) * (z ? z*sigmoid(z) : 1).
 * u, z and out are indexed by position p; the per-direction Delta, B, C are
 * indexed by scan step s (each direction's own order).
 * Channel d uses group g = d / (dim / ngroups).
 *
 * Everything is float64 and strictly sequential; libm exp/log1p only.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

/* Traversal orders of one direction. */
#define SSOR_ORDER_FWD 0     /* positions 0, 1, ..., L-1 (row-major for a map) */
#define SSOR_ORDER_REV 1     /* positions L-1, ..., 0                          */
#define SSOR_ORDER_COL 2     /* column-major over an H x W map                 */
#define SSOR_ORDER_COL_REV 3 /* reverse of column-major                        */
/* Windowed orders ("LocalMamba: Visual State Space Model with Windowed Selective
 * Scan", abstract: the image is divided into windows and scanned window by
 * window).  Read here as: the map is cut into w x w windows -- the windows of
 * the last band of rows and of the last column are cut short when w does not
 * divide H or W -- and the windows are visited one after another. */
#define SSOR_ORDER_WIN 4         /* windows row-major, each window row-major          */
#define SSOR_ORDER_WIN_REV 5     /* reverse of SSOR_ORDER_WIN                          */
#define SSOR_ORDER_WIN_COL 6     /* windows column-major, each window column-major     */
#define SSOR_ORDER_WIN_COL_REV 7 /* reverse of SSOR_ORDER_WIN_COL                      */

/* softplus(x) = log(1 + exp(x)), written in the overflow-free form. */
static double ssor_softplus(double x) {
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* Position visited at scan step s by a direction with the given order, for an
 * H x W map stored row-major (a plain sequence is H = 1, W = L). */
static int64_t ssor_position(int order, int64_t s, int64_t H, int64_t W) {
    int64_t L = H * W;
    int64_t r;
    switch (order) {
    case SSOR_ORDER_FWD: return s;
    case SSOR_ORDER_REV: return L - 1 - s;
    case SSOR_ORDER_COL: return (s % H) * W + s / H;
    case SSOR_ORDER_COL_REV: r = L - 1 - s; return (r % H) * W + r / H;
    default: return -1;
    }
}

/* Positions of a windowed order, step by step, written out by nested loops over
 * the windows and the cells inside each (col = 0: rows outer; col = 1: the
 * transposed map, columns outer).  Fills pos[0 .. H*W). */
static void ssor_window_walk(int64_t H, int64_t W, int64_t w, int col, int64_t *pos) {
    int64_t s = 0;
    if (!col) {
        for (int64_t r0 = 0; r0 < H; r0 += w)
            for (int64_t c0 = 0; c0 < W; c0 += w)
                for (int64_t r = r0; r < r0 + w && r < H; ++r)
                    for (int64_t c = c0; c < c0 + w && c < W; ++c) pos[s++] = r * W + c;
    } else {
        for (int64_t c0 = 0; c0 < W; c0 += w)
            for (int64_t r0 = 0; r0 < H; r0 += w)
                for (int64_t c = c0; c < c0 + w && c < W; ++c)
                    for (int64_t r = r0; r < r0 + w && r < H; ++r) pos[s++] = r * W + c;
    }
}

/* Position table of any order (win: window size of the windowed orders, >= 1).
 * Returns 0, or -1 for an unknown order or a bad window size. */
int ssor_order_table(int order, int64_t H, int64_t W, int64_t win, int64_t *pos) {
    const int64_t L = H * W;
    if (H <= 0 || W <= 0 || !pos) return -1;
    if (order >= SSOR_ORDER_WIN && order <= SSOR_ORDER_WIN_COL_REV) {
        if (win < 1) return -1;
        const int col = (order == SSOR_ORDER_WIN_COL || order == SSOR_ORDER_WIN_COL_REV);
        ssor_window_walk(H, W, win, col, pos);
        if (order == SSOR_ORDER_WIN_REV || order == SSOR_ORDER_WIN_COL_REV)
            for (int64_t i = 0, j = L - 1; i < j; ++i, --j) {
                const int64_t t = pos[i];
                pos[i] = pos[j];
                pos[j] = t;
            }
        return 0;
    }
    for (int64_t s = 0; s < L; ++s) {
        pos[s] = ssor_position(order, s, H, W);
        if (pos[s] < 0) return -1;
    }
    return 0;
}

/*
 * ssor_scan: the general oracle.
 *
 * Layouts (all float64, C-contiguous):
 *   u          [batch, dim, L]              L = H*W
 *   delta      [batch, K, dim, L]            (scan order of each direction)
 *   A          [K*dim, N]
 *   Bm, Cm     [batch, K, ngroups, N, L]     (scan order of each direction)
 *   Dv         [K*dim]        (NULL: no skip term)
 *   z          [batch, dim, L] (NULL: no gate)
 *   bias       [K*dim]        (NULL: zero)
 *   h0         [batch, K, dim, N] (NULL: zero initial state)
 *   out        [batch, dim, L]
 *   last_state [batch, K, dim, N] (NULL: not written)
 *   orders     [K]  one SSOR_ORDER_* per direction
 *   win        window size of the windowed orders (ignored by the others)
 * Returns 0, or -1 on an invalid argument.
 */
int ssor_scan(int64_t batch, int64_t dim, int64_t H, int64_t W, int64_t N, int64_t ngroups,
              int64_t K, const int *orders, int64_t win,
              const double *u, const double *delta, const double *A, const double *Bm,
              const double *Cm, const double *Dv, const double *z, const double *bias,
              int delta_softplus, int zoh, const double *h0, double *out, double *last_state,
              double *h_work /* scratch of N doubles */) {
    if (batch < 0 || dim <= 0 || H <= 0 || W <= 0 || N <= 0 || ngroups <= 0 || K <= 0) return -1;
    if (dim % ngroups != 0) return -1;
    if (!orders || !u || !delta || !A || !Bm || !Cm || !out || !h_work) return -1;
    const int64_t L = H * W;
    const int64_t dpg = dim / ngroups;

    for (int64_t i = 0; i < batch * dim * L; ++i) out[i] = 0.0;

    /* windowed orders: the position of each step from a table */
    int64_t *wtab = NULL;
    for (int64_t k = 0; k < K; ++k)
        if (orders[k] >= SSOR_ORDER_WIN) {
            wtab = (int64_t *)malloc(sizeof(int64_t) * L * K);
            if (!wtab) return -1;
            break;
        }
    for (int64_t k = 0; wtab && k < K; ++k)
        if (orders[k] >= SSOR_ORDER_WIN && ssor_order_table(orders[k], H, W, win, wtab + k * L)) {
            free(wtab);
            return -1;
        }

    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t k = 0; k < K; ++k) {
            for (int64_t d = 0; d < dim; ++d) {
                const int64_t g = d / dpg;
                const double *A_row = A + (k * dim + d) * N;
                const double Dd = Dv ? Dv[k * dim + d] : 0.0;
                const double bd = bias ? bias[k * dim + d] : 0.0;
                const double *u_row = u + (b * dim + d) * L;
                const double *dl_row = delta + ((b * K + k) * dim + d) * L;
                const double *B_grp = Bm + ((b * K + k) * ngroups + g) * N * L;
                const double *C_grp = Cm + ((b * K + k) * ngroups + g) * N * L;
                double *o_row = out + (b * dim + d) * L;
                double *h = h_work;
                for (int64_t n = 0; n < N; ++n)
                    h[n] = h0 ? h0[((b * K + k) * dim + d) * N + n] : 0.0;

                for (int64_t s = 0; s < L; ++s) {
                    const int64_t p = orders[k] >= SSOR_ORDER_WIN ? wtab[k * L + s]
                                                                  : ssor_position(orders[k], s, H, W);
                    if (p < 0) {
                        free(wtab);
                        return -1;
                    }
                    double dt = dl_row[s] + bd;
                    if (delta_softplus) dt = ssor_softplus(dt);
                    const double up = u_row[p];
                    double y = 0.0;
                    for (int64_t n = 0; n < N; ++n) {
                        const double a = A_row[n];
                        const double abar = exp(dt * a);
                        double bbar;
                        if (zoh && a != 0.0)
                            bbar = (abar - 1.0) / a * B_grp[n * L + s];   /* (dA)^-1 (e^{dA}-1) dB */
                        else
                            bbar = dt * B_grp[n * L + s];                 /* Euler: dB */
                        h[n] = abar * h[n] + bbar * up;
                        y += C_grp[n * L + s] * h[n];
                    }
                    o_row[p] += y + Dd * up;
                }
                if (last_state)
                    for (int64_t n = 0; n < N; ++n)
                        last_state[((b * K + k) * dim + d) * N + n] = h[n];
            }
        }
    }
    free(wtab);

    if (z) {
        for (int64_t i = 0; i < batch * dim * L; ++i) {
            const double zi = z[i];
            out[i] *= zi / (1.0 + exp(-zi));   /* SiLU(z) = z * sigmoid(z) */
        }
    }
    return 0;
}

/*
 * ssor_conv_silu: the Mamba block's input branch before the scan ("Mamba
 * Series ...", block diagram "Mamba Block (1D)": Conv1D(k=4) -> SiLU -> SSM):
 * a causal depthwise convolution of width KW along the sequence, plus a bias,
 * then SiLU:
 *     v = bias[d] + sum_{j=0..KW-1} w[d, j] * x[b, d, t - (KW-1) + j]
 *     u[b, d, t] = v * sigmoid(v)
 * Steps before the sequence read x0[b, d, 0..KW-2] (the KW-1 inputs that came
 * before it, oldest first), or zeros when x0 is NULL.
 *   x, u [batch, dim, L]; w [dim, KW]; bias [dim] (NULL: 0).  Returns 0 or -1.
 */
int ssor_conv_silu(int64_t batch, int64_t dim, int64_t L, int64_t KW, const double *x,
                   const double *w, const double *bias, const double *x0, double *u) {
    if (batch < 0 || dim <= 0 || L < 0 || KW <= 0 || !x || !w || !u) return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const double *xr = x + (b * dim + d) * L;
            const double *x0r = x0 ? x0 + (b * dim + d) * (KW - 1) : NULL;
            for (int64_t t = 0; t < L; ++t) {
                double v = bias ? bias[d] : 0.0;
                for (int64_t j = 0; j < KW; ++j) {
                    const int64_t s = t - (KW - 1) + j;   /* input step */
                    double xv;
                    if (s >= 0) xv = xr[s];
                    else xv = x0r ? x0r[(KW - 1) + s] : 0.0;
                    v += w[d * KW + j] * xv;
                }
                u[(b * dim + d) * L + t] = v / (1.0 + exp(-v));
            }
        }
    }
    return 0;
}

/*
 * ssor_dwconv3x3_silu: the input branch of VMamba's SS2D block ("Mamba Series
 * ...", VSS block structure and SS2Dv0.forwardv0: DWConv 3x3 -> SiLU): a
 * depthwise 3 x 3 cross-correlation with zero padding of one cell and a bias,
 * then SiLU:
 *     v = bias[d] + sum_{i,j in -1..1} w[d, i+1, j+1] * x[b, d, r+i, c+j]   (0 outside the map)
 *     u[b, d, r, c] = v * sigmoid(v)
 *   x, u [batch, dim, H, W]; w [dim, 3, 3]; bias [dim] (NULL: 0).  Returns 0 or -1.
 */
int ssor_dwconv3x3_silu(int64_t batch, int64_t dim, int64_t H, int64_t W, const double *x,
                        const double *w, const double *bias, double *u) {
    if (batch < 0 || dim <= 0 || H <= 0 || W <= 0 || !x || !w || !u) return -1;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const double *xp = x + (b * dim + d) * H * W;
            for (int64_t r = 0; r < H; ++r) {
                for (int64_t c = 0; c < W; ++c) {
                    double v = bias ? bias[d] : 0.0;
                    for (int64_t i = -1; i <= 1; ++i) {
                        for (int64_t j = -1; j <= 1; ++j) {
                            const int64_t rr = r + i, cc = c + j;
                            if (rr < 0 || rr >= H || cc < 0 || cc >= W) continue;
                            v += w[d * 9 + (i + 1) * 3 + (j + 1)] * xp[rr * W + cc];
                        }
                    }
                    u[((b * dim + d) * H + r) * W + c] = v / (1.0 + exp(-v));
                }
            }
        }
    }
    return 0;
}

/*
 * ssor_scan_bwd: gradients of the single-direction scan (Euler input matrix,
 * zero initial state) for an upstream gradient dy of out.  The forward pass is
 * the recurrence above; the pages state that the backward pass recomputes the
 * intermediate states rather than storing them ("Mamba Series ...", core
 * insight 1, item 3; reading notes 3.3.2) -- here simply by storing one row's
 * states in h_work.  Per (b, d), with s_t = C_t . h_t + D u_t and y_t = s_t g_t,
 * g = SiLU(z):
 *     ds_t  = dy_t g_t;            dz_t = dy_t s_t SiLU'(z_t)
 *     dh_t  = ds_t C_t + abar_{t+1} (.) dh_{t+1}          (reverse in t)
 *     dabar = dh_t (.) h_{t-1}
 *     dDelta'_t = sum_n (dabar A abar + dh B u)_n;  dDelta_t = dDelta'_t softplus'(.)
 *     dA_n += dabar abar Delta';  dB_t += dh Delta' u;  dC_t += ds h;
 *     du_t  = ds D + sum_n dh Delta' B;  dD += ds u;  dbias += dDelta_t
 * dA, dD, dbias sum over the batch; dB, dC sum over the channels of a group.
 * Layouts as ssor_scan with K = 1; h_work holds L*N doubles.  Outputs are
 * overwritten.  Returns 0 or -1.
 *
 * The forward options of ssor_scan change the recurrence as follows.
 *   zoh: the input term is q_n = (abar_n - 1)/a_n * B_n u ("Mamba Series ...",
 *     discretisation rule; the Euler term Delta' B_n u where a_n = 0, its limit),
 *     so, from dq/dDelta' = abar B u and dq/da = B u (Delta' abar a - (abar - 1)) / a^2:
 *       dDelta'_t += dh abar B u (in place of dh B u),
 *       dA_n += dh B u (Delta' abar a - (abar - 1)) / a^2,
 *       dB_t += dh (abar - 1)/a u,   du_t += sum_n dh (abar - 1)/a B.
 *   h0 [batch, dim, N] (NULL: zero): the state before step 0, so step 0's decay
 *     term uses it, and its gradient is dh0 = abar_0 (.) dh_0, written to dh0
 *     (nullable).
 */
int ssor_scan_bwd_ext(int64_t batch, int64_t dim, int64_t L, int64_t N, int64_t ngroups,
                      const double *u, const double *delta, const double *A, const double *Bm,
                      const double *Cm, const double *Dv, const double *z, const double *bias,
                      int delta_softplus, int zoh, const double *h0, const double *dy, double *du,
                      double *ddelta, double *dA, double *dB, double *dC, double *dD, double *dz,
                      double *dbias, double *dh0, double *h_work) {
    if (batch < 0 || dim <= 0 || L <= 0 || N <= 0 || ngroups <= 0 || dim % ngroups) return -1;
    if (!u || !delta || !A || !Bm || !Cm || !dy || !du || !ddelta || !dA || !dB || !dC || !h_work)
        return -1;
    const int64_t dpg = dim / ngroups;
    for (int64_t i = 0; i < batch * dim * L; ++i) du[i] = ddelta[i] = 0.0;
    if (dz) for (int64_t i = 0; i < batch * dim * L; ++i) dz[i] = 0.0;
    for (int64_t i = 0; i < dim * N; ++i) dA[i] = 0.0;
    for (int64_t i = 0; i < batch * ngroups * N * L; ++i) dB[i] = dC[i] = 0.0;
    if (dD) for (int64_t i = 0; i < dim; ++i) dD[i] = 0.0;
    if (dbias) for (int64_t i = 0; i < dim; ++i) dbias[i] = 0.0;

    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t grp = d / dpg;
            const double *Ar = A + d * N;
            const double Dd = Dv ? Dv[d] : 0.0;
            const double bd = bias ? bias[d] : 0.0;
            const int64_t row = (b * dim + d) * L;
            const double *Bg = Bm + (b * ngroups + grp) * N * L;
            const double *Cg = Cm + (b * ngroups + grp) * N * L;
            double *dBg = dB + (b * ngroups + grp) * N * L;
            double *dCg = dC + (b * ngroups + grp) * N * L;
            const double *h0r = h0 ? h0 + (b * dim + d) * N : NULL;
            /* forward: states of every step */
            for (int64_t t = 0; t < L; ++t) {
                double dt = delta[row + t] + bd;
                if (delta_softplus) dt = ssor_softplus(dt);
                for (int64_t n = 0; n < N; ++n) {
                    const double a = Ar[n];
                    const double abar = exp(a * dt);
                    const double prev = t ? h_work[(t - 1) * N + n] : (h0r ? h0r[n] : 0.0);
                    const double bq = (zoh && a != 0.0) ? (abar - 1.0) / a : dt;  /* Bbar / B */
                    h_work[t * N + n] = abar * prev + bq * Bg[n * L + t] * u[row + t];
                }
            }
            /* reverse: dh carries the gradient of the state after step t */
            double dh_next_scaled[64 + 1];
            double *carry = N <= 64 ? dh_next_scaled : NULL;
            if (!carry) return -1;
            for (int64_t n = 0; n < N; ++n) carry[n] = 0.0;   /* abar_{t+1} dh_{t+1} */
            for (int64_t t = L - 1; t >= 0; --t) {
                const double r = delta[row + t] + bd;
                const double dt = delta_softplus ? ssor_softplus(r) : r;
                const double dsp = delta_softplus ? 1.0 / (1.0 + exp(-r)) : 1.0;  /* softplus' */
                double s = Dd * u[row + t];
                for (int64_t n = 0; n < N; ++n) s += Cg[n * L + t] * h_work[t * N + n];
                double gate = 1.0;
                if (z) {
                    const double zz = z[row + t];
                    const double sg = 1.0 / (1.0 + exp(-zz));
                    gate = zz * sg;
                    dz[row + t] = dy[row + t] * s * sg * (1.0 + zz * (1.0 - sg));
                }
                const double ds = dy[row + t] * gate;
                if (dD) dD[d] += ds * u[row + t];
                double dut = ds * Dd;
                double ddt = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double a = Ar[n];
                    const double abar = exp(a * dt);
                    const double prev = t ? h_work[(t - 1) * N + n] : (h0r ? h0r[n] : 0.0);
                    const double dh = ds * Cg[n * L + t] + carry[n];
                    dCg[n * L + t] += ds * h_work[t * N + n];
                    const double dabar = dh * prev;
                    if (zoh && a != 0.0) {
                        const double bq = (abar - 1.0) / a;
                        const double bu = Bg[n * L + t] * u[row + t];
                        ddt += dabar * abar * a + dh * abar * bu;
                        dA[d * N + n] += dabar * abar * dt + dh * bu * (dt * abar * a - (abar - 1.0)) / (a * a);
                        dBg[n * L + t] += dh * bq * u[row + t];
                        dut += dh * bq * Bg[n * L + t];
                    } else {
                        ddt += dabar * abar * a + dh * Bg[n * L + t] * u[row + t];
                        dA[d * N + n] += dabar * abar * dt;
                        dBg[n * L + t] += dh * dt * u[row + t];
                        dut += dh * dt * Bg[n * L + t];
                    }
                    carry[n] = abar * dh;
                }
                du[row + t] = dut;
                ddelta[row + t] = ddt * dsp;
                if (dbias) dbias[d] += ddt * dsp;
            }
            if (dh0)
                for (int64_t n = 0; n < N; ++n) dh0[(b * dim + d) * N + n] = carry[n];
        }
    }
    return 0;
}

/* The Euler, zero-initial-state case of ssor_scan_bwd_ext. */
int ssor_scan_bwd(int64_t batch, int64_t dim, int64_t L, int64_t N, int64_t ngroups,
                  const double *u, const double *delta, const double *A, const double *Bm,
                  const double *Cm, const double *Dv, const double *z, const double *bias,
                  int delta_softplus, const double *dy, double *du, double *ddelta, double *dA,
                  double *dB, double *dC, double *dD, double *dz, double *dbias,
                  double *h_work) {
    return ssor_scan_bwd_ext(batch, dim, L, N, ngroups, u, delta, A, Bm, Cm, Dv, z, bias,
                             delta_softplus, 0, NULL, dy, du, ddelta, dA, dB, dC, dD, dz, dbias,
                             NULL, h_work);
}

/*
 * ssor_conv_silu_bwd: gradients of ssor_conv_silu for an upstream gradient du
 * of u.  With v_t the pre-activation, dv_t = du_t SiLU'(v_t),
 * SiLU'(v) = sigmoid(v) (1 + v (1 - sigmoid(v))), and, for each tap j reading
 * input step s = t - (KW-1) + j:
 *     dx[s] += w[j] dv_t  (s >= 0),   dx0[(KW-1) + s] += w[j] dv_t  (s < 0)
 *     dw[d, j] += x[s] dv_t (x0 for s < 0),   dbias[d] += dv_t
 * dw and dbias sum over the batch.  dx [batch, dim, L]; dw [dim, KW]; dbias
 * [dim] and dx0 [batch, dim, KW-1] nullable.  Outputs are overwritten.
 * Returns 0 or -1.
 */
int ssor_conv_silu_bwd(int64_t batch, int64_t dim, int64_t L, int64_t KW, const double *x,
                       const double *w, const double *bias, const double *x0, const double *du,
                       double *dx, double *dw, double *dbias, double *dx0) {
    if (batch < 0 || dim <= 0 || L < 0 || KW <= 0 || !x || !w || !du || !dx || !dw) return -1;
    for (int64_t i = 0; i < batch * dim * L; ++i) dx[i] = 0.0;
    for (int64_t i = 0; i < dim * KW; ++i) dw[i] = 0.0;
    if (dbias) for (int64_t i = 0; i < dim; ++i) dbias[i] = 0.0;
    if (dx0) for (int64_t i = 0; i < batch * dim * (KW - 1); ++i) dx0[i] = 0.0;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const double *xr = x + (b * dim + d) * L;
            const double *x0r = x0 ? x0 + (b * dim + d) * (KW - 1) : NULL;
            double *dxr = dx + (b * dim + d) * L;
            double *dx0r = dx0 ? dx0 + (b * dim + d) * (KW - 1) : NULL;
            for (int64_t t = 0; t < L; ++t) {
                double v = bias ? bias[d] : 0.0;
                for (int64_t j = 0; j < KW; ++j) {
                    const int64_t s = t - (KW - 1) + j;
                    v += w[d * KW + j] * (s >= 0 ? xr[s] : (x0r ? x0r[(KW - 1) + s] : 0.0));
                }
                const double sg = 1.0 / (1.0 + exp(-v));
                const double dv = du[(b * dim + d) * L + t] * sg * (1.0 + v * (1.0 - sg));
                if (dbias) dbias[d] += dv;
                for (int64_t j = 0; j < KW; ++j) {
                    const int64_t s = t - (KW - 1) + j;
                    if (s >= 0) {
                        dxr[s] += w[d * KW + j] * dv;
                        dw[d * KW + j] += xr[s] * dv;
                    } else {
                        if (dx0r) dx0r[(KW - 1) + s] += w[d * KW + j] * dv;
                        if (x0r) dw[d * KW + j] += x0r[(KW - 1) + s] * dv;
                    }
                }
            }
        }
    }
    return 0;
}

/* Exposed for the oracle's own pin tests: the softplus used above. */
double ssor_softplus_scalar(double x) { return ssor_softplus(x); }

/* Exposed for the oracle's own pin tests: the position map used above. */
int64_t ssor_position_of(int order, int64_t s, int64_t H, int64_t W) {
    return ssor_position(order, s, H, W);
}
