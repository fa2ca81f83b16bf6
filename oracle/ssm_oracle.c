/*
 * ssm_oracle.c -- plain, slow, sequential fp64 CPU oracle of the selective
 * state-space (S6) hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header or constant with the
 * CUDA path.
 *
 * Every routine walks the definition in the order the sources state it:
 * one channel (b, d) at a time, one time step at a time, one state index n at
 * a time, in double precision, with no blocking, fusion or reordering.
 *
 * Sources (pages on the selective state-space model, "Mamba"):
 *  [P1] "Mamba 模型" (gaos6e.github.io), block flowchart: conv node
 *       "Uc_t = sum_i W_conv_i * U_(t-i)", SiLU node "Xc_t = Uc_t*sigmoid(Uc_t)",
 *       softplus node "Delta_t = softplus(dt_raw_t W_dt + b_dt)", discretise
 *       node "Abar_t = exp(Delta_t A)", scan node
 *       "h_t = Abar_t h_(t-1) + Bbar_t Xc_t", readout node
 *       "Y_t = C_t h_t + D Xc_t", gate nodes "G_t = Z_t*sigmoid(Z_t)",
 *       "Yg_t = Y_t * G_t"; section "为什么 Mamba 推理更省" for the one-token
 *       update state <- update(state, x_t).
 *  [P3] "Mamba 与状态空间模型" (world.lapla.si), section "模型省略了什么":
 *       the simplified rule Bbar = Delta*B; section 03: the short conv keeps
 *       the last 4 inputs.
 *  [P4] pnsm.cn overview, section "状态空间模型（SSM）基础": zero-order-hold
 *       discretisation; section "Mamba-1：选择性状态空间": diagonal A, one
 *       independent SSM per channel.
 *  [P5] mhpn.cn, section 3.1: Abar = exp(Delta A), Bbar = (Abar - I) A^-1 B.
 *
 * Parity pins (all in the CPU test suite): Theorem 1 gate reduction, ODE
 * (matrix-exponential) check of the zero-order-hold step, the LTI convolution
 * identity, the unrolled closed form, the Delta limits, chunk invariance,
 * a library conv1d, decode/scan agreement and central finite differences for
 * the backward.  No routine here is "parity unpinned".
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

/* softplus(x) = log(1 + e^x), written as max(x,0) + log1p(e^-|x|) so that it
 * neither overflows nor loses the small-x tail.  [P1] softplus node. */
static double o_softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

static double o_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* SiLU(x) = x * sigmoid(x).  [P1] SiLU node and gate node. */
static double o_silu(double x) { return x * o_sigmoid(x); }

/* Zero-order-hold input coefficient (e^{delta A} - 1) / A, and its limit
 * delta as A -> 0.  [P5] section 3.1 (Bbar = (Abar - I) A^-1 B, diagonal A);
 * [P4] ZOH discretisation.  Simplified rule: the coefficient is delta.
 * [P3] "模型省略了什么". */
static double o_bbar_coef(double delta, double A, int zoh)
{
    if (!zoh) return delta;
    if (A == 0.0) return delta;
    return expm1(delta * A) / A;
}

/* d/dA of the ZOH coefficient: delta^2 * phi(delta A) with
 * phi(x) = (x e^x - (e^x - 1)) / x^2 = sum_{m>=2} x^{m-2} (m-1)/m!.
 * The series is used near 0, where the closed form cancels. */
static double o_phi(double x)
{
    if (fabs(x) < 1e-2) {
        double s = 0.0, term_pow = 1.0, fact = 2.0; /* m = 2: x^0 * 1/2! */
        for (int m = 2; m < 14; m++) {
            s += term_pow * (double)(m - 1) / fact;
            term_pow *= x;
            fact *= (double)(m + 1);
        }
        return s;
    }
    return (x * exp(x) - expm1(x)) / (x * x);
}

/* ------------------------------------------------------------------------ */
/* Selective scan, forward.  [P1] softplus, discretise, scan, readout and gate
 * nodes, in that order; [P4] one independent N-state SSM per channel.
 *
 * Layouts (all contiguous, row-major):
 *   u, dt, z, out : (batch, dim, seqlen)
 *   A             : (dim, dstate)
 *   Bm, Cm        : (batch, dstate, seqlen)  -- shared by every channel d
 *   Dskip, bias   : (dim)                   -- NULL means zero
 *   h0, hN        : (batch, dim, dstate)    -- NULL means zero / not wanted
 *   z             : NULL means no gate
 * Only channels c = b*dim + d with ch_begin <= c < ch_end are computed.
 * Returns 0, or -1 on a bad argument. */
int oracle_scan_fwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                    const double* u, const double* dt, const double* z,
                    const double* A, const double* Bm, const double* Cm,
                    const double* Dskip, const double* bias,
                    const double* h0, int zoh, int delta_softplus,
                    double* out, double* hN, int64_t ch_begin, int64_t ch_end)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return -1;
    if (ch_begin < 0 || ch_end > batch * dim || ch_begin > ch_end) return -1;
    double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
    if (!h) return -1;
    for (int64_t c = ch_begin; c < ch_end; c++) {
        const int64_t b = c / dim, d = c % dim;
        const double* uc = u + c * seqlen;
        const double* dtc = dt + c * seqlen;
        const double* zc = z ? z + c * seqlen : NULL;
        const double* Bb = Bm + b * dstate * seqlen;
        const double* Cb = Cm + b * dstate * seqlen;
        const double* Ad = A + d * dstate;
        const double Dd = Dskip ? Dskip[d] : 0.0;
        const double bd = bias ? bias[d] : 0.0;
        for (int64_t n = 0; n < dstate; n++) h[n] = h0 ? h0[c * dstate + n] : 0.0;
        for (int64_t t = 0; t < seqlen; t++) {
            const double v = dtc[t] + bd;
            const double delta = delta_softplus ? o_softplus(v) : v;
            double y = 0.0;
            for (int64_t n = 0; n < dstate; n++) {
                const double a = exp(delta * Ad[n]);                        /* Abar */
                const double bbar = o_bbar_coef(delta, Ad[n], zoh) * Bb[n * seqlen + t];
                h[n] = a * h[n] + bbar * uc[t];                            /* scan */
                y += Cb[n * seqlen + t] * h[n];                            /* C_t h_t */
            }
            y += Dd * uc[t];                                               /* + D u_t */
            out[c * seqlen + t] = zc ? y * o_silu(zc[t]) : y;              /* gate */
        }
        if (hN)
            for (int64_t n = 0; n < dstate; n++) hN[c * dstate + n] = h[n];
    }
    free(h);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Selective scan, backward: the reverse-mode derivative of oracle_scan_fwd
 * with respect to every input, for the loss  sum(dout * out) + sum(dhN * hN).
 * The pages state that the backward recomputes h instead of storing it; they
 * print no formulas, so these are derived from the forward above by the chain
 * rule.  Here h_t is simply recomputed by a forward sweep per channel and kept
 * (seqlen x dstate doubles), then a reverse sweep accumulates the adjoint
 *   G_t[n] = dy_t C_t[n] + Abar_{t+1}[n] G_{t+1}[n].
 *
 * Outputs (caller-zeroed accumulators marked "+="):
 *   du, ddt, dz  : (batch, dim, seqlen)           written for the channel range
 *   dA           : (dim, dstate)          +=
 *   dBm, dCm     : (batch, dstate, seqlen) +=      (summed over channels d)
 *   dDskip, dbias: (dim)                   +=
 *   dh0          : (batch, dim, dstate)           written, may be NULL
 * dz may be NULL when z is NULL; dhN may be NULL (zero). */
int oracle_scan_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t dstate,
                    const double* u, const double* dt, const double* z,
                    const double* A, const double* Bm, const double* Cm,
                    const double* Dskip, const double* bias,
                    const double* h0, int zoh, int delta_softplus,
                    const double* dout, const double* dhN,
                    double* du, double* ddt, double* dz, double* dA,
                    double* dBm, double* dCm, double* dDskip, double* dbias,
                    double* dh0, int64_t ch_begin, int64_t ch_end)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || dstate < 1) return -1;
    if (ch_begin < 0 || ch_end > batch * dim || ch_begin > ch_end) return -1;
    const size_t LN = (size_t)(seqlen + 1) * (size_t)dstate;
    double* H = (double*)malloc(sizeof(double) * LN);          /* H[(t+1)*N+n] = h_t, H[n] = h_{-1} */
    double* G = (double*)malloc(sizeof(double) * (size_t)dstate);
    double* delta = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    double* y = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    if (!H || !G || !delta || !y) { free(H); free(G); free(delta); free(y); return -1; }
    for (int64_t c = ch_begin; c < ch_end; c++) {
        const int64_t b = c / dim, d = c % dim;
        const double* uc = u + c * seqlen;
        const double* dtc = dt + c * seqlen;
        const double* zc = z ? z + c * seqlen : NULL;
        const double* Bb = Bm + b * dstate * seqlen;
        const double* Cb = Cm + b * dstate * seqlen;
        double* dBb = dBm + b * dstate * seqlen;
        double* dCb = dCm + b * dstate * seqlen;
        const double* Ad = A + d * dstate;
        const double Dd = Dskip ? Dskip[d] : 0.0;
        const double bd = bias ? bias[d] : 0.0;

        /* forward sweep: recompute delta_t, h_t and the pre-gate y_t */
        for (int64_t n = 0; n < dstate; n++) H[n] = h0 ? h0[c * dstate + n] : 0.0;
        for (int64_t t = 0; t < seqlen; t++) {
            const double v = dtc[t] + bd;
            delta[t] = delta_softplus ? o_softplus(v) : v;
            double yt = 0.0;
            for (int64_t n = 0; n < dstate; n++) {
                const double a = exp(delta[t] * Ad[n]);
                const double bbar = o_bbar_coef(delta[t], Ad[n], zoh) * Bb[n * seqlen + t];
                H[(t + 1) * dstate + n] = a * H[t * dstate + n] + bbar * uc[t];
                yt += Cb[n * seqlen + t] * H[(t + 1) * dstate + n];
            }
            y[t] = yt + Dd * uc[t];
        }

        /* reverse sweep */
        for (int64_t n = 0; n < dstate; n++) G[n] = dhN ? dhN[c * dstate + n] : 0.0;
        double dD_acc = 0.0, dbias_acc = 0.0;
        for (int64_t t = seqlen - 1; t >= 0; t--) {
            double dy;
            if (zc) {
                const double s = o_sigmoid(zc[t]);
                dy = dout[c * seqlen + t] * zc[t] * s;
                dz[c * seqlen + t] = dout[c * seqlen + t] * y[t] * s * (1.0 + zc[t] * (1.0 - s));
            } else {
                dy = dout[c * seqlen + t];
            }
            double du_t = dy * Dd;
            double ddelta = 0.0;
            dD_acc += dy * uc[t];
            for (int64_t n = 0; n < dstate; n++) {
                const double hprev = H[t * dstate + n];
                const double hcur = H[(t + 1) * dstate + n];
                const double a = exp(delta[t] * Ad[n]);
                const double coef = o_bbar_coef(delta[t], Ad[n], zoh);
                const double Bv = Bb[n * seqlen + t];
                /* G_t = dy_t C_t + (Abar_{t+1} G_{t+1}, already in G) */
                G[n] += dy * Cb[n * seqlen + t];
                dCb[n * seqlen + t] += dy * hcur;
                const double da = G[n] * hprev;          /* d loss / d Abar_t   */
                const double dbb = G[n] * uc[t];         /* d loss / d Bbar_t   */
                du_t += G[n] * coef * Bv;
                dBb[n * seqlen + t] += dbb * coef;
                const double dcoef = dbb * Bv;           /* d loss / d coef     */
                /* Abar = e^{delta A}: dAbar/ddelta = A Abar, dAbar/dA = delta Abar */
                ddelta += da * Ad[n] * a;
                dA[d * dstate + n] += da * delta[t] * a;
                if (zoh) {
                    /* coef = (e^{delta A}-1)/A: dcoef/ddelta = e^{delta A},
                       dcoef/dA = delta^2 phi(delta A)  (limit delta^2/2 at A=0) */
                    ddelta += dcoef * a;
                    dA[d * dstate + n] += dcoef * delta[t] * delta[t] * o_phi(delta[t] * Ad[n]);
                } else {
                    ddelta += dcoef;                     /* coef = delta */
                }
                G[n] *= a;                               /* becomes Abar_t G_t for step t-1 */
            }
            du[c * seqlen + t] = du_t;
            const double v = dtc[t] + bd;
            const double dv = delta_softplus ? ddelta * o_sigmoid(v) : ddelta;
            ddt[c * seqlen + t] = dv;
            dbias_acc += dv;
        }
        if (dh0)
            for (int64_t n = 0; n < dstate; n++) dh0[c * dstate + n] = G[n];
        if (dDskip) dDskip[d] += dD_acc;
        if (dbias) dbias[d] += dbias_acc;
    }
    free(H); free(G); free(delta); free(y);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Single-token decode step: state <- update(state, x_t), then the readout and
 * gate for that token.  [P1] section "为什么 Mamba 推理更省" and the scan,
 * readout and gate nodes for one t.
 *   x, dt, z, out : (batch, dim)       (x is the scan input u_t; z may be NULL)
 *   Bm, Cm        : (batch, dstate)
 *   state         : (batch, dim, dstate), read and overwritten */
int oracle_state_update(int64_t batch, int64_t dim, int64_t dstate,
                        const double* x, const double* dt, const double* z,
                        const double* A, const double* Bm, const double* Cm,
                        const double* Dskip, const double* bias,
                        int zoh, int delta_softplus, double* state, double* out)
{
    if (batch < 0 || dim < 0 || dstate < 1) return -1;
    for (int64_t b = 0; b < batch; b++) {
        for (int64_t d = 0; d < dim; d++) {
            const int64_t c = b * dim + d;
            const double v = dt[c] + (bias ? bias[d] : 0.0);
            const double delta = delta_softplus ? o_softplus(v) : v;
            double y = 0.0;
            for (int64_t n = 0; n < dstate; n++) {
                const double Adn = A[d * dstate + n];
                const double a = exp(delta * Adn);
                const double bbar = o_bbar_coef(delta, Adn, zoh) * Bm[b * dstate + n];
                double* hs = &state[c * dstate + n];
                *hs = a * (*hs) + bbar * x[c];
                y += Cm[b * dstate + n] * (*hs);
            }
            y += (Dskip ? Dskip[d] : 0.0) * x[c];
            out[c] = z ? y * o_silu(z[c]) : y;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Causal depthwise conv1d (width W) + SiLU over a sequence.
 * [P1] conv node Uc_t = sum_i W_i U_{t-i} (tap i = 0 is the current token)
 * and SiLU node; [P3] section 03: the short conv keeps the last 4 inputs.
 *   x, out      : (batch, dim, seqlen)
 *   w           : (dim, width), w[d, i] multiplies x[t - i]
 *   bias        : (dim) or NULL
 *   state_in    : (batch, dim, width) or NULL: the `width` inputs that came
 *                 before t = 0, oldest first (x[-width] .. x[-1]); NULL = zeros
 *   state_out   : (batch, dim, width) or NULL: the last `width` inputs seen,
 *                 oldest first (x[seqlen-width] .. x[seqlen-1], reaching into
 *                 state_in when seqlen < width) */
int oracle_conv1d_silu(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                       const double* x, const double* w, const double* bias,
                       const double* state_in, double* out, double* state_out)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1) return -1;
    for (int64_t c = 0; c < batch * dim; c++) {
        const int64_t d = c % dim;
        const double* xc = x + c * seqlen;
        /* x at a (possibly negative) time index */
#define XAT(tt) ((tt) >= 0 ? xc[(tt)] : (state_in ? state_in[c * width + width + (tt)] : 0.0))
        for (int64_t t = 0; t < seqlen; t++) {
            double acc = bias ? bias[d] : 0.0;
            for (int64_t i = 0; i < width; i++) {
                const int64_t tt = t - i;
                if (tt < -width) continue;
                acc += w[d * width + i] * XAT(tt);
            }
            out[c * seqlen + t] = o_silu(acc);
        }
        if (state_out) {
            for (int64_t k = 0; k < width; k++) {
                const int64_t tt = seqlen - width + k;
                state_out[c * width + k] = (tt >= -width) ? XAT(tt) : 0.0;
            }
        }
#undef XAT
    }
    return 0;
}

/* Backward of oracle_conv1d_silu for the loss sum(dout * out): the chain rule
 * of the conv node and the SiLU node of [P1], one channel and one step at a
 * time.  With pre_t = bias + sum_i w_i x_(t-i) and out_t = silu(pre_t):
 *   dpre_t       = dout_t * silu'(pre_t),  silu'(p) = s (1 + p (1 - s)), s = sigmoid(p)
 *   dx_s         = sum_i w_i dpre_(s+i)                  (s + i < seqlen)
 *   dw[d, i]     = sum over b, t of dpre_t x_(t-i)       (x before t = 0 from state_in)
 *   dbias[d]     = sum over b, t of dpre_t
 *   dstate_in[k] = sum_i w_i dpre_(k-width+i)            (0 <= k-width+i < seqlen)
 *   dout, dx : (batch, dim, seqlen); dw (dim, width); dbias (dim) or NULL;
 *   dstate_in (batch, dim, width) or NULL */
int oracle_conv1d_silu_bwd(int64_t batch, int64_t dim, int64_t seqlen, int64_t width,
                           const double* x, const double* w, const double* bias,
                           const double* state_in, const double* dout,
                           double* dx, double* dw, double* dbias, double* dstate_in)
{
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1) return -1;
    double* dpre = (double*)malloc((size_t)(seqlen > 0 ? seqlen : 1) * sizeof(double));
    if (!dpre) return -2;
    for (int64_t i = 0; i < dim * width; i++) dw[i] = 0.0;
    if (dbias) for (int64_t d = 0; d < dim; d++) dbias[d] = 0.0;
    for (int64_t c = 0; c < batch * dim; c++) {
        const int64_t d = c % dim;
        const double* xc = x + c * seqlen;
#define XAT(tt) ((tt) >= 0 ? xc[(tt)] : (state_in ? state_in[c * width + width + (tt)] : 0.0))
        for (int64_t t = 0; t < seqlen; t++) {
            double pre = bias ? bias[d] : 0.0;
            for (int64_t i = 0; i < width; i++) {
                const int64_t tt = t - i;
                if (tt < -width) continue;
                pre += w[d * width + i] * XAT(tt);
            }
            const double s = o_sigmoid(pre);
            dpre[t] = dout[c * seqlen + t] * s * (1.0 + pre * (1.0 - s));
        }
        for (int64_t t = 0; t < seqlen; t++) {
            if (dbias) dbias[d] += dpre[t];
            for (int64_t i = 0; i < width; i++) {
                const int64_t tt = t - i;
                if (tt < -width) continue;
                dw[d * width + i] += dpre[t] * XAT(tt);
            }
        }
        for (int64_t s = 0; s < seqlen; s++) {
            double g = 0.0;
            for (int64_t i = 0; i < width; i++)
                if (s + i < seqlen) g += w[d * width + i] * dpre[s + i];
            dx[c * seqlen + s] = g;
        }
        if (dstate_in) {
            for (int64_t k = 0; k < width; k++) {
                double g = 0.0;
                for (int64_t i = 0; i < width; i++) {
                    const int64_t t = k - width + i;
                    if (t >= 0 && t < seqlen) g += w[d * width + i] * dpre[t];
                }
                dstate_in[c * width + k] = g;
            }
        }
#undef XAT
    }
    free(dpre);
    return 0;
}

/* One-token conv update: shift x_t into the stored window, then the conv and
 * SiLU for that token.  [P1] conv node for one t; [P3] section 03.
 *   state : (batch, dim, width), oldest first, read and overwritten
 *   x,out : (batch, dim) */
int oracle_conv1d_silu_update(int64_t batch, int64_t dim, int64_t width,
                              const double* x, const double* w, const double* bias,
                              double* state, double* out)
{
    if (batch < 0 || dim < 0 || width < 1) return -1;
    for (int64_t c = 0; c < batch * dim; c++) {
        const int64_t d = c % dim;
        double* s = state + c * width;
        for (int64_t k = 0; k + 1 < width; k++) s[k] = s[k + 1];
        s[width - 1] = x[c];
        double acc = bias ? bias[d] : 0.0;
        for (int64_t i = 0; i < width; i++) acc += w[d * width + i] * s[width - 1 - i];
        out[c] = o_silu(acc);
    }
    return 0;
}

/*
 * Mamba-2 state-space-duality layer, computed as its recurrence.
 *
 * [P3] "Mamba 与状态空间模型", section "09 Mamba-2：两种算法": A is one number
 * times the identity (per head), and the layer is the product with a lower
 * triangular matrix whose (i, j) entry is C at step i times B at step j times
 * the whole decay between the two steps; the recurrence is one of the two
 * algorithms that evaluate it.  [P4] pnsm.cn overview, section "Mamba-2：状态
 * 空间对偶性": scalar transition, blocks inside / recurrence between.  The
 * input enters scaled by the step size (Bbar = Delta B, the simplified rule of
 * [P3] "模型省略了什么"), so per (b, head h), with state H (N x P):
 *
 *   Delta_t = softplus(dt[b,t,h] + dt_bias[h])   (or dt + dt_bias)
 *   H       = exp(Delta_t A[h]) H + Delta_t B_t x_t^T
 *   y_t     = C_t^T H + D[h] x_t
 *
 * Layouts: x, out (batch, L, H, P); dt (batch, L, H); B, C (batch, L, G, N)
 * with head h reading group h / (H / G); h0, hN (batch, H, N, P).  Units
 * [u_begin, u_end) index (b, h) pairs.
 */
int oracle_ssd_fwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                   int64_t ngroups, const double* x, const double* dt, const double* A,
                   const double* Bm, const double* Cm, const double* Dskip, const double* dt_bias,
                   const double* h0, int delta_softplus, double* out, double* hN,
                   int64_t u_begin, int64_t u_end)
{
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1) return -1;
    if (nheads % ngroups != 0) return -1;
    if (u_begin < 0 || u_end > batch * nheads || u_begin > u_end) return -1;
    const int64_t P = headdim, N = dstate, H = nheads, G = ngroups;
    double* S = (double*)malloc(sizeof(double) * (size_t)(N * P));
    if (!S) return -1;
    for (int64_t unit = u_begin; unit < u_end; unit++) {
        const int64_t b = unit / H, h = unit % H, g = h / (H / G);
        for (int64_t i = 0; i < N * P; i++) S[i] = h0 ? h0[unit * N * P + i] : 0.0;
        for (int64_t t = 0; t < seqlen; t++) {
            const double v = dt[(b * seqlen + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);
            const double delta = delta_softplus ? o_softplus(v) : v;
            const double a = exp(delta * A[h]);
            const double* Bt = Bm + ((b * seqlen + t) * G + g) * N;
            const double* Ct = Cm + ((b * seqlen + t) * G + g) * N;
            const double* xt = x + ((b * seqlen + t) * H + h) * P;
            double* yt = out + ((b * seqlen + t) * H + h) * P;
            for (int64_t n = 0; n < N; n++)
                for (int64_t p = 0; p < P; p++)
                    S[n * P + p] = a * S[n * P + p] + delta * Bt[n] * xt[p];
            for (int64_t p = 0; p < P; p++) {
                double y = 0.0;
                for (int64_t n = 0; n < N; n++) y += Ct[n] * S[n * P + p];
                yt[p] = y + (Dskip ? Dskip[h] : 0.0) * xt[p];
            }
        }
        if (hN)
            for (int64_t i = 0; i < N * P; i++) hN[unit * N * P + i] = S[i];
    }
    free(S);
    return 0;
}

/*
 * Mamba-2 SSD layer, reverse mode: the gradients of
 *   loss = sum(dout * out) + sum(dhN * hN)
 * for the recurrence of oracle_ssd_fwd ("Mamba 与状态空间模型" section 09;
 * pnsm.cn overview, section "Mamba-2：状态空间对偶性"), by the adjoint of that
 * recurrence walked backwards one step at a time.  Per (b, head h) the states
 * H_0 .. H_L (H_t = the state after step t, H_0 = h0) are kept; then, from
 * t = L - 1 down to 0, with G the adjoint of the state (starting at dhN):
 *
 *   y_t = C_t^T H_(t+1) + D x_t         ->  dC_t += H_(t+1) dy_t,  dD += x_t . dy_t,
 *                                           dx_t  = D dy_t,        G += C_t dy_t^T
 *   H_(t+1) = a_t H_t + Delta_t B_t x_t^T, a_t = exp(Delta_t A)
 *                                       ->  dx_t += Delta_t G^T B_t,
 *                                           dB_t += Delta_t G x_t,
 *                                           dDelta_t = <G, A a_t H_t + B_t x_t^T>,
 *                                           dA += <G, Delta_t a_t H_t>,
 *                                           G <- a_t G
 *   Delta_t = softplus(v), v = dt + dt_bias  ->  ddt_t = dDelta_t sigmoid(v)
 *                                           (= dDelta_t without softplus),
 *                                           ddt_bias += ddt_t
 *
 * and dh0 = G at the end.  dx, ddt, dh0 are written for the units in
 * [u_begin, u_end); dA, dD, ddt_bias (H) and dB, dC (batch, L, G, N) are ADDED
 * to (so that threads working on disjoint units can keep partial sums).
 */
int oracle_ssd_bwd(int64_t batch, int64_t seqlen, int64_t nheads, int64_t headdim, int64_t dstate,
                   int64_t ngroups, const double* x, const double* dt, const double* A,
                   const double* Bm, const double* Cm, const double* Dskip, const double* dt_bias,
                   const double* h0, int delta_softplus, const double* dout, const double* dhN,
                   double* dx, double* ddt, double* dA, double* dB, double* dC, double* dD,
                   double* ddt_bias, double* dh0, int64_t u_begin, int64_t u_end)
{
    if (batch < 0 || seqlen < 0 || nheads < 1 || headdim < 1 || dstate < 1 || ngroups < 1) return -1;
    if (nheads % ngroups != 0) return -1;
    if (u_begin < 0 || u_end > batch * nheads || u_begin > u_end) return -1;
    const int64_t P = headdim, N = dstate, H = nheads, G = ngroups, NP = dstate * headdim;
    double* Hs = (double*)malloc(sizeof(double) * (size_t)((seqlen + 1) * NP));
    double* Gs = (double*)malloc(sizeof(double) * (size_t)NP);
    double* delta = (double*)malloc(sizeof(double) * (size_t)(seqlen > 0 ? seqlen : 1));
    if (!Hs || !Gs || !delta) {
        free(Hs); free(Gs); free(delta);
        return -1;
    }
    for (int64_t unit = u_begin; unit < u_end; unit++) {
        const int64_t b = unit / H, h = unit % H, g = h / (H / G);
        const double Dh = Dskip ? Dskip[h] : 0.0;
        /* forward: every state of the sequence */
        for (int64_t i = 0; i < NP; i++) Hs[i] = h0 ? h0[unit * NP + i] : 0.0;
        for (int64_t t = 0; t < seqlen; t++) {
            const double v = dt[(b * seqlen + t) * H + h] + (dt_bias ? dt_bias[h] : 0.0);
            delta[t] = delta_softplus ? o_softplus(v) : v;
            const double a = exp(delta[t] * A[h]);
            const double* Bt = Bm + ((b * seqlen + t) * G + g) * N;
            const double* xt = x + ((b * seqlen + t) * H + h) * P;
            const double* Hp = Hs + t * NP;
            double* Hn = Hs + (t + 1) * NP;
            for (int64_t n = 0; n < N; n++)
                for (int64_t p = 0; p < P; p++)
                    Hn[n * P + p] = a * Hp[n * P + p] + delta[t] * Bt[n] * xt[p];
        }
        /* reverse */
        for (int64_t i = 0; i < NP; i++) Gs[i] = dhN ? dhN[unit * NP + i] : 0.0;
        for (int64_t t = seqlen - 1; t >= 0; t--) {
            const int64_t row = (b * seqlen + t) * H + h;
            const double v = dt[row] + (dt_bias ? dt_bias[h] : 0.0);
            const double a = exp(delta[t] * A[h]);
            const double* Bt = Bm + ((b * seqlen + t) * G + g) * N;
            const double* Ct = Cm + ((b * seqlen + t) * G + g) * N;
            double* dBt = dB + ((b * seqlen + t) * G + g) * N;
            double* dCt = dC + ((b * seqlen + t) * G + g) * N;
            const double* xt = x + row * P;
            const double* dyt = dout + row * P;
            double* dxt = dx + row * P;
            const double* Hp = Hs + t * NP;
            const double* Hn = Hs + (t + 1) * NP;
            /* readout */
            for (int64_t n = 0; n < N; n++) {
                double acc = 0.0;
                for (int64_t p = 0; p < P; p++) acc += Hn[n * P + p] * dyt[p];
                dCt[n] += acc;
            }
            for (int64_t p = 0; p < P; p++) {
                dD[h] += xt[p] * dyt[p];
                dxt[p] = Dh * dyt[p];
            }
            for (int64_t n = 0; n < N; n++)
                for (int64_t p = 0; p < P; p++) Gs[n * P + p] += Ct[n] * dyt[p];
            /* state update */
            for (int64_t p = 0; p < P; p++) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; n++) acc += Gs[n * P + p] * Bt[n];
                dxt[p] += delta[t] * acc;
            }
            for (int64_t n = 0; n < N; n++) {
                double acc = 0.0;
                for (int64_t p = 0; p < P; p++) acc += Gs[n * P + p] * xt[p];
                dBt[n] += delta[t] * acc;
            }
            double dd = 0.0, da = 0.0;
            for (int64_t n = 0; n < N; n++)
                for (int64_t p = 0; p < P; p++) {
                    dd += Gs[n * P + p] * (A[h] * a * Hp[n * P + p] + Bt[n] * xt[p]);
                    da += Gs[n * P + p] * delta[t] * a * Hp[n * P + p];
                }
            dA[h] += da;
            for (int64_t i = 0; i < NP; i++) Gs[i] *= a;
            const double dv = delta_softplus ? dd * o_sigmoid(v) : dd;
            ddt[row] = dv;
            ddt_bias[h] += dv;
        }
        for (int64_t i = 0; i < NP; i++) dh0[unit * NP + i] = Gs[i];
    }
    free(Hs);
    free(Gs);
    free(delta);
    return 0;
}
