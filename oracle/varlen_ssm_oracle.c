/*
 * varlen_ssm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of what the packed Mamba-1
 * sequence-wise operators compute.  Only the test-suite, the smoke check and
 * the benchmark's CPU-baseline leg may load this file's library; the product
 * path (the CUDA library and its Python binding) never does.
 *
 * Every function walks the pack ONE SEQUENCE AT A TIME, using cu_seqlens
 * directly: a sequence s owns tokens [cu[s], cu[s+1]).  Nothing is chunked,
 * fused or reordered; the state is a plain array reset to zero at the start of
 * each sequence.  That is the definition the packed method must reproduce:
 * the article "Shanghai AI Lab: packed variable-length Mamba training"
 * (gitcode.csdn, sections "conv1d_pack 算子" and "SSM_pack算子") asks that
 * sequences in one pack do not interfere, i.e. give the same result as if
 * each sequence were run alone.
 *
 * Conventions (shared with the CUDA library only through the written
 * specification, never through code):
 *   - (T, D) tensors are row-major with the channel index fastest.
 *   - B, C are (T, N); A is (D, N); conv weight is (D, W) with w[d][W-1]
 *     multiplying the current token (PyTorch depthwise Conv1d layout).
 *   - Optional arrays may be NULL: bias, Dskip, z, dt_bias.
 *   - d_begin/d_end select a channel range so that callers can split the
 *     work across threads or sample channels; arrays are still full-size.
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_CU (-1)
#define ORACLE_ERR_ALLOC (-2)

/* softplus(x) = log(1 + e^x), written in the overflow-free form
 * max(x, 0) + log1p(e^{-|x|}). */
static double softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* SiLU(x) = x * sigmoid(x) and its derivative sigmoid(x) * (1 + x (1 - sigmoid(x))). */
static double silu(double x) { return x * sigmoid(x); }
static double silu_grad(double x) {
    double s = sigmoid(x);
    return s * (1.0 + x * (1.0 - s));
}

/* cu_seqlens must start at 0, never decrease, and end at T. */
static int check_cu(const int32_t* cu, int32_t num_seqs, int64_t T) {
    if (num_seqs < 0) return ORACLE_ERR_CU;
    if (cu[0] != 0) return ORACLE_ERR_CU;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (cu[s + 1] < cu[s]) return ORACLE_ERR_CU;
    if ((int64_t)cu[num_seqs] != T) return ORACLE_ERR_CU;
    return ORACLE_OK;
}

/* position_indices: each token's 0-based position inside its own sequence
 * (the auxiliary structure built at pack time; article section
 * "conv1d_pack 算子", figure (a)). */
int oracle_position_indices(const int32_t* cu, int32_t num_seqs, int64_t T, int32_t* pos) {
    if (check_cu(cu, num_seqs, T) != ORACLE_OK) return ORACLE_ERR_CU;
    for (int32_t s = 0; s < num_seqs; ++s)
        for (int64_t t = cu[s]; t < cu[s + 1]; ++t) pos[t] = (int32_t)(t - cu[s]);
    return ORACLE_OK;
}

/* Depthwise causal conv1d on one pack, one sequence at a time.  The taps of
 * a sequence's token never reach into the previous sequence (the early stop
 * of the article's conv1d_pack); instead, the W-1 positions before the
 * sequence's first token hold its tail values: x_init[s][d][0..W-2] (the
 * last W-1 inputs of a cut sequence's previous part), or zeros when x_init is
 * NULL, which is the plain per-sequence zero padding.  With xe the
 * sequence's inputs preceded by that tail (xe[p] for p = -(W-1) .. L-1):
 *     pre[p,d] = bias[d] + sum_{k=0}^{W-1} w[d][W-1-k] xe[p-k]
 *     u[p,d]   = apply_silu ? SiLU(pre) : pre
 * x_last (nullable, (num_seqs, D, W-1)) receives each sequence's last W-1
 * entries of xe: the tail the sequence's next part starts from.            */
static void fill_tail(double* xe, const double* x, const double* x_init, int32_t s, int64_t start,
                      int64_t L, int32_t d, int32_t D, int32_t W) {
    for (int32_t j = 0; j < W - 1; ++j)
        xe[j] = x_init ? x_init[((int64_t)s * D + d) * (W - 1) + j] : 0.0;
    for (int64_t p = 0; p < L; ++p) xe[W - 1 + p] = x[(start + p) * D + d];
}

int oracle_conv1d_fwd(const double* x, const double* w, const double* bias,
                      const int32_t* cu, int32_t num_seqs, int64_t T, int32_t D, int32_t W,
                      int32_t apply_silu, int32_t d_begin, int32_t d_end, const double* x_init,
                      double* u, double* x_last) {
    if (check_cu(cu, num_seqs, T) != ORACLE_OK) return ORACLE_ERR_CU;
    int64_t max_len = 0;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (cu[s + 1] - cu[s] > max_len) max_len = cu[s + 1] - cu[s];
    double* xe = (double*)malloc(sizeof(double) * (size_t)(W - 1 + max_len + 1));
    if (!xe) return ORACLE_ERR_ALLOC;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t start = cu[s], L = cu[s + 1] - cu[s];
        for (int32_t d = d_begin; d < d_end; ++d) {
            fill_tail(xe, x, x_init, s, start, L, d, D, W);
            for (int64_t p = 0; p < L; ++p) {
                double pre = bias ? bias[d] : 0.0;
                for (int32_t k = 0; k < W; ++k) pre += w[(int64_t)d * W + (W - 1 - k)] * xe[W - 1 + p - k];
                u[(start + p) * D + d] = apply_silu ? silu(pre) : pre;
            }
            if (x_last)
                for (int32_t j = 0; j < W - 1; ++j) x_last[((int64_t)s * D + d) * (W - 1) + j] = xe[L + j];
        }
    }
    free(xe);
    return ORACLE_OK;
}

/* Reverse-mode adjoint of oracle_conv1d_fwd, per sequence, on the same
 * extended inputs xe.  Gradients are written (not accumulated): dx over the
 * channel range, dw and dbias rows d_begin..d_end-1, and (nullable) dx_init,
 * the gradient reaching each sequence's tail values.  dx_last (nullable,
 * (num_seqs, D, W-1)) is the gradient reaching each sequence's x_last from
 * outside; it adds to the xe entries x_last was read from.  The reverse early
 * stop of the article (read the position of the token conv_width-1 places
 * later) is the same condition seen from the other end: xe[q] feeds pre[p]
 * only when p is a token of q's own sequence.                              */
int oracle_conv1d_bwd(const double* x, const double* w, const double* bias, const double* du,
                      const int32_t* cu, int32_t num_seqs, int64_t T, int32_t D, int32_t W,
                      int32_t apply_silu, int32_t d_begin, int32_t d_end, const double* x_init,
                      const double* dx_last, double* dx, double* dw, double* dbias, double* dx_init) {
    if (check_cu(cu, num_seqs, T) != ORACLE_OK) return ORACLE_ERR_CU;
    int64_t max_len = 0;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (cu[s + 1] - cu[s] > max_len) max_len = cu[s + 1] - cu[s];
    const size_t ne = (size_t)(W - 1 + max_len + 1);
    double* xe = (double*)malloc(sizeof(double) * ne);
    double* dxe = (double*)malloc(sizeof(double) * ne);
    if (!xe || !dxe) {
        free(xe); free(dxe);
        return ORACLE_ERR_ALLOC;
    }
    for (int32_t d = d_begin; d < d_end; ++d) {
        for (int32_t k = 0; k < W; ++k) dw[(int64_t)d * W + k] = 0.0;
        if (dbias) dbias[d] = 0.0;
        for (int64_t t = 0; t < T; ++t) dx[t * D + d] = 0.0;
    }
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t start = cu[s], L = cu[s + 1] - cu[s];
        for (int32_t d = d_begin; d < d_end; ++d) {
            fill_tail(xe, x, x_init, s, start, L, d, D, W);
            for (size_t i = 0; i < (size_t)(W - 1 + L); ++i) dxe[i] = 0.0;
            if (dx_last)
                for (int32_t j = 0; j < W - 1; ++j) dxe[L + j] += dx_last[((int64_t)s * D + d) * (W - 1) + j];
            for (int64_t p = 0; p < L; ++p) {
                double pre = bias ? bias[d] : 0.0;
                for (int32_t k = 0; k < W; ++k) pre += w[(int64_t)d * W + (W - 1 - k)] * xe[W - 1 + p - k];
                const double gpre = apply_silu ? du[(start + p) * D + d] * silu_grad(pre) : du[(start + p) * D + d];
                if (dbias) dbias[d] += gpre;
                for (int32_t k = 0; k < W; ++k) {
                    dw[(int64_t)d * W + (W - 1 - k)] += gpre * xe[W - 1 + p - k];
                    dxe[W - 1 + p - k] += w[(int64_t)d * W + (W - 1 - k)] * gpre;
                }
            }
            for (int64_t p = 0; p < L; ++p) dx[(start + p) * D + d] = dxe[W - 1 + p];
            if (dx_init)
                for (int32_t j = 0; j < W - 1; ++j) dx_init[((int64_t)s * D + d) * (W - 1) + j] = dxe[j];
        }
    }
    free(xe); free(dxe);
    return ORACLE_OK;
}

/* Selective scan forward, one sequence at a time (state reset at the
 * sequence start, the article's "SSM_pack" requirement):
 *     r_t   = delta_raw[t,d] + dt_bias[d]
 *     dlt_t = delta_softplus ? softplus(r_t) : r_t
 *     h_t[n] = exp(dlt_t A[d,n]) h_{t-1}[n] + dlt_t B[t,n] u[t,d],
 *              h_{start-1} = h_init[s] (or 0 when h_init is NULL)
 *     y_t   = sum_n C[t,n] h_t[n] + Dskip[d] u[t,d]
 *     out_t = z ? y_t (SiLU(z[t,d]) + gate_floor) : y_t
 * h_init (num_seqs, D, N) is the state a sequence starts from: the state a
 * cut sequence's first part ended in, so that a long sequence can be split
 * across packs and still pass its state on (the article's future work); the
 * gate floor is the positive bias on the gate of the GateFloor variant.  If
 * h_last is non-NULL it receives the state after each sequence's last token,
 * laid out (num_seqs, D, N) (h_init for an empty sequence).                  */
int oracle_scan_fwd(const double* u, const double* delta_raw, const double* A,
                    const double* B, const double* C, const double* Dskip, const double* z,
                    const double* dt_bias, int32_t delta_softplus, double gate_floor,
                    const double* h_init,
                    const int32_t* cu, int32_t num_seqs, int64_t T, int32_t D, int32_t N,
                    int32_t d_begin, int32_t d_end, double* out, double* h_last) {
    if (check_cu(cu, num_seqs, T) != ORACLE_OK) return ORACLE_ERR_CU;
    double* h = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!h) return ORACLE_ERR_ALLOC;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t start = cu[s], end = cu[s + 1];
        for (int32_t d = d_begin; d < d_end; ++d) {
            for (int32_t n = 0; n < N; ++n) h[n] = h_init ? h_init[((int64_t)s * D + d) * N + n] : 0.0;
            for (int64_t t = start; t < end; ++t) {
                const double r = delta_raw[t * D + d] + (dt_bias ? dt_bias[d] : 0.0);
                const double dlt = delta_softplus ? softplus(r) : r;
                const double ut = u[t * D + d];
                double y = 0.0;
                for (int32_t n = 0; n < N; ++n) {
                    const double a = exp(dlt * A[(int64_t)d * N + n]);
                    h[n] = a * h[n] + dlt * B[t * N + n] * ut;
                    y += C[t * N + n] * h[n];
                }
                y += (Dskip ? Dskip[d] : 0.0) * ut;
                out[t * D + d] = z ? y * (silu(z[t * D + d]) + gate_floor) : y;
            }
            if (h_last)
                for (int32_t n = 0; n < N; ++n) h_last[((int64_t)s * D + d) * N + n] = h[n];
        }
    }
    free(h);
    return ORACLE_OK;
}

/* Hand-derived reverse-mode adjoint of oracle_scan_fwd, one sequence at a
 * time.  The forward states of the sequence are kept in full, then walked
 * backwards; the state gradient starts after each sequence's last token at
 * dh_last[s] (the gradient that reaches the final state from outside, e.g.
 * from the next part of a cut sequence; zero when dh_last is NULL), which is
 * the reverse scan that resets at sequence ends.
 * Outputs are overwritten (gradients over the channel range):
 *   du, ddelta_raw, dz            (T, D) columns d_begin..d_end-1
 *   dA (D, N), dDskip, d_dt_bias  rows d_begin..d_end-1
 *   dB, dC (T, N)                 sum over the channel range only
 *   dh_init (num_seqs, D, N)      the gradient reaching each sequence's
 *                                 starting state (nullable)
 * dz, dDskip, d_dt_bias may be NULL when z, Dskip, dt_bias are NULL.      */
int oracle_scan_bwd(const double* u, const double* delta_raw, const double* A,
                    const double* B, const double* C, const double* Dskip, const double* z,
                    const double* dt_bias, int32_t delta_softplus, double gate_floor,
                    const double* h_init, const double* dh_last, const double* dout,
                    const int32_t* cu, int32_t num_seqs, int64_t T, int32_t D, int32_t N,
                    int32_t d_begin, int32_t d_end,
                    double* du, double* ddelta_raw, double* dA, double* dB, double* dC,
                    double* dDskip, double* dz, double* d_dt_bias, double* dh_init) {
    if (check_cu(cu, num_seqs, T) != ORACLE_OK) return ORACLE_ERR_CU;
    int64_t max_len = 0;
    for (int32_t s = 0; s < num_seqs; ++s)
        if (cu[s + 1] - cu[s] > max_len) max_len = cu[s + 1] - cu[s];
    const size_t nn = (size_t)(N > 0 ? N : 1);
    double* H = (double*)malloc(sizeof(double) * nn * (size_t)(max_len > 0 ? max_len : 1));
    double* Y = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double* dh = (double*)malloc(sizeof(double) * nn);
    if (!H || !Y || !dh) {
        free(H); free(Y); free(dh);
        return ORACLE_ERR_ALLOC;
    }
    for (int64_t t = 0; t < T; ++t)
        for (int32_t n = 0; n < N; ++n) { dB[t * N + n] = 0.0; dC[t * N + n] = 0.0; }
    for (int32_t d = d_begin; d < d_end; ++d) {
        for (int32_t n = 0; n < N; ++n) dA[(int64_t)d * N + n] = 0.0;
        if (dDskip) dDskip[d] = 0.0;
        if (d_dt_bias) d_dt_bias[d] = 0.0;
    }
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int64_t start = cu[s], end = cu[s + 1];
        for (int32_t d = d_begin; d < d_end; ++d) {
            const double Dd = Dskip ? Dskip[d] : 0.0;
            const double bias = dt_bias ? dt_bias[d] : 0.0;
            const int64_t sd = ((int64_t)s * D + d) * N;  /* this (sequence, channel)'s state row */
            /* forward, keeping every state */
            for (int64_t t = start; t < end; ++t) {
                const int64_t i = t - start;
                const double r = delta_raw[t * D + d] + bias;
                const double dlt = delta_softplus ? softplus(r) : r;
                const double ut = u[t * D + d];
                double y = 0.0;
                for (int32_t n = 0; n < N; ++n) {
                    const double hprev = i > 0 ? H[(size_t)(i - 1) * nn + n] : (h_init ? h_init[sd + n] : 0.0);
                    const double a = exp(dlt * A[(int64_t)d * N + n]);
                    const double hn = a * hprev + dlt * B[t * N + n] * ut;
                    H[(size_t)i * nn + n] = hn;
                    y += C[t * N + n] * hn;
                }
                Y[i] = y + Dd * ut;
            }
            /* backward */
            for (int32_t n = 0; n < N; ++n) dh[n] = dh_last ? dh_last[sd + n] : 0.0;
            for (int64_t t = end - 1; t >= start; --t) {
                const int64_t i = t - start;
                const double r = delta_raw[t * D + d] + bias;
                const double dlt = delta_softplus ? softplus(r) : r;
                const double ut = u[t * D + d];
                const double go = dout[t * D + d];
                double g = go;                      /* dL/dy_t */
                if (z) {
                    const double zt = z[t * D + d];
                    g = go * (silu(zt) + gate_floor);
                    dz[t * D + d] = go * Y[i] * silu_grad(zt);
                }
                double ddlt = 0.0, dut = 0.0;
                for (int32_t n = 0; n < N; ++n) {
                    const double An = A[(int64_t)d * N + n];
                    const double a = exp(dlt * An);
                    const double hprev = i > 0 ? H[(size_t)(i - 1) * nn + n] : (h_init ? h_init[sd + n] : 0.0);
                    dh[n] += C[t * N + n] * g;                 /* total dL/dh_t[n] */
                    dC[t * N + n] += g * H[(size_t)i * nn + n];
                    dB[t * N + n] += dh[n] * dlt * ut;
                    dut += dh[n] * dlt * B[t * N + n];
                    ddlt += dh[n] * (An * a * hprev + B[t * N + n] * ut);
                    dA[(int64_t)d * N + n] += dh[n] * dlt * a * hprev;
                    dh[n] *= a;                                 /* to h_{t-1} */
                }
                dut += Dd * g;
                if (dDskip) dDskip[d] += g * ut;
                du[t * D + d] = dut;
                const double dr = delta_softplus ? ddlt * sigmoid(r) : ddlt;
                ddelta_raw[t * D + d] = dr;
                if (d_dt_bias) d_dt_bias[d] += dr;
            }
            /* dh now holds the gradient reaching the state before the first token */
            if (dh_init)
                for (int32_t n = 0; n < N; ++n) dh_init[sd + n] = dh[n];
        }
    }
    free(H); free(Y); free(dh);
    return ORACLE_OK;
}
