/*
 * fp64 CPU oracle for the selective state-space (S6) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously-correct definition that
 * the CUDA path is checked against. It shares no code, header or table with the CUDA
 * library, and only the test suite, the smoke check and the benchmark's CPU-baseline
 * leg may load it. The product path never calls it.
 *
 * What it computes, and where the definition comes from:
 *   - "Mamba and State Space Models" (world.lapla.si), section "A State of Fixed Size":
 *     each input updates the state once, h <- Abar*h + Bbar*x, and the output is read
 *     from the updated state, y = C*h.
 *   - same page, section "Chosen by the Token": Delta, B and C are computed per token,
 *     A is fixed, and the retained fraction of the state is exp(Delta*A).
 *   - same page, section "A Scan on the Chip": Delta, A, B, C are discretised and then
 *     run through the recurrence (the discretisation rule of B is not stated there).
 *   - The remaining choices are the plain reading used throughout this project:
 *     Delta = softplus(delta + delta_bias) (or delta + delta_bias with the flag off),
 *     Euler discretisation of B (Bbar*x = Delta*B*u; zero-order hold as an option, which
 *     makes the one-number gate of "Chosen by the Token" exact), a skip term D*u added to C*h,
 *     and the result gated by silu(z) = z*sigmoid(z). The initial state is zero unless
 *     one is given.
 * Everything is evaluated in double precision, strictly sequentially in t, with the
 * readout summed in increasing n. Rows (b, d) are independent and are spread over
 * OpenMP threads; nothing inside a row is reordered.
 *
 * Layouts (all contiguous, row-major):
 *   u, delta, z, out      (batch, dim, seqlen)
 *   B, C                  (batch, dstate, seqlen)
 *   A                     (dim, dstate)
 *   D, delta_bias         (dim)
 *   initial_state, final_state, state   (batch, dim, dstate)
 *   state-update per-token tensors: x, dt, z, out (batch, dim); B, C (batch, dstate)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* softplus(x) = log(1 + e^x), written in the form that neither overflows nor loses
 * the small result for very negative x. */
static double softplus(double x) { return fmax(x, 0.0) + log1p(exp(-fabs(x))); }

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z). */
static double silu(double z) { return z / (1.0 + exp(-z)); }

/* Factor f with Bbar*x = f * B * x for one state with decay rate a. Euler (the default):
 * f = Delta. Zero-order hold of the continuous system h' = a h + B x over a step of length
 * Delta (option, zoh != 0): f = (exp(Delta*a) - 1) / a, which tends to Delta as a -> 0. */
static double bbar_factor(double dlt, double a, int zoh) {
    if (!zoh || a == 0.0) return dlt;
    return expm1(dlt * a) / a;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* One row (b, d) of the scan: the recurrence over t = 0 .. seqlen-1. */
static void scan_row(const double* u, const double* delta, const double* A_d, const double* Bb,
                     const double* Cb, double D_d, const double* z, double bias, int softplus_on,
                     int zoh, int64_t dstate, int64_t seqlen, double* h, double* out) {
    for (int64_t t = 0; t < seqlen; ++t) {
        double x = delta[t] + bias;
        double dlt = softplus_on ? softplus(x) : x;
        for (int64_t n = 0; n < dstate; ++n) {
            double abar = exp(dlt * A_d[n]);
            double bbar_x = bbar_factor(dlt, A_d[n], zoh) * Bb[n * seqlen + t] * u[t];
            h[n] = abar * h[n] + bbar_x;
        }
        double y = 0.0;
        for (int64_t n = 0; n < dstate; ++n) y += Cb[n * seqlen + t] * h[n];
        y += D_d * u[t];
        if (z) y *= silu(z[t]);
        out[t] = y;
    }
}

/* Full forward scan. Optional pointers (D, z, delta_bias, initial_state, final_state) may
 * be NULL: D and delta_bias then count as zero, z as no gate, initial_state as zeros. */
void oracle_scan_fwd(const double* u, const double* delta, const double* A, const double* B,
                     const double* C, const double* D, const double* z, const double* delta_bias,
                     int delta_softplus, int zoh, const double* initial_state, double* out,
                     double* final_state, int64_t batch, int64_t dim, int64_t dstate,
                     int64_t seqlen) {
    int64_t rows = batch * dim;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t b = r / dim, d = r % dim;
        double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
        for (int64_t n = 0; n < dstate; ++n)
            h[n] = initial_state ? initial_state[r * dstate + n] : 0.0;
        const int64_t off = r * seqlen;
        scan_row(u + off, delta + off, A + d * dstate, B + b * dstate * seqlen,
                 C + b * dstate * seqlen, D ? D[d] : 0.0, z ? z + off : NULL,
                 delta_bias ? delta_bias[d] : 0.0, delta_softplus, zoh, dstate, seqlen, h,
                 out + off);
        if (final_state)
            for (int64_t n = 0; n < dstate; ++n) final_state[r * dstate + n] = h[n];
        free(h);
    }
}

/* Scan over a subset of rows: rows[i] = b*dim + d. Outputs are packed per listed row:
 * out (nrows, seqlen), final_state (nrows, dstate). Inputs keep their full layouts. */
void oracle_scan_fwd_rows(const double* u_rows, const double* delta_rows, const double* A,
                          const double* B, const double* C, const double* D, const double* z_rows,
                          const double* delta_bias, int delta_softplus, int zoh,
                          const double* initial_state_rows, double* out_rows,
                          double* final_state_rows, const int64_t* rows, int64_t nrows,
                          int64_t dim, int64_t dstate, int64_t seqlen) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < nrows; ++i) {
        int64_t b = rows[i] / dim, d = rows[i] % dim;
        double* h = (double*)malloc(sizeof(double) * (size_t)dstate);
        for (int64_t n = 0; n < dstate; ++n)
            h[n] = initial_state_rows ? initial_state_rows[i * dstate + n] : 0.0;
        const int64_t off = i * seqlen;
        scan_row(u_rows + off, delta_rows + off, A + d * dstate, B + b * dstate * seqlen,
                 C + b * dstate * seqlen, D ? D[d] : 0.0, z_rows ? z_rows + off : NULL,
                 delta_bias ? delta_bias[d] : 0.0, delta_softplus, zoh, dstate, seqlen, h,
                 out_rows + off);
        if (final_state_rows)
            for (int64_t n = 0; n < dstate; ++n) final_state_rows[i * dstate + n] = h[n];
        free(h);
    }
}

/* One generated token ("The head reads one token and computes Delta, B and C ... That is
 * one step", section "Taken Apart"): the same update once, with the state read from and
 * written back to `state`. */
void oracle_state_update(double* state, const double* x, const double* dt, const double* A,
                         const double* B, const double* C, const double* D, const double* z,
                         const double* dt_bias, int dt_softplus, int zoh, double* out,
                         int64_t batch, int64_t dim, int64_t dstate) {
    int64_t rows = batch * dim;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t b = r / dim, d = r % dim;
        double* h = state + r * dstate;
        double xx = dt[r] + (dt_bias ? dt_bias[d] : 0.0);
        double dlt = dt_softplus ? softplus(xx) : xx;
        for (int64_t n = 0; n < dstate; ++n) {
            double abar = exp(dlt * A[d * dstate + n]);
            double f = bbar_factor(dlt, A[d * dstate + n], zoh);
            h[n] = abar * h[n] + f * B[b * dstate + n] * x[r];
        }
        double y = 0.0;
        for (int64_t n = 0; n < dstate; ++n) y += C[b * dstate + n] * h[n];
        y += (D ? D[d] : 0.0) * x[r];
        if (z) y *= silu(z[r]);
        out[r] = y;
    }
}

/* One decode step of the short causal convolution of the Mamba block ("Mamba and State Space
 * Models", section "A State of Fixed Size": each channel keeps "a short convolution that holds
 * the last 4 inputs"). conv_state (batch, dim, width) holds the last `width` inputs of each
 * channel, oldest first. The new input x enters at the end and the oldest leaves; the output is
 * the depthwise convolution over the window, u = sum_k w[d,k] * window[k] + bias[d], optionally
 * passed through silu. u: (batch, dim). */
void oracle_conv_step(double* conv_state, const double* x, const double* w, const double* bias,
                      int silu_on, double* u, int64_t batch, int64_t dim, int64_t width) {
    int64_t rows = batch * dim;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t d = r % dim;
        double* s = conv_state + r * width;
        for (int64_t k = 0; k + 1 < width; ++k) s[k] = s[k + 1];
        s[width - 1] = x[r];
        double acc = bias ? bias[d] : 0.0;
        for (int64_t k = 0; k < width; ++k) acc += w[d * width + k] * s[k];
        u[r] = silu_on ? silu(acc) : acc;
    }
}

/* Gradients of the scan (Euler discretisation) by reverse-mode differentiation of the loss
 * sum_t dout[t]*out[t] + sum_n dfinal[n]*final_state[n]. Every forward state of the row is
 * kept (this is the slow reference; the library recomputes them instead). Recurrences, per
 * row, with x_t = delta_t + bias, Delta_t = softplus(x_t) (or x_t), Abar = exp(Delta*A),
 * k = Delta*u, s_t = C_t . h_t + D u_t, out_t = s_t * silu(z_t):
 *   ds_t = dout_t * silu(z_t),       dz_t = dout_t * s_t * silu'(z_t)
 *   g_t  = ds_t * C_t + Abar_{t+1} * g_{t+1}     (g_{L-1} also receives dfinal)
 *   dAbar_t[n] = g_t[n] * h_{t-1}[n],  dk_t = sum_n g_t[n] * B_t[n]
 *   dDelta_t = sum_n dAbar_t[n] * Abar_t[n] * A[n] + dk_t * u_t,  du_t = dk_t * Delta_t + ds_t * D
 *   ddelta_t = dDelta_t * sigmoid(x_t) (softplus) or dDelta_t;  dbias += ddelta_t
 *   dA[n] += dAbar_t[n] * Abar_t[n] * Delta_t;  dD += ds_t * u_t
 *   dB_t[n] += g_t[n] * k_t;  dC_t[n] += ds_t * h_t[n];  dinitial = Abar_0 * g_0
 * dA, dB, dC, dD, dbias accumulate over rows (they are shared by channels or batches) and must
 * be zeroed by the caller; the others are written. */
void oracle_scan_bwd(const double* u, const double* delta, const double* A, const double* B,
                     const double* C, const double* D, const double* z, const double* delta_bias,
                     int delta_softplus, const double* initial_state, const double* dout,
                     const double* dfinal, double* du, double* ddelta, double* dA, double* dB,
                     double* dC, double* dD, double* dz, double* dbias, double* dinitial,
                     int64_t batch, int64_t dim, int64_t dstate, int64_t seqlen) {
    const int64_t L = seqlen, N = dstate;
    for (int64_t r = 0; r < batch * dim; ++r) {  /* sequential: shared gradients accumulate */
        const int64_t b = r / dim, d = r % dim, off = r * L;
        const double* Bb = B + b * N * L;
        const double* Cb = C + b * N * L;
        double* hs = (double*)malloc(sizeof(double) * (size_t)((L + 1) * N));  /* h_{-1} .. h_{L-1} */
        double* dl = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double* sg = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));  /* s_t */
        double* g = (double*)malloc(sizeof(double) * (size_t)N);
        const double bias = delta_bias ? delta_bias[d] : 0.0;
        const double Dd = D ? D[d] : 0.0;
        for (int64_t n = 0; n < N; ++n) hs[n] = initial_state ? initial_state[r * N + n] : 0.0;
        for (int64_t t = 0; t < L; ++t) {  /* forward, keeping every state */
            const double x = delta[off + t] + bias;
            const double dlt = delta_softplus ? softplus(x) : x;
            dl[t] = dlt;
            double s = Dd * u[off + t];
            for (int64_t n = 0; n < N; ++n) {
                const double h = exp(dlt * A[d * N + n]) * hs[t * N + n] + dlt * Bb[n * L + t] * u[off + t];
                hs[(t + 1) * N + n] = h;
                s += Cb[n * L + t] * h;
            }
            sg[t] = s;
        }
        for (int64_t n = 0; n < N; ++n) g[n] = dfinal ? dfinal[r * N + n] : 0.0;
        for (int64_t t = L - 1; t >= 0; --t) {
            const double x = delta[off + t] + bias;
            double ds = dout[off + t];
            if (z) {
                const double zz = z[off + t], sig = 1.0 / (1.0 + exp(-zz));
                dz[off + t] = dout[off + t] * sg[t] * (sig * (1.0 + zz * (1.0 - sig)));
                ds = dout[off + t] * zz * sig;
            }
            double dk = 0.0, dDelta = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const double abar = exp(dl[t] * A[d * N + n]);
                g[n] += ds * Cb[n * L + t];
                dC[b * N * L + n * L + t] += ds * hs[(t + 1) * N + n];
                dB[b * N * L + n * L + t] += g[n] * dl[t] * u[off + t];
                dk += g[n] * Bb[n * L + t];
                const double dabar = g[n] * hs[t * N + n];
                dDelta += dabar * abar * A[d * N + n];
                dA[d * N + n] += dabar * abar * dl[t];
                g[n] *= abar;  /* now Abar_t * g_t: the part that flows into h_{t-1} */
            }
            dDelta += dk * u[off + t];
            du[off + t] = dk * dl[t] + ds * Dd;
            const double dx = delta_softplus ? dDelta / (1.0 + exp(-x)) : dDelta;
            ddelta[off + t] = dx;
            if (dbias) dbias[d] += dx;
            if (dD) dD[d] += ds * u[off + t];
        }
        if (dinitial)
            for (int64_t n = 0; n < N; ++n) dinitial[r * N + n] = g[n];
        free(hs); free(dl); free(sg); free(g);
    }
}

/* ---- Mamba-2 state space duality layer (SSD) ----
 *
 * "Mamba and State Space Models" (world.lapla.si), section "Mamba-2": A is one number per head
 * times the identity, so a head's whole state (headdim x dstate numbers) decays by the same
 * factor exp(Delta_t * A_h) each token. Row by row the layer is this recurrence, per (b, h):
 *   Delta_t  = softplus(dt[b,t,h] + dt_bias[h])   (dt + dt_bias with the flag off)
 *   H_t[p,n] = exp(Delta_t A_h) H_{t-1}[p,n] + Delta_t x[b,t,h,p] B[b,t,g,n]
 *   y[b,t,h,p] = sum_n C[b,t,g,n] H_t[p,n] + D_h x[b,t,h,p],  then times silu(z[b,t,h,p])
 * with g = h / (nheads / ngroups) the group whose B and C head h reads. The page's other form,
 * one lower-triangular matrix per head (entry i, j = C_i . B_j times the decay in between), is
 * the same map; the tests check the two against each other. Evaluated in double precision,
 * sequential in t, the readout summed in increasing n; heads are spread over OpenMP threads.
 *
 * Layouts (contiguous, row-major):
 *   x, z, y          (batch, seqlen, nheads, headdim)
 *   dt               (batch, seqlen, nheads)
 *   A, D, dt_bias    (nheads)
 *   B, C             (batch, seqlen, ngroups, dstate)
 *   initial_state, final_state  (batch, nheads, headdim, dstate)
 * D, z, dt_bias, initial_state, final_state may be NULL (zero / no gate / zero / not written).
 */
void oracle_ssd_fwd(const double* x, const double* dt, const double* A, const double* B,
                    const double* C, const double* D, const double* z, const double* dt_bias,
                    int dt_softplus, const double* initial_state, double* y,
                    double* final_state, int64_t batch, int64_t seqlen, int64_t nheads,
                    int64_t headdim, int64_t ngroups, int64_t dstate) {
    const int64_t P = headdim, N = dstate, heads_per_group = nheads / ngroups;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < batch * nheads; ++bh) {
        const int64_t b = bh / nheads, h = bh % nheads, g = h / heads_per_group;
        double* H = (double*)malloc(sizeof(double) * (size_t)(P * N));
        for (int64_t i = 0; i < P * N; ++i) H[i] = initial_state ? initial_state[bh * P * N + i] : 0.0;
        for (int64_t t = 0; t < seqlen; ++t) {
            const double xr = dt[(b * seqlen + t) * nheads + h] + (dt_bias ? dt_bias[h] : 0.0);
            const double dlt = dt_softplus ? softplus(xr) : xr;
            const double decay = exp(dlt * A[h]);
            const double* xt = x + ((b * seqlen + t) * nheads + h) * P;
            const double* Bt = B + ((b * seqlen + t) * ngroups + g) * N;
            const double* Ct = C + ((b * seqlen + t) * ngroups + g) * N;
            for (int64_t p = 0; p < P; ++p) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    H[p * N + n] = decay * H[p * N + n] + dlt * xt[p] * Bt[n];
                    acc += Ct[n] * H[p * N + n];
                }
                acc += (D ? D[h] : 0.0) * xt[p];
                if (z) acc *= silu(z[((b * seqlen + t) * nheads + h) * P + p]);
                y[((b * seqlen + t) * nheads + h) * P + p] = acc;
            }
        }
        if (final_state)
            for (int64_t i = 0; i < P * N; ++i) final_state[bh * P * N + i] = H[i];
        free(H);
    }
}
