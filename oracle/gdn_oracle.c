/*
 * gdn_oracle.c -- plain, slow, fp64 CPU oracle for the Gated DeltaNet layer.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The CUDA path never calls
 * it and shares no code with it.
 *
 * What it computes, token by token (no chunking, no blocking, no fusion):
 *
 *  1. causal depthwise conv1d over the [q|k|v] channels, last tap = current
 *     token, history from the stored conv state (zeros if none), then SiLU;
 *     the stored conv state is the last d_conv-1 RAW inputs.  The conv part of
 *     the per-layer state is stated in bytes in "Hybrid transformers under
 *     load: where Gated DeltaNet loses to full attention", section 4.1
 *     (49,152 B = 3 rows x 8192 channels x 2 B), which fixes its content as the
 *     previous raw inputs; the [q|k|v] channel sum is the ModelGeometry of
 *     "Chapter 6: engine start-up and memory plan", section 6.2.
 *  2. L2 normalisation of q and k per k-head: q^ = q_scale q / sqrt(sum q^2 + eps).
 *  3. gates per v-head: g = -exp(A_log) softplus(a + dt_bias), alpha = exp(g),
 *     beta = sigmoid(b).
 *  4. the gated delta rule (braintools.ru page, section 3: the state is
 *     partly erased by a gate and corrected by a delta-rule write), in the
 *     form S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
 *     o_t = S_t q_t, written as the three steps
 *         S <- alpha S;  e = v - S k;  S <- S + beta e k^T;  o = S q.
 *     v-head j reads k-head floor(j / G), G = H_v / H_k (contiguous groups).
 *  5. output: y = norm_w * o / sqrt(mean(o^2) + eps_n) * silu(z), per v-head.
 *
 * "Prefill is the decode path one token at a time" (Strata chapter 6,
 * section 6.9) is exactly how this file evaluates every mode.
 *
 * The `mutant` field plants a known mistake (mutant > 0).  It exists only so
 * the tests can show that every pin of this oracle catches such mistakes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GDN_OF_RAW_QKV 1u      /* x already holds [q|k|v]; no conv, no SiLU */
#define GDN_OF_NO_L2NORM 2u    /* q^ = q_scale q, k^ = k */
#define GDN_OF_GATES_DIRECT 4u /* a holds g = log(alpha), b holds beta */
#define GDN_OF_NO_OUTNORM 8u   /* y = o */

typedef struct {
    int32_t n_k_heads, n_v_heads, d_k, d_v, d_conv;
    int32_t mutant;
    double q_scale, l2_eps, norm_eps;
    uint32_t flags;
} gdn_oracle_geom;

static int64_t conv_channels(const gdn_oracle_geom* g) {
    return 2 * (int64_t)g->n_k_heads * g->d_k + (int64_t)g->n_v_heads * g->d_v;
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

static double softplus(double x) {
    /* log(1 + e^x), evaluated without overflow */
    return (x > 0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* raw conv input at token tau (tau < 0 reads the stored conv state) */
static double conv_input(const gdn_oracle_geom* g, int64_t C, int64_t tau, int64_t ch,
                         const double* x, const double* conv0) {
    if (tau >= 0) return x[tau * C + ch];
    if (!conv0) return 0.0;
    return conv0[(g->d_conv - 1 + tau) * C + ch];
}

/* u[t][i] = silu(sum_j w[ch][j] x_{t-(d_conv-1)+j}[ch] + b[ch]), ch = c0 + i */
void gdn_oracle_conv_silu(const gdn_oracle_geom* g, int64_t T, const double* x,
                          const double* conv0, const double* w, const double* bias,
                          int64_t c0, int64_t nc, double* u) {
    const int64_t C = conv_channels(g);
    const int K = g->d_conv;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t i = 0; i < nc; ++i) {
            const int64_t ch = c0 + i;
            double c = bias ? bias[ch] : 0.0;
            for (int j = 0; j < K; ++j) {
                int jw = (g->mutant == 5) ? (K - 1 - j) : j; /* mutant 5: taps reversed */
                c += w[ch * K + jw] * conv_input(g, C, t - (K - 1) + j, ch, x, conv0);
            }
            u[t * nc + i] = c * sigmoid(c);
        }
    }
}

/* conv_out[i][ch] = the last d_conv-1 raw inputs after T tokens */
void gdn_oracle_conv_final(const gdn_oracle_geom* g, int64_t T, const double* x,
                           const double* conv0, double* conv_out) {
    const int64_t C = conv_channels(g);
    const int K = g->d_conv;
    for (int i = 0; i < K - 1; ++i) {
        const int64_t tau = T - (K - 1) + i;
        for (int64_t ch = 0; ch < C; ++ch) {
            double v = conv_input(g, C, tau, ch, x, conv0);
            if (g->mutant == 11) v = v * sigmoid(v); /* mutant 11: stores activated values */
            conv_out[(int64_t)i * C + ch] = v;
        }
    }
}

/*
 * One sequence, one v-head j.  S [d_v][d_k] holds the initial state on entry
 * and the final state on return; y [T][d_v] receives this head's output.
 * Returns 0, or -1 on a bad argument or allocation failure.
 */
int gdn_oracle_head(const gdn_oracle_geom* g, int32_t j, int64_t T,
                    const double* x, const double* conv0,
                    const double* conv_w, const double* conv_b,
                    const double* z, const double* a, const double* b,
                    const double* A_log, const double* dt_bias, const double* norm_w,
                    double* S, double* y) {
    const int Hk = g->n_k_heads, Hv = g->n_v_heads, dk = g->d_k, dv = g->d_v;
    if (Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || j < 0 || j >= Hv || T < 0) return -1;
    const int G = Hv / Hk;
    const int h = (g->mutant == 6) ? (j % Hk) : (j / G); /* mutant 6: interleaved groups */
    const int64_t C = conv_channels(g);
    const int64_t cq = (int64_t)h * dk, ck = (int64_t)Hk * dk + (int64_t)h * dk;
    const int64_t cv = 2 * (int64_t)Hk * dk + (int64_t)j * dv;

    double* q = (double*)malloc(sizeof(double) * dk);
    double* k = (double*)malloc(sizeof(double) * dk);
    double* v = (double*)malloc(sizeof(double) * dv);
    double* e = (double*)malloc(sizeof(double) * dv);
    double* o = (double*)malloc(sizeof(double) * dv);
    if (!q || !k || !v || !e || !o) {
        free(q); free(k); free(v); free(e); free(o);
        return -1;
    }

    for (int64_t t = 0; t < T; ++t) {
        /* 1-2: conv + SiLU for the channels this head reads, then split */
        if (g->flags & GDN_OF_RAW_QKV) {
            for (int c = 0; c < dk; ++c) { q[c] = x[t * C + cq + c]; k[c] = x[t * C + ck + c]; }
            for (int i = 0; i < dv; ++i) v[i] = x[t * C + cv + i];
        } else {
            /* the conv of token t only looks back d_conv-1 tokens: evaluate it
               directly on the window (same definition as gdn_oracle_conv_silu) */
            const int K = g->d_conv;
            for (int part = 0; part < 3; ++part) {
                const int64_t c0 = part == 0 ? cq : (part == 1 ? ck : cv);
                const int n = part == 2 ? dv : dk;
                double* dst = part == 0 ? q : (part == 1 ? k : v);
                for (int i = 0; i < n; ++i) {
                    const int64_t ch = c0 + i;
                    double c = conv_b ? conv_b[ch] : 0.0;
                    for (int jj = 0; jj < K; ++jj) {
                        int jw = (g->mutant == 5) ? (K - 1 - jj) : jj;
                        c += conv_w[ch * K + jw] * conv_input(g, C, t - (K - 1) + jj, ch, x, conv0);
                    }
                    dst[i] = c * sigmoid(c);
                }
            }
        }

        /* 3: L2 normalisation */
        if (g->flags & GDN_OF_NO_L2NORM) {
            for (int c = 0; c < dk; ++c) q[c] *= g->q_scale;
        } else {
            double sq = 0.0, sk = 0.0;
            for (int c = 0; c < dk; ++c) { sq += q[c] * q[c]; sk += k[c] * k[c]; }
            const double rq = g->q_scale / sqrt(sq + g->l2_eps);
            const double rk = 1.0 / sqrt(sk + g->l2_eps);
            for (int c = 0; c < dk; ++c) { q[c] *= rq; k[c] *= rk; }
        }

        /* 4: gates */
        double gl, beta;
        if (g->flags & GDN_OF_GATES_DIRECT) {
            gl = a[t * Hv + j];
            beta = b[t * Hv + j];
        } else {
            const double dt = dt_bias ? dt_bias[j] : 0.0;
            const double sp = (g->mutant == 7) ? (a[t * Hv + j] + dt) /* mutant 7: no softplus */
                                               : softplus(a[t * Hv + j] + dt);
            gl = -exp(A_log[j]) * sp;
            beta = sigmoid(b[t * Hv + j]);
        }
        const double alpha = exp(gl);

        /* 5: gated delta rule */
        if (g->mutant == 3) { /* mutant 3: output read before the write */
            for (int i = 0; i < dv; ++i) {
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += alpha * S[(int64_t)i * dk + c] * q[c];
                o[i] = s;
            }
        }
        for (int i = 0; i < dv; ++i) {
            double* Si = S + (int64_t)i * dk;
            double sk = 0.0;
            if (g->mutant == 1) { /* mutant 1: error measured against the undecayed state */
                for (int c = 0; c < dk; ++c) sk += Si[c] * k[c];
                for (int c = 0; c < dk; ++c) Si[c] *= alpha;
            } else {
                for (int c = 0; c < dk; ++c) Si[c] *= alpha;
                for (int c = 0; c < dk; ++c) sk += Si[c] * k[c];
            }
            e[i] = v[i] - sk;
            const double sgn = (g->mutant == 2) ? -1.0 : 1.0; /* mutant 2: write sign flipped */
            for (int c = 0; c < dk; ++c) Si[c] += sgn * beta * e[i] * k[c];
            if (g->mutant != 3) {
                const double* rd = (g->mutant == 4) ? k : q; /* mutant 4: reads with k */
                double s = 0.0;
                for (int c = 0; c < dk; ++c) s += Si[c] * rd[c];
                o[i] = s;
            }
        }

        /* 6: gated RMSNorm */
        double* yt = y + t * dv;
        if (g->flags & GDN_OF_NO_OUTNORM) {
            for (int i = 0; i < dv; ++i) yt[i] = o[i];
        } else {
            double ss = 0.0;
            for (int i = 0; i < dv; ++i) ss += o[i] * o[i];
            const double ms = (g->mutant == 8) ? ss : ss / dv; /* mutant 8: sum, not mean */
            const double r = 1.0 / sqrt(ms + g->norm_eps);
            for (int i = 0; i < dv; ++i) {
                const double zz = z[t * (int64_t)Hv * dv + (int64_t)j * dv + i];
                const double gate = (g->mutant == 9) ? zz : zz * sigmoid(zz); /* mutant 9 */
                yt[i] = norm_w[i] * o[i] * r * gate;
            }
        }
    }
    free(q); free(k); free(v); free(e); free(o);
    return 0;
}
