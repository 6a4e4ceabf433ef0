/*
 * Gated DeltaNet (GDN) linear-attention layer core -- CPU oracle, float64.
 *
 * TEST INFRASTRUCTURE.  This file is the slow, plain statement of what the
 * layer core computes.  Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline leg load it; the library's compute path never does,
 * and this file shares no code, header or table with the CUDA kernels.
 *
 * Source of the definitions (cited per function below):
 *   [cortex]  commit "feat(stage-8c): linear-attention layer (Qwen3-Next
 *             GatedDeltaNet)" of the cortex project -- sections "Block",
 *             "Discretisation", "Delta rule (recurrent, per-token)", "Output",
 *             "State (GatedDeltaNetState)", and its unit-test list.
 *   [nxdi-173] NxD-Inference PR "Add Qwen3.6-27B hybrid DeltaNet/GQA contrib
 *             model and vLLM serving path" -- Summary (recurrent and
 *             convolution state checkpoints for hybrid prefix caching).
 *
 * Readings where the pages leave a step open (each is also listed in the
 * design notes): conv state keeps the K-1 newest raw inputs, column 0 oldest;
 * no conv bias; tap w[c][K-1] multiplies the current token; SiLU on every conv
 * channel; channels are [q | k | v], heads contiguous; v-head h reads k-head
 * h / (H_v/H_k) (repeat_interleave); l2norm and RMSNormGated both use eps
 * inside the square root; softplus switches to the identity above 20; the
 * read-out uses the state after the token's own update.
 *
 * All arithmetic is in double.  Nothing is blocked, fused or reordered: each
 * function loops over tokens in order exactly as the recurrence is stated.
 * Independent (sequence, head) or channel units may run on separate threads;
 * that changes no operation inside a unit.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int pick_threads(int nthreads) {
#ifdef _OPENMP
    return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

int oracle_max_threads(void) { return pick_threads(0); }

static double silu(double x) { return x / (1.0 + exp(-x)); }

/* softplus with the two branches of the [cortex] unit test "softplus
 * small/large branches": identity above 20, log1p(exp(x)) otherwise. */
static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

/* ------------------------------------------------------------------------ */
/* [cortex] "Block": depthwise causal Conv1d (k=4) with state-aware prepend,
 * then SiLU.  [cortex] "State": conv_state is the left-padded tail of raw
 * inputs.  [nxdi-173] Summary: convolution state checkpoints.
 *
 * For sequence i (tokens cu[i] .. cu[i+1]-1, local position p) the extended
 * input is  xt(p) = x[cu[i]+p]            for p >= 0
 *                   state_in[i][c][K-1+p] for -(K-1) <= p < 0  (0 if NULL)
 * and y[p][c] = sum_{j=0}^{K-1} w[c][j] * xt(p-(K-1)+j), then y <- silu(y).
 * state_out[i][c][j] = xt(L-(K-1)+j); checkpoint m (m*N <= L) holds
 * xt(m*N-(K-1)+j).  Checkpoint rows are numbered over sequences in order.
 *
 * x [T][C], w [C][K], state_in/state_out [n_seq][C][K-1], y [T][C],
 * ckpt_out [n_ckpt][C][K-1].  state_out must not alias state_in here.
 */
static double conv_xt(const double* x, const double* st, int64_t t0, int64_t C, int64_t K,
                      int64_t i, int64_t p, int64_t c) {
    if (p >= 0) return x[(t0 + p) * C + c];
    if (!st) return 0.0;
    return st[(i * C + c) * (K - 1) + (K - 1) + p];
}

void oracle_conv1d(const double* x, const double* w, const int64_t* cu, int64_t n_seq,
                   int64_t C, int64_t K, const double* state_in, int apply_silu, double* y,
                   double* state_out, int64_t ckpt_every, double* ckpt_out, int nthreads) {
    int nt = pick_threads(nthreads);
    (void)nt;
    for (int64_t i = 0; i < n_seq; ++i) {
        const int64_t t0 = cu[i], L = cu[i + 1] - cu[i];
        int64_t ck0 = 0;
        if (ckpt_every > 0)
            for (int64_t j = 0; j < i; ++j) ck0 += (cu[j + 1] - cu[j]) / ckpt_every;
#pragma omp parallel for num_threads(nt) schedule(static)
        for (int64_t c = 0; c < C; ++c) {
            for (int64_t p = 0; p < L; ++p) {
                double acc = 0.0;
                for (int64_t j = 0; j < K; ++j)
                    acc += w[c * K + j] * conv_xt(x, state_in, t0, C, K, i, p - (K - 1) + j, c);
                y[(t0 + p) * C + c] = apply_silu ? silu(acc) : acc;
            }
            if (state_out)
                for (int64_t j = 0; j < K - 1; ++j)
                    state_out[(i * C + c) * (K - 1) + j] =
                        conv_xt(x, state_in, t0, C, K, i, L - (K - 1) + j, c);
            if (ckpt_every > 0 && ckpt_out)
                for (int64_t m = 1; m * ckpt_every <= L; ++m)
                    for (int64_t j = 0; j < K - 1; ++j)
                        ckpt_out[((ck0 + m - 1) * C + c) * (K - 1) + j] =
                            conv_xt(x, state_in, t0, C, K, i, m * ckpt_every - (K - 1) + j, c);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* [cortex] "Discretisation": g = -exp(A_log) * softplus(a + dt_bias),
 * beta = sigmoid(b).   a, b, g, beta [T][H]; A_log, dt_bias [H]. */
void oracle_gates(const double* a, const double* b, const double* A_log, const double* dt_bias,
                  int64_t T, int64_t H, double* g, double* beta) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            g[t * H + h] = -exp(A_log[h]) * softplus(a[t * H + h] + dt_bias[h]);
            beta[t * H + h] = 1.0 / (1.0 + exp(-b[t * H + h]));
        }
}

/* [cortex] "Block": L2norm on q,k; unit test "l2norm hand-calc + zero-vector
 * stability".  x <- x / sqrt(sum x^2 + eps), in place, per row of length d. */
void oracle_l2norm(double* x, int64_t rows, int64_t d, double eps) {
    for (int64_t r = 0; r < rows; ++r) {
        double ss = 0.0;
        for (int64_t i = 0; i < d; ++i) ss += x[r * d + i] * x[r * d + i];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int64_t i = 0; i < d; ++i) x[r * d + i] *= inv;
    }
}

/* ------------------------------------------------------------------------ */
/* [cortex] "Delta rule (recurrent, per-token)", per (sequence, v-head), tokens
 * in order, with k-head kh = h / (H_v / H_k) ([cortex] unit test
 * "repeat_interleave round-trip"):
 *     state *= exp(g_t)
 *     kv_mem = state^T k_t
 *     delta  = (v_t - kv_mem) * beta_t
 *     state += outer(k_t, delta)
 *     out_t  = state^T q_t
 * q_t and k_t are first l2-normalised (when l2norm_qk) and q_t is multiplied
 * by `scale`.  The state starts from S0 (or zeros: [cortex] "State" -- cleared
 * at the start of every new request).  Checkpoint m of a sequence is the state
 * after its first m*ckpt_every tokens ([nxdi-173] Summary: recurrent state
 * checkpoints); rows are numbered over sequences in order.
 *
 * q, k [T][H_k][d_k]; v [T][H_v][d_v]; g, beta [T][H_v];
 * S0, S_final [n_seq][H_v][d_k][d_v]; o [T][H_v][d_v];
 * ckpt [n_ckpt][H_v][d_k][d_v].
 */
void oracle_delta_rule(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const int64_t* cu, int64_t n_seq, int64_t H_k,
                       int64_t H_v, int64_t d_k, int64_t d_v, const double* S0, double scale,
                       int l2norm_qk, double eps, double* o, double* S_final, int64_t ckpt_every,
                       double* ckpt, int nthreads) {
    const int64_t r = H_v / H_k;
    const int64_t units = n_seq * H_v;
    int nt = pick_threads(nthreads);
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        const int64_t i = u / H_v, h = u % H_v, kh = h / r;
        const int64_t t0 = cu[i], L = cu[i + 1] - cu[i];
        int64_t ck0 = 0;
        if (ckpt_every > 0)
            for (int64_t j = 0; j < i; ++j) ck0 += (cu[j + 1] - cu[j]) / ckpt_every;

        double* S = (double*)malloc(sizeof(double) * d_k * d_v);
        double* qv = (double*)malloc(sizeof(double) * d_k);
        double* kv = (double*)malloc(sizeof(double) * d_k);
        double* mem = (double*)malloc(sizeof(double) * d_v);
        double* dl = (double*)malloc(sizeof(double) * d_v);
        if (S0)
            memcpy(S, S0 + (i * H_v + h) * d_k * d_v, sizeof(double) * d_k * d_v);
        else
            memset(S, 0, sizeof(double) * d_k * d_v);

        for (int64_t p = 0; p < L; ++p) {
            const int64_t t = t0 + p;
            memcpy(qv, q + (t * H_k + kh) * d_k, sizeof(double) * d_k);
            memcpy(kv, k + (t * H_k + kh) * d_k, sizeof(double) * d_k);
            if (l2norm_qk) {
                oracle_l2norm(qv, 1, d_k, eps);
                oracle_l2norm(kv, 1, d_k, eps);
            }
            for (int64_t a = 0; a < d_k; ++a) qv[a] *= scale;

            const double decay = exp(g[t * H_v + h]);
            for (int64_t e = 0; e < d_k * d_v; ++e) S[e] *= decay;
            for (int64_t j = 0; j < d_v; ++j) {
                double acc = 0.0;
                for (int64_t a = 0; a < d_k; ++a) acc += S[a * d_v + j] * kv[a];
                mem[j] = acc;
            }
            const double bt = beta[t * H_v + h];
            const double* vt = v + (t * H_v + h) * d_v;
            for (int64_t j = 0; j < d_v; ++j) dl[j] = (vt[j] - mem[j]) * bt;
            for (int64_t a = 0; a < d_k; ++a)
                for (int64_t j = 0; j < d_v; ++j) S[a * d_v + j] += kv[a] * dl[j];
            double* ot = o + (t * H_v + h) * d_v;
            for (int64_t j = 0; j < d_v; ++j) {
                double acc = 0.0;
                for (int64_t a = 0; a < d_k; ++a) acc += S[a * d_v + j] * qv[a];
                ot[j] = acc;
            }
            if (ckpt_every > 0 && ckpt && (p + 1) % ckpt_every == 0)
                memcpy(ckpt + ((ck0 + (p + 1) / ckpt_every - 1) * H_v + h) * d_k * d_v, S,
                       sizeof(double) * d_k * d_v);
        }
        if (S_final) memcpy(S_final + (i * H_v + h) * d_k * d_v, S, sizeof(double) * d_k * d_v);
        free(S); free(qv); free(kv); free(mem); free(dl);
    }
}

/* ------------------------------------------------------------------------ */
/* [cortex] "Output": RMSNormGated(core_attn_out, z): per (token, v-head),
 *   out[j] = w[j] * o[j] / sqrt(mean_j o[j]^2 + eps) * silu(z[j]).
 * o [T][H][d]; z, out [T][H*d]; w [d] shared by all heads. */
void oracle_rmsnorm_gated(const double* o, const double* z, const double* w, double eps,
                          int64_t T, int64_t H, int64_t d, double* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t h = 0; h < H; ++h) {
            const double* ov = o + (t * H + h) * d;
            double ms = 0.0;
            for (int64_t j = 0; j < d; ++j) ms += ov[j] * ov[j];
            ms /= (double)d;
            const double rs = 1.0 / sqrt(ms + eps);
            for (int64_t j = 0; j < d; ++j)
                out[(t * H + h) * d + j] = w[j] * (ov[j] * rs) * silu(z[(t * H + h) * d + j]);
        }
}
