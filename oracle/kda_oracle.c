/*
 * kda_oracle.c -- plain fp64 CPU oracle for the Kimi Delta Attention (KDA)
 * operator and its prologue.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the yardstick the CUDA library is
 * measured against; it is never part of the product path.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA sources.
 *
 * Sources (page title -- section):
 *  [B5]  "From GPT-2 to Kimi K3, from first principles" -- Chapter 5
 *        "Kimi Delta Attention: channel-wise forgetting" (the recurrence, the
 *        four verbs retain / erase / write / read, the lower-bounded decay
 *        g = gmin * sigmoid(z) with gmin = -5, where q,k,v,alpha,beta come from).
 *  [B6]  same page -- Chapter 6 "The GPU problem" (read after the update: the
 *        local causal matrix keeps its diagonal).
 *  [E3]  "Kimi K3 Architecture Explained" -- "Step 3: Forgetting, Channel by
 *        Channel" (S_t = (I - b k k^T) Diag(alpha_t) S_{t-1} + b k v^T, one row
 *        of the state per key channel) and "Inside a KDA Layer".
 *  [D1]  "An infra-oriented diagram of Kimi K3" -- "Kimi Delta Attention:
 *        fixed-state sequence mixing" (width-4 depthwise causal conv, Swish,
 *        L2Norm of q and k, scaled sigmoid, beta = sigmoid; "Head RMSNorm +
 *        gate, full-rank 7168 -> 12288 gate") and the packed-token note
 *        (cumulative sequence offsets keep document boundaries).
 *  [B5g] "From GPT-2 to Kimi K3", Chapter 5, "A third gate: control what
 *        leaves the module" (head-wise RMSNorm and sigmoid(W_g x) after the
 *        recurrent read).
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *  - query scale 1: o_t = S_t^T q_t exactly as written;
 *  - alpha = exp(g) (natural log);
 *  - conv: no bias, zero history before each document start, tap 3 is the
 *    current token (y_t = sum_j w_j x_{t-3+j});
 *  - L2 norm: x / sqrt(sum x^2 + eps), eps passed by the caller;
 *  - documents in a packed batch never see each other (state and conv
 *    history restart at every cu_seqlens entry);
 *  - output gate: RMSNorm over the d channels of one head and token,
 *    x / sqrt(mean x^2 + eps) * w with a per-channel weight w shared by the
 *    heads, then times sigmoid of the gate logit of the same channel.
 *
 * Every routine is written as the plain definition, element by element, in
 * double precision.  OpenMP only distributes independent (document, head)
 * units; it never reorders the arithmetic inside one unit.
 *
 * Pins: each routine is checked by the CPU test suite against closed forms,
 * special cases (DeltaNet, Gated DeltaNet, exact overwrite, decay only),
 * the explicit product of transition matrices, exact rational arithmetic and
 * library routines (scipy lfilter / expit).  No routine here is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_OK 0
#define KDA_ORACLE_BAD_ARGS 1
#define KDA_ORACLE_NO_MEMORY 2

/* cu_seqlens must start at 0, never decrease and end at T. */
static int offsets_are_valid(const int64_t *cu_seqlens, int32_t N, int64_t T)
{
    if (N < 1 || cu_seqlens == NULL || cu_seqlens[0] != 0 || cu_seqlens[N] != T)
        return 0;
    for (int32_t n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return 0;
    return 1;
}

static void set_threads(int32_t num_threads)
{
#ifdef _OPENMP
    if (num_threads > 0)
        omp_set_num_threads(num_threads);
#else
    (void)num_threads;
#endif
}

/*
 * The KDA recurrence, token by token, for every (document, head).
 *
 *   S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 *   alpha_t = exp(g_t),   o_t = S_t^T q_t                       [E3], [B5]
 *
 * carried out as the four verbs of [B5]:
 *   retain : R = Diag(alpha_t) S_{t-1}       (row i of the state is scaled
 *                                             by alpha_t[i]; rows are key
 *                                             channels [E3])
 *   erase+write : S_t = R + beta_t k_t (v_t - R^T k_t)^T
 *                 which is (I - beta k k^T) R + beta k v^T multiplied out
 *   read   : o_t = S_t^T q_t                 (after the update [B5], [B6])
 *
 * Layout (row-major, contiguous):
 *   q, k, g : [T, H, dk]   v, out : [T, H, dv]   beta : [T, H]
 *   init_state, final_state : [N, H, dk, dv]  (row = key channel)
 *   cu_seqlens : [N + 1] document offsets into the packed token axis.
 * init_state may be NULL (zero state); final_state may be NULL.
 * Zero-length documents are allowed: their final state is the initial one.
 */
int kda_oracle_recurrence(const double *q, const double *k, const double *v,
                          const double *g, const double *beta,
                          const double *init_state, const int64_t *cu_seqlens,
                          int32_t N, int64_t T, int32_t H, int32_t dk,
                          int32_t dv, double *out, double *final_state,
                          int32_t num_threads)
{
    if (H < 1 || dk < 1 || dv < 1 || T < 0 || q == NULL || k == NULL ||
        v == NULL || g == NULL || beta == NULL || (T > 0 && out == NULL))
        return KDA_ORACLE_BAD_ARGS;
    if (!offsets_are_valid(cu_seqlens, N, T))
        return KDA_ORACLE_BAD_ARGS;
    set_threads(num_threads);

    int failed = 0;
    const int64_t units = (int64_t)N * H;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t unit = 0; unit < units; ++unit) {
        const int32_t n = (int32_t)(unit / H);
        const int32_t h = (int32_t)(unit % H);
        const size_t state_len = (size_t)dk * (size_t)dv;
        double *S = (double *)malloc(state_len * sizeof(double));
        double *err = (double *)malloc((size_t)dv * sizeof(double));
        if (S == NULL || err == NULL) {
            free(S);
            free(err);
#pragma omp atomic write
            failed = 1;
            continue;
        }
        if (init_state != NULL)
            memcpy(S, init_state + (size_t)unit * state_len,
                   state_len * sizeof(double));
        else
            memset(S, 0, state_len * sizeof(double));

        for (int64_t t = cu_seqlens[n]; t < cu_seqlens[n + 1]; ++t) {
            const size_t row = (size_t)t * H + h;
            const double *qt = q + row * dk;
            const double *kt = k + row * dk;
            const double *gt = g + row * dk;
            const double *vt = v + row * dv;
            const double bt = beta[row];

            /* retain: row i of the state keeps exp(g_t[i]) of itself */
            for (int32_t i = 0; i < dk; ++i) {
                const double alpha = exp(gt[i]);
                for (int32_t j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] *= alpha;
            }
            /* erase + write: error of the retained memory along k_t */
            for (int32_t j = 0; j < dv; ++j) {
                double pred = 0.0;
                for (int32_t i = 0; i < dk; ++i)
                    pred += S[(size_t)i * dv + j] * kt[i];
                err[j] = vt[j] - pred;
            }
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] += bt * kt[i] * err[j];
            /* read the updated state with the query */
            double *ot = out + row * dv;
            for (int32_t j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int32_t i = 0; i < dk; ++i)
                    acc += S[(size_t)i * dv + j] * qt[i];
                ot[j] = acc;
            }
        }
        if (final_state != NULL)
            memcpy(final_state + (size_t)unit * state_len, S,
                   state_len * sizeof(double));
        free(S);
        free(err);
    }
    return failed ? KDA_ORACLE_NO_MEMORY : KDA_ORACLE_OK;
}

/*
 * Width-W depthwise causal convolution, one filter per channel [D1], [B5]:
 *   y[t, c] = sum_{j=0}^{W-1} w[c, j] * x[t - (W-1) + j, c]
 * with x taken as zero before the first token of t's document (the packed
 * documents of [D1] never see each other).  No bias.
 * x, y : [T, C]     w : [C, W]
 */
int kda_oracle_short_conv(const double *x, const double *w,
                          const int64_t *cu_seqlens, int32_t N, int64_t T,
                          int32_t C, int32_t W, double *y, int32_t num_threads)
{
    if (x == NULL || w == NULL || y == NULL || C < 1 || W < 1)
        return KDA_ORACLE_BAD_ARGS;
    if (!offsets_are_valid(cu_seqlens, N, T))
        return KDA_ORACLE_BAD_ARGS;
    set_threads(num_threads);
    for (int32_t n = 0; n < N; ++n) {
        const int64_t start = cu_seqlens[n];
        const int64_t end = cu_seqlens[n + 1];
#pragma omp parallel for schedule(static)
        for (int64_t t = start; t < end; ++t) {
            for (int32_t c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int32_t j = 0; j < W; ++j) {
                    const int64_t src = t - (W - 1) + j;
                    if (src >= start)
                        acc += w[(size_t)c * W + j] * x[(size_t)src * C + c];
                }
                y[(size_t)t * C + c] = acc;
            }
        }
    }
    return KDA_ORACLE_OK;
}

/* Swish (SiLU): x * sigmoid(x) = x / (1 + exp(-x)), in place [D1]. */
int kda_oracle_swish(double *x, int64_t count)
{
    if (x == NULL || count < 0)
        return KDA_ORACLE_BAD_ARGS;
    for (int64_t i = 0; i < count; ++i)
        x[i] = x[i] / (1.0 + exp(-x[i]));
    return KDA_ORACLE_OK;
}

/*
 * Per-head L2 normalisation of queries and keys, in place [D1], [B5]:
 *   x[t, h, :] <- x[t, h, :] / sqrt(sum_c x[t, h, c]^2 + eps)
 */
int kda_oracle_l2norm(double *x, int64_t rows, int32_t d, double eps)
{
    if (x == NULL || rows < 0 || d < 1 || eps < 0.0)
        return KDA_ORACLE_BAD_ARGS;
    for (int64_t r = 0; r < rows; ++r) {
        double *xr = x + (size_t)r * d;
        double ss = 0.0;
        for (int32_t c = 0; c < d; ++c)
            ss += xr[c] * xr[c];
        const double inv = 1.0 / sqrt(ss + eps);
        for (int32_t c = 0; c < d; ++c)
            xr[c] *= inv;
    }
    return KDA_ORACLE_OK;
}

/*
 * Lower-bounded channel-wise log-decay [B5], [D1]:
 *   g = gmin * sigmoid(z) = gmin / (1 + exp(-z)),  gmin = -5 in K3,
 * so g lies in (gmin, 0) and alpha = exp(g) in (exp(gmin), 1).
 */
int kda_oracle_decay_gate(const double *z, int64_t count, double gmin,
                          double *g)
{
    if (z == NULL || g == NULL || count < 0)
        return KDA_ORACLE_BAD_ARGS;
    for (int64_t i = 0; i < count; ++i)
        g[i] = gmin / (1.0 + exp(-z[i]));
    return KDA_ORACLE_OK;
}

/* Write strength beta = sigmoid(z), one value per head and token [D1], [E3]. */
int kda_oracle_sigmoid(const double *z, int64_t count, double *out)
{
    if (z == NULL || out == NULL || count < 0)
        return KDA_ORACLE_BAD_ARGS;
    for (int64_t i = 0; i < count; ++i)
        out[i] = 1.0 / (1.0 + exp(-z[i]));
    return KDA_ORACLE_OK;
}

/*
 * Head-wise RMSNorm and the full-rank output gate [B5g], [D1], [E3] ("The
 * result is normalised, multiplied element-wise by an output gate"):
 *   y[r, c] = o[r, c] / sqrt(mean_c' o[r, c']^2 + eps) * w[c] * sigmoid(z[r, c])
 * o, z, y : [rows, d] (one row per token and head);  w : [d] or NULL (ones).
 */
int kda_oracle_output_gate(const double *o, const double *z, const double *w,
                           int64_t rows, int32_t d, double eps, double *y)
{
    if (o == NULL || z == NULL || y == NULL || rows < 0 || d < 1 || eps < 0.0)
        return KDA_ORACLE_BAD_ARGS;
    for (int64_t r = 0; r < rows; ++r) {
        const double *orow = o + (size_t)r * d;
        double ss = 0.0;
        for (int32_t c = 0; c < d; ++c)
            ss += orow[c] * orow[c];
        const double inv_rms = 1.0 / sqrt(ss / d + eps);
        for (int32_t c = 0; c < d; ++c) {
            const double gate = 1.0 / (1.0 + exp(-z[(size_t)r * d + c]));
            y[(size_t)r * d + c] = orow[c] * inv_rms * (w ? w[c] : 1.0) * gate;
        }
    }
    return KDA_ORACLE_OK;
}
