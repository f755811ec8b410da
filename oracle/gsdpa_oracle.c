/*
 * gsdpa_oracle.c -- float64 CPU oracle for the G1 gated attention layer.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain definition of what the
 * layer computes, written out in double precision with no tiling, fusion or
 * reordering. Only the test suite, the smoke check and the benchmark's CPU
 * baseline leg may load it. The GPU library never links or calls it, and it
 * shares no code with the GPU library.
 *
 * What it computes, for every batch b, query head h and query row i
 * (sources, by page title and section):
 *
 *   a      = L_k - L_q + i         absolute position of query i; the causal
 *                                  mask is aligned bottom-right so that one
 *                                  decode query sees the whole cache (the
 *                                  pages are silent for L_q < L_k; this is
 *                                  the reading taken).
 *   kv(h)  = h / (H_q / H_kv)      contiguous query-head groups share one
 *                                  K/V head ("GatedAttention [2025]",
 *                                  sec. 1.3.1, the GQA description: h query
 *                                  heads in g groups).
 *   s_j    = <Q[b,i,h,:], K[b,j,kv(h),:]> / sqrt(d_k)
 *                                  for j <= a when causal, all j otherwise
 *                                  ("GatedAttention [2025]", sec. 1.2.1, the
 *                                  SDPA equation; sec. 1.4.1, the per-head
 *                                  output sums over j = 0..i).
 *   p_j    = exp(s_j - max s) / sum_j exp(s_j - max s)
 *                                  (row-stochastic softmax, sec. 1.2.1).
 *   y_c    = sum_j p_j V[b,j,kv(h),c]
 *   gl     = sum_m X[b,i,m] W_g[m, h*d_k + c]   elementwise gate, n x q x d_k
 *          = sum_m X[b,i,m] W_g[m, h]           headwise gate,    n x q
 *                                  ("GatedAttention [2025]", sec. 1.2.2, the
 *                                  gating equation Y' = Y (.) sigma(X W);
 *                                  "10 . 门控", sec. 3.2, the G1 module: no
 *                                  bias, head-major gate columns, one scalar
 *                                  per head when headwise).
 *   O[b,i,h,c] = y_c * 1/(1 + exp(-gl))         (gate NONE: O = y)
 *
 * Gate variants (gsdpa_oracle_fwd_variant; "GatedAttention [2025]", sec.
 * 1.2.2 items (3)-(5), sec. 1.4.1 and sec. 1.4.2):
 *   shapes: head-shared elementwise, W_g [d_model, d_k], gl = sum_m X W_g[m, c];
 *           head-shared headwise, W_g [d_model, 1], gl = sum_m X W_g[m, 0]
 *           (W_theta and the scores shared by every head, item (3b));
 *           input-independent, theta [H_q, d_k] in place of W_g, gl = theta[h, c]
 *           (a free parameter per head and column, sec. 1.4.2 (iii)).
 *   functions of gl and the combination with y:
 *           sigmoid, multiplied        O = y * s(gl),             s(x) = 1/(1+e^-x)
 *           NS-sigmoid, multiplied     O = y * (0.5 + 0.5 s(gl))  (sec. 1.4.2 (iv))
 *           sigmoid, added             O = y + s(gl)              (item (4b))
 *           SiLU, added                O = y + gl s(gl)           (item (5); sec. 1.4.1)
 *           identity, added            O = y + gl                 (sec. 1.4.1 (ii))
 *   shapes averaged over the heads ("GatedAttention [2025]", sec. 1.3.2 (ii):
 *           the n x q x d_k scores averaged over the q query heads into one
 *           n x d_k score every head uses): headwise averaged, W_g [d_model,
 *           H_q]; elementwise averaged, W_g [d_model, H_q*d_k]; the value is
 *           vbar = (1/H_q) sum_h' v(gl_h') with v the function below (its
 *           value part), combined with y as the function says.
 *   without W_g:
 *           SiLU of the output         O = y * s(y)               (sec. 1.4.1 (i))
 *           per-head RMSNorm           O = y / sqrt(mean_c y_c^2 + eps) * gamma[h, c]
 *                                      (sec. 1.4.1, the norm applied to each
 *                                      head's output before concatenation;
 *                                      gamma given in place of W_g, or 1)
 *   p0[b,i,h]  = p_0, the attention weight on key 0 ("10 . 门控", sec. 3.4,
 *                the share of attention that lands on the first token).
 *   lse[b,i,h] = max s + log sum_j exp(s_j - max s), the log of the softmax
 *                denominator (natural log), which a backward pass needs to
 *                rebuild p without the forward's running statistics.
 *
 * The backward pass (gsdpa_oracle_bwd) is the chain rule of the same
 * definition, given dO = dL/dO, written out term by term:
 *   dy_c   = dO_c g_c                          (g = 1 without a gate)
 *   dgl_c  = dO_c y_c g_c (1 - g_c)            elementwise; headwise: the sum
 *                                              over c of the same product
 *            ("解密NeurIPS最佳论文：Gated Attention…", sec. 2.2: the loss's
 *            gradient on the gate is the upstream gradient times the ungated
 *            context, and on the gate's input that times sigma (1 - sigma))
 *   dW_g[m, col] += X[b,i,m] dgl_col,   dX[b,i,m] += sum_col dgl_col W_g[m, col]
 *                                              (the gate path's share of dX)
 *   dV[b,j,kv(h),c] += p_j dy_c
 *   dp_j   = sum_c dy_c V[b,j,kv(h),c]
 *   ds_j   = p_j (dp_j - sum_k p_k dp_k)       (softmax Jacobian)
 *   dQ[b,i,h,:]     += sum_j ds_j K[b,j,kv(h),:] / sqrt(d_k)
 *   dK[b,j,kv(h),:] += ds_j Q[b,i,h,:] / sqrt(d_k)
 *
 * Precision: every input arrives as double (the exact upcast of the fp32 or
 * bf16 values the GPU sees); nothing is rounded.
 *
 * Rows: the caller passes either all rows (n_rows < 0) or a list of (b, i)
 * pairs; each listed row is computed exactly as above. Sampling rows changes
 * nothing in the arithmetic of a row.
 */
#include <math.h>
#include <stdlib.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_GATE_NONE = 0, ORACLE_GATE_HEADWISE = 1, ORACLE_GATE_ELEMENTWISE = 2,
       ORACLE_GATE_HEADWISE_SHARED = 3, ORACLE_GATE_ELEMENTWISE_SHARED = 4, ORACLE_GATE_STATIC = 5,
       ORACLE_GATE_HEADWISE_AVERAGED = 6, ORACLE_GATE_ELEMENTWISE_AVERAGED = 7 };
enum { ORACLE_FN_SIGMOID_MUL = 0, ORACLE_FN_NS_SIGMOID_MUL = 1, ORACLE_FN_SIGMOID_ADD = 2,
       ORACLE_FN_SILU_ADD = 3, ORACLE_FN_IDENTITY_ADD = 4, ORACLE_FN_SILU_SELF = 5, ORACLE_FN_RMSNORM = 6 };

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* columns of W_g for a gate shape (0: no W_g read from X) */
static long gate_width(int gate_mode, int Hq, int dk)
{
    switch (gate_mode) {
    case ORACLE_GATE_HEADWISE: case ORACLE_GATE_HEADWISE_AVERAGED: return Hq;
    case ORACLE_GATE_ELEMENTWISE: case ORACLE_GATE_ELEMENTWISE_AVERAGED: return (long)Hq * dk;
    case ORACLE_GATE_HEADWISE_SHARED: return 1;
    case ORACLE_GATE_ELEMENTWISE_SHARED: return dk;
    default: return 0;
    }
}

/* gate logit of head h, column c of row x */
static double gate_logit(const double* x, const double* Wg, int gate_mode, int d_model, int Hq, int dk, int h, int c)
{
    if (gate_mode == ORACLE_GATE_STATIC) return Wg[(long)h * dk + c];
    long col;
    switch (gate_mode) {
    case ORACLE_GATE_HEADWISE: case ORACLE_GATE_HEADWISE_AVERAGED: col = h; break;
    case ORACLE_GATE_ELEMENTWISE: case ORACLE_GATE_ELEMENTWISE_AVERAGED: col = (long)h * dk + c; break;
    case ORACLE_GATE_HEADWISE_SHARED: col = 0; break;
    default: col = c; break;   /* elementwise, shared by the heads */
    }
    const long G = gate_width(gate_mode, Hq, dk);
    double gl = 0.0;
    for (int m = 0; m < d_model; ++m) gl += x[m] * Wg[(long)m * G + col];
    return gl;
}

/* the gate's value from its logit (the function part of gate_apply) */
static double gate_value_of(double gl, int gate_fn)
{
    switch (gate_fn) {
    case ORACLE_FN_NS_SIGMOID_MUL: return 0.5 + 0.5 * sigmoid(gl);
    case ORACLE_FN_SILU_ADD: return gl * sigmoid(gl);
    case ORACLE_FN_IDENTITY_ADD: return gl;
    default: return sigmoid(gl);   /* sigmoid, multiplied or added */
    }
}

/* the gated output from y and a gate value: added for the additive functions, else multiplied */
static double gate_combine_value(double y, double v, int gate_fn)
{
    return (gate_fn == ORACLE_FN_SIGMOID_ADD || gate_fn == ORACLE_FN_SILU_ADD || gate_fn == ORACLE_FN_IDENTITY_ADD)
               ? y + v : y * v;
}

/* the gated output from y and the gate logit */
static double gate_apply(double y, double gl, int gate_fn)
{
    switch (gate_fn) {
    case ORACLE_FN_NS_SIGMOID_MUL: return y * (0.5 + 0.5 * sigmoid(gl));
    case ORACLE_FN_SIGMOID_ADD: return y + sigmoid(gl);
    case ORACLE_FN_SILU_ADD: return y + gl * sigmoid(gl);
    case ORACLE_FN_IDENTITY_ADD: return y + gl;
    default: return y * sigmoid(gl);
    }
}

/* One query row (b, i), all heads. s is scratch of length >= L_k. */
static void oracle_row(const double* X, const double* Q, const double* K, const double* V,
                       const double* Wg, double* O_row, double* p0_row, double* lse_row, double* s,
                       int b, int i, int Lq, int Lk, int d_model, int Hq, int Hkv, int dk,
                       int gate_mode, int gate_fn, double eps, int causal)
{
    const int group = Hq / Hkv;
    const long a = (long)Lk - Lq + i;
    const long n_keys = causal ? a + 1 : Lk;
    const double inv_sqrt_dk = 1.0 / sqrt((double)dk);
    const double* x = X ? X + ((long)b * Lq + i) * d_model : 0;

    for (int h = 0; h < Hq; ++h) {
        const int kvh = h / group;
        const double* q = Q + (((long)b * Lq + i) * Hq + h) * dk;

        /* scores */
        double mx = -INFINITY;
        for (long j = 0; j < n_keys; ++j) {
            const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
            double dot = 0.0;
            for (int c = 0; c < dk; ++c) dot += q[c] * k[c];
            s[j] = dot * inv_sqrt_dk;
            if (s[j] > mx) mx = s[j];
        }
        /* softmax */
        double denom = 0.0;
        for (long j = 0; j < n_keys; ++j) {
            s[j] = exp(s[j] - mx);
            denom += s[j];
        }
        for (long j = 0; j < n_keys; ++j) s[j] /= denom;
        if (p0_row) p0_row[h] = s[0];
        if (lse_row) lse_row[h] = mx + log(denom);

        double* o = O_row + (long)h * dk;
        for (int c = 0; c < dk; ++c) {
            double y = 0.0;
            for (long j = 0; j < n_keys; ++j)
                y += s[j] * V[(((long)b * Lk + j) * Hkv + kvh) * dk + c];
            o[c] = y;
        }
        if (gate_mode == ORACLE_GATE_HEADWISE_AVERAGED || gate_mode == ORACLE_GATE_ELEMENTWISE_AVERAGED) {
            /* every head's gate value of its own logit, averaged over the heads */
            for (int c = 0; c < dk; ++c) {
                double vbar = 0.0;
                for (int hh = 0; hh < Hq; ++hh)
                    vbar += gate_value_of(gate_logit(x, Wg, gate_mode, d_model, Hq, dk, hh, c), gate_fn);
                o[c] = gate_combine_value(o[c], vbar / Hq, gate_fn);
            }
        } else if (gate_mode != ORACLE_GATE_NONE) {
            for (int c = 0; c < dk; ++c)
                o[c] = gate_apply(o[c], gate_logit(x, Wg, gate_mode, d_model, Hq, dk, h, c), gate_fn);
        } else if (gate_fn == ORACLE_FN_SILU_SELF) {
            for (int c = 0; c < dk; ++c) o[c] = o[c] * sigmoid(o[c]);
        } else if (gate_fn == ORACLE_FN_RMSNORM) {
            double ss = 0.0;
            for (int c = 0; c < dk; ++c) ss += o[c] * o[c];
            const double r = 1.0 / sqrt(ss / dk + eps);
            for (int c = 0; c < dk; ++c) o[c] = o[c] * r * (Wg ? Wg[(long)h * dk + c] : 1.0);
        }
    }
}

/*
 * Returns 0 on success, -1 on a shape the definition does not cover.
 *   O    : [B, L_q, H_q, d_k] when n_rows < 0, else [n_rows, H_q, d_k]
 *   p0   : [B, L_q, H_q]      when n_rows < 0, else [n_rows, H_q]   (nullable)
 *   lse  : same shape as p0 (nullable)
 *   rows_b, rows_i : the (b, i) pairs when n_rows >= 0
 *   n_threads : OpenMP threads (<= 0: library default)
 */
int gsdpa_oracle_fwd_variant(const double* X, const double* Q, const double* K, const double* V,
                             const double* Wg, double* O, double* p0, double* lse,
                             int B, int Lq, int Lk, int d_model, int Hq, int Hkv, int dk,
                             int gate_mode, int gate_fn, double eps, int causal,
                             const int* rows_b, const int* rows_i, long n_rows, int n_threads)
{
    if (B < 1 || Lq < 1 || Lk < 1 || dk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return -1;
    if (Lq > Lk) return -1;
    if (gate_mode < ORACLE_GATE_NONE || gate_mode > ORACLE_GATE_ELEMENTWISE_AVERAGED) return -1;
    if (gate_fn < ORACLE_FN_SIGMOID_MUL || gate_fn > ORACLE_FN_RMSNORM) return -1;
    /* the functions of the output alone take no gate; the gates take one of the five functions of gl */
    if (gate_mode == ORACLE_GATE_NONE && gate_fn != ORACLE_FN_SIGMOID_MUL && gate_fn < ORACLE_FN_SILU_SELF) return -1;
    if (gate_mode != ORACLE_GATE_NONE && gate_fn >= ORACLE_FN_SILU_SELF) return -1;
    if (gate_mode == ORACLE_GATE_STATIC && !Wg) return -1;
    if (gate_width(gate_mode, Hq, dk) > 0 && (d_model < 1 || !X || !Wg)) return -1;
    if (gate_fn == ORACLE_FN_RMSNORM && !(eps >= 0.0)) return -1;

    const long total = (n_rows < 0) ? (long)B * Lq : n_rows;
    for (long r = 0; n_rows >= 0 && r < n_rows; ++r)
        if (rows_b[r] < 0 || rows_b[r] >= B || rows_i[r] < 0 || rows_i[r] >= Lq) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < total; ++r) {
            if (!s) continue;
            int b, i;
            if (n_rows < 0) { b = (int)(r / Lq); i = (int)(r % Lq); }
            else            { b = rows_b[r];     i = rows_i[r]; }
            oracle_row(X, Q, K, V, Wg, O + r * (long)Hq * dk, p0 ? p0 + r * (long)Hq : 0,
                       lse ? lse + r * (long)Hq : 0, s,
                       b, i, Lq, Lk, d_model, Hq, Hkv, dk, gate_mode, gate_fn, eps, causal);
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/*
 * The softmax statistics of every query row and head, without the values or
 * the gate: p0[b,i,h] = p_0 (the attention weight on key 0, "10 . 门控",
 * sec. 3.4, the first-token share) and lse[b,i,h] = max s + log sum_j
 * exp(s_j - max s), from the scores s_j of the header's definition (the SDPA
 * equation of "GatedAttention [2025]", sec. 1.2.1, causal sum over j <= a).
 * The same arithmetic as the scores and softmax of gsdpa_oracle_fwd, for
 * problems where the full layer would cost twice as much (no P V products).
 *   p0, lse : [B, L_q, H_q] (either may be null)
 * Returns 0, or -1 on a shape the definition does not cover.
 */
int gsdpa_oracle_softmax_stats(const double* Q, const double* K, double* p0, double* lse,
                               int B, int Lq, int Lk, int Hq, int Hkv, int dk, int causal, int n_threads)
{
    if (B < 1 || Lq < 1 || Lk < 1 || dk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return -1;
    if (Lq > Lk) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    const int group = Hq / Hkv;
    const double inv_sqrt_dk = 1.0 / sqrt((double)dk);
    const long total = (long)B * Lq * Hq;
    int failed = 0;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)Lk);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < total; ++r) {
            if (!s) continue;
            const int h = (int)(r % Hq);
            const int i = (int)((r / Hq) % Lq);
            const int b = (int)(r / ((long)Hq * Lq));
            const int kvh = h / group;
            const long a = (long)Lk - Lq + i;
            const long n_keys = causal ? a + 1 : Lk;
            const double* q = Q + (((long)b * Lq + i) * Hq + h) * dk;
            double mx = -INFINITY;
            for (long j = 0; j < n_keys; ++j) {
                const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
                double dot = 0.0;
                for (int c = 0; c < dk; ++c) dot += q[c] * k[c];
                s[j] = dot * inv_sqrt_dk;
                if (s[j] > mx) mx = s[j];
            }
            double denom = 0.0;
            for (long j = 0; j < n_keys; ++j) denom += exp(s[j] - mx);
            if (p0) p0[r] = exp(s[0] - mx) / denom;
            if (lse) lse[r] = mx + log(denom);
        }
        free(s);
    }
    return failed ? -1 : 0;
}

/* The layer with the default gate function (sigmoid, multiplied). */
int gsdpa_oracle_fwd(const double* X, const double* Q, const double* K, const double* V,
                     const double* Wg, double* O, double* p0, double* lse,
                     int B, int Lq, int Lk, int d_model, int Hq, int Hkv, int dk,
                     int gate_mode, int causal,
                     const int* rows_b, const int* rows_i, long n_rows, int n_threads)
{
    if (gate_mode < ORACLE_GATE_NONE || gate_mode > ORACLE_GATE_ELEMENTWISE) return -1;
    return gsdpa_oracle_fwd_variant(X, Q, K, V, Wg, O, p0, lse, B, Lq, Lk, d_model, Hq, Hkv, dk, gate_mode,
                                    ORACLE_FN_SIGMOID_MUL, 0.0, causal, rows_b, rows_i, n_rows, n_threads);
}

/*
 * Backward of the layer (the chain rule in the header), serial: dK, dV and
 * dW_g gather contributions from every row. Every output is overwritten.
 *   dO          : [B, L_q, H_q, d_k]
 *   dQ          : [B, L_q, H_q, d_k];  dK, dV : [B, L_k, H_kv, d_k]
 *   dX, dW_g    : the gate path's gradients, shaped like X and W_g
 *                 (ignored, and may be null, when gate_mode is NONE)
 * Returns 0, or -1 on a shape the definition does not cover.
 */
int gsdpa_oracle_bwd(const double* X, const double* Q, const double* K, const double* V,
                     const double* Wg, const double* dO,
                     double* dX, double* dQ, double* dK, double* dV, double* dWg,
                     int B, int Lq, int Lk, int d_model, int Hq, int Hkv, int dk,
                     int gate_mode, int causal)
{
    if (B < 1 || Lq < 1 || Lk < 1 || dk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0) return -1;
    if (Lq > Lk) return -1;
    if (gate_mode < 0 || gate_mode > 2) return -1;
    const int gated = gate_mode != ORACLE_GATE_NONE;
    if (gated && (d_model < 1 || !X || !Wg || !dX || !dWg)) return -1;

    const int group = Hq / Hkv;
    const double inv_sqrt_dk = 1.0 / sqrt((double)dk);
    const long gate_cols = (gate_mode == ORACLE_GATE_ELEMENTWISE) ? (long)Hq * dk : Hq;
    for (long e = 0; e < (long)B * Lq * Hq * dk; ++e) dQ[e] = 0.0;
    for (long e = 0; e < (long)B * Lk * Hkv * dk; ++e) dK[e] = dV[e] = 0.0;
    if (gated) {
        for (long e = 0; e < (long)B * Lq * d_model; ++e) dX[e] = 0.0;
        for (long e = 0; e < (long)d_model * gate_cols; ++e) dWg[e] = 0.0;
    }
    double* p = (double*)malloc(sizeof(double) * (size_t)Lk);
    double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);
    double* y = (double*)malloc(sizeof(double) * (size_t)dk);
    double* g = (double*)malloc(sizeof(double) * (size_t)dk);
    double* dy = (double*)malloc(sizeof(double) * (size_t)dk);
    if (!p || !dp || !y || !g || !dy) {
        free(p); free(dp); free(y); free(g); free(dy);
        return -1;
    }
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < Lq; ++i) {
            const long a = (long)Lk - Lq + i;
            const long n_keys = causal ? a + 1 : Lk;
            const double* x = gated ? X + ((long)b * Lq + i) * d_model : 0;
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / group;
                const double* q = Q + (((long)b * Lq + i) * Hq + h) * dk;
                const double* dout = dO + (((long)b * Lq + i) * Hq + h) * dk;
                /* forward quantities of the row: p, y, g */
                double mx = -INFINITY;
                for (long j = 0; j < n_keys; ++j) {
                    const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    double dot = 0.0;
                    for (int c = 0; c < dk; ++c) dot += q[c] * k[c];
                    p[j] = dot * inv_sqrt_dk;
                    if (p[j] > mx) mx = p[j];
                }
                double denom = 0.0;
                for (long j = 0; j < n_keys; ++j) {
                    p[j] = exp(p[j] - mx);
                    denom += p[j];
                }
                for (long j = 0; j < n_keys; ++j) p[j] /= denom;
                for (int c = 0; c < dk; ++c) {
                    double acc = 0.0;
                    for (long j = 0; j < n_keys; ++j) acc += p[j] * V[(((long)b * Lk + j) * Hkv + kvh) * dk + c];
                    y[c] = acc;
                }
                if (gate_mode == ORACLE_GATE_HEADWISE) {
                    double gl = 0.0;
                    for (int m = 0; m < d_model; ++m) gl += x[m] * Wg[(long)m * gate_cols + h];
                    const double gh = 1.0 / (1.0 + exp(-gl));
                    for (int c = 0; c < dk; ++c) g[c] = gh;
                } else if (gate_mode == ORACLE_GATE_ELEMENTWISE) {
                    for (int c = 0; c < dk; ++c) {
                        double gl = 0.0;
                        const long col = (long)h * dk + c;
                        for (int m = 0; m < d_model; ++m) gl += x[m] * Wg[(long)m * gate_cols + col];
                        g[c] = 1.0 / (1.0 + exp(-gl));
                    }
                } else {
                    for (int c = 0; c < dk; ++c) g[c] = 1.0;
                }
                /* gate path */
                for (int c = 0; c < dk; ++c) dy[c] = dout[c] * g[c];
                if (gate_mode == ORACLE_GATE_ELEMENTWISE) {
                    for (int c = 0; c < dk; ++c) {
                        const double dgl = dout[c] * y[c] * g[c] * (1.0 - g[c]);
                        const long col = (long)h * dk + c;
                        double* dx = dX + ((long)b * Lq + i) * d_model;
                        for (int m = 0; m < d_model; ++m) {
                            dWg[(long)m * gate_cols + col] += x[m] * dgl;
                            dx[m] += dgl * Wg[(long)m * gate_cols + col];
                        }
                    }
                } else if (gate_mode == ORACLE_GATE_HEADWISE) {
                    double dgl = 0.0;
                    for (int c = 0; c < dk; ++c) dgl += dout[c] * y[c] * g[c] * (1.0 - g[c]);
                    double* dx = dX + ((long)b * Lq + i) * d_model;
                    for (int m = 0; m < d_model; ++m) {
                        dWg[(long)m * gate_cols + h] += x[m] * dgl;
                        dx[m] += dgl * Wg[(long)m * gate_cols + h];
                    }
                }
                /* attention path */
                double sum_pdp = 0.0;
                for (long j = 0; j < n_keys; ++j) {
                    const double* v = V + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    double* dv = dV + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) {
                        acc += dy[c] * v[c];
                        dv[c] += p[j] * dy[c];
                    }
                    dp[j] = acc;
                    sum_pdp += p[j] * acc;
                }
                double* dq = dQ + (((long)b * Lq + i) * Hq + h) * dk;
                for (long j = 0; j < n_keys; ++j) {
                    const double ds = p[j] * (dp[j] - sum_pdp) * inv_sqrt_dk;
                    const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    double* dkk = dK + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    for (int c = 0; c < dk; ++c) {
                        dq[c] += ds * k[c];
                        dkk[c] += ds * q[c];
                    }
                }
            }
        }
    free(p); free(dp); free(y); free(g); free(dy);
    return 0;
}

/*
 * The backward's outputs on sampled rows only, for problems too large for
 * gsdpa_oracle_bwd: the same chain rule, in two passes.
 *   Pass 1, every row (b, i) and head h (parallel over rows): the row's
 *   softmax p, its log-denominator lse, the gate g, dy = dO g and
 *   Dsum = sum_j p_j dp_j (= sum_c dy_c y_c); dQ for the listed query rows
 *   and, with a gate and dX_rows non-null, their dX = dGl W_g^T (dGl = dO y
 *   sigma (1 - sigma), y = sum_j p_j V_j, summed over the head for a
 *   headwise gate).
 *   Pass 2, every listed key row (b, j) (parallel over them): for each head h
 *   of kv(j)'s group and each query i that sees j,
 *     p_ij = exp(s_ij - lse_i), dp_ij = sum_c dy_ic V_jc,
 *     ds_ij = p_ij (dp_ij - Dsum_i),
 *     dK_j += ds_ij Q_i / sqrt(d_k),   dV_j += p_ij dy_i.
 *   qb, qi [nq]: query rows;  kb, kj [nk]: key rows
 *   dQ_rows [nq, H_q, d_k];  dK_rows, dV_rows [nk, H_kv, d_k];  dX_rows [nq, d_model] or null
 * Returns 0, or -1 on a shape the definition does not cover or no memory.
 */
int gsdpa_oracle_bwd_rows(const double* X, const double* Q, const double* K, const double* V,
                          const double* Wg, const double* dO,
                          int B, int Lq, int Lk, int d_model, int Hq, int Hkv, int dk, int gate_mode, int causal,
                          const int* qb, const int* qi, long nq, const int* kb, const int* kj, long nk,
                          double* dQ_rows, double* dK_rows, double* dV_rows, double* dX_rows, int n_threads)
{
    if (B < 1 || Lq < 1 || Lk < 1 || dk < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lq > Lk) return -1;
    if (gate_mode < 0 || gate_mode > 2) return -1;
    if (gate_mode != ORACLE_GATE_NONE && (d_model < 1 || !X || !Wg)) return -1;
    for (long r = 0; r < nq; ++r)
        if (qb[r] < 0 || qb[r] >= B || qi[r] < 0 || qi[r] >= Lq) return -1;
    for (long r = 0; r < nk; ++r)
        if (kb[r] < 0 || kb[r] >= B || kj[r] < 0 || kj[r] >= Lk) return -1;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    const int group = Hq / Hkv;
    const double inv_sqrt_dk = 1.0 / sqrt((double)dk);
    const long gate_cols = (gate_mode == ORACLE_GATE_ELEMENTWISE) ? (long)Hq * dk : Hq;
    const long rows = (long)B * Lq;
    double* lse = (double*)malloc(sizeof(double) * (size_t)rows * Hq);
    double* dsum = (double*)malloc(sizeof(double) * (size_t)rows * Hq);
    double* dy_all = (double*)malloc(sizeof(double) * (size_t)rows * Hq * dk);
    /* which query rows are listed (row -> index + 1) */
    long* qidx = (long*)calloc((size_t)rows, sizeof(long));
    if (!lse || !dsum || !dy_all || !qidx) {
        free(lse); free(dsum); free(dy_all); free(qidx);
        return -1;
    }
    for (long r = 0; r < nq; ++r) qidx[(long)qb[r] * Lq + qi[r]] = r + 1;
    int failed = 0;
    /* pass 1 */
#pragma omp parallel
    {
        double* p = (double*)malloc(sizeof(double) * (size_t)Lk);
        double* dp = (double*)malloc(sizeof(double) * (size_t)Lk);
        double* y = (double*)malloc(sizeof(double) * (size_t)dk);
        double* gv = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!p || !dp || !y || !gv) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < rows; ++r) {
            if (!p || !dp || !y || !gv) continue;
            const int b = (int)(r / Lq), i = (int)(r % Lq);
            const long a = (long)Lk - Lq + i;
            const long n_keys = causal ? a + 1 : Lk;
            const double* x = gate_mode != ORACLE_GATE_NONE ? X + r * d_model : 0;
            for (int h = 0; h < Hq; ++h) {
                const int kvh = h / group;
                const double* q = Q + (r * Hq + h) * dk;
                const double* dout = dO + (r * Hq + h) * dk;
                double* dy = dy_all + (r * Hq + h) * dk;
                double mx = -INFINITY;
                for (long j = 0; j < n_keys; ++j) {
                    const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    double dot = 0.0;
                    for (int c = 0; c < dk; ++c) dot += q[c] * k[c];
                    p[j] = dot * inv_sqrt_dk;
                    if (p[j] > mx) mx = p[j];
                }
                double denom = 0.0;
                for (long j = 0; j < n_keys; ++j) {
                    p[j] = exp(p[j] - mx);
                    denom += p[j];
                }
                for (long j = 0; j < n_keys; ++j) p[j] /= denom;
                lse[r * Hq + h] = mx + log(denom);
                double g_head = 1.0;
                if (gate_mode == ORACLE_GATE_HEADWISE) {
                    double gl = 0.0;
                    for (int m = 0; m < d_model; ++m) gl += x[m] * Wg[(long)m * gate_cols + h];
                    g_head = 1.0 / (1.0 + exp(-gl));
                }
                for (int c = 0; c < dk; ++c) {
                    double g = g_head;
                    if (gate_mode == ORACLE_GATE_ELEMENTWISE) {
                        double gl = 0.0;
                        const long col = (long)h * dk + c;
                        for (int m = 0; m < d_model; ++m) gl += x[m] * Wg[(long)m * gate_cols + col];
                        g = 1.0 / (1.0 + exp(-gl));
                    }
                    gv[c] = g;
                    dy[c] = dout[c] * g;
                }
                double ds_sum = 0.0;
                for (long j = 0; j < n_keys; ++j) {
                    const double* v = V + (((long)b * Lk + j) * Hkv + kvh) * dk;
                    double acc = 0.0;
                    for (int c = 0; c < dk; ++c) acc += dy[c] * v[c];
                    dp[j] = acc;
                    ds_sum += p[j] * acc;
                }
                dsum[r * Hq + h] = ds_sum;
                const long qr = qidx[r] - 1;
                if (qr >= 0) {
                    double* dq = dQ_rows + (qr * Hq + h) * dk;
                    for (int c = 0; c < dk; ++c) dq[c] = 0.0;
                    for (long j = 0; j < n_keys; ++j) {
                        const double ds = p[j] * (dp[j] - ds_sum) * inv_sqrt_dk;
                        const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
                        for (int c = 0; c < dk; ++c) dq[c] += ds * k[c];
                    }
                    if (dX_rows && gate_mode != ORACLE_GATE_NONE) {
                        /* the gate's input gradient: dGl = dO . Y . sigma (1 - sigma) with Y = P V
                         * the ungated output (summed over the head's columns for a headwise
                         * gate), then dX = dGl W_g^T, accumulated over the heads */
                        double* dx = dX_rows + qr * d_model;
                        if (h == 0)
                            for (int m = 0; m < d_model; ++m) dx[m] = 0.0;
                        for (int c = 0; c < dk; ++c) y[c] = 0.0;
                        for (long j = 0; j < n_keys; ++j) {
                            const double* v = V + (((long)b * Lk + j) * Hkv + kvh) * dk;
                            for (int c = 0; c < dk; ++c) y[c] += p[j] * v[c];
                        }
                        if (gate_mode == ORACLE_GATE_ELEMENTWISE) {
                            for (int c = 0; c < dk; ++c) {
                                const double dgl = dout[c] * y[c] * gv[c] * (1.0 - gv[c]);
                                const long col = (long)h * dk + c;
                                for (int m = 0; m < d_model; ++m) dx[m] += dgl * Wg[(long)m * gate_cols + col];
                            }
                        } else {
                            double dgl = 0.0;
                            for (int c = 0; c < dk; ++c) dgl += dout[c] * y[c];
                            dgl *= g_head * (1.0 - g_head);
                            for (int m = 0; m < d_model; ++m) dx[m] += dgl * Wg[(long)m * gate_cols + h];
                        }
                    }
                }
            }
        }
        free(p); free(dp); free(y); free(gv);
    }
    /* pass 2 */
    if (!failed) {
#pragma omp parallel for schedule(dynamic, 1)
        for (long t = 0; t < nk; ++t) {
            const int b = kb[t], j = kj[t];
            for (int kvh = 0; kvh < Hkv; ++kvh) {
                const double* k = K + (((long)b * Lk + j) * Hkv + kvh) * dk;
                const double* v = V + (((long)b * Lk + j) * Hkv + kvh) * dk;
                double* dkr = dK_rows + (t * Hkv + kvh) * dk;
                double* dvr = dV_rows + (t * Hkv + kvh) * dk;
                for (int c = 0; c < dk; ++c) dkr[c] = dvr[c] = 0.0;
                for (int h = kvh * group; h < (kvh + 1) * group; ++h)
                    for (int i = 0; i < Lq; ++i) {
                        if (causal && (long)Lk - Lq + i < j) continue;   /* query i does not see key j */
                        const long r = (long)b * Lq + i;
                        const double* q = Q + (r * Hq + h) * dk;
                        const double* dy = dy_all + (r * Hq + h) * dk;
                        double s = 0.0, dpv = 0.0;
                        for (int c = 0; c < dk; ++c) {
                            s += q[c] * k[c];
                            dpv += dy[c] * v[c];
                        }
                        const double pij = exp(s * inv_sqrt_dk - lse[r * Hq + h]);
                        const double ds = pij * (dpv - dsum[r * Hq + h]) * inv_sqrt_dk;
                        for (int c = 0; c < dk; ++c) {
                            dkr[c] += ds * q[c];
                            dvr[c] += pij * dy[c];
                        }
                    }
            }
        }
    }
    free(lse); free(dsum); free(dy_all); free(qidx);
    return failed ? -1 : 0;
}

/*
 * The gate's scores sigma(X W_g) of every row and gate column, for the gate
 * statistics ("GatedAttention [2025]", sec. 1.4.2 (i), Table 4 and Figure 3:
 * the mean gating score and the distribution of the scores):
 *   scores[r, col] = 1 / (1 + exp(-sum_m X[r, m] W_g[m, col])),
 *   r over the B * L_q rows, col over the H_q * d_k (elementwise) or H_q
 *   (headwise) gate columns.
 * Returns 0, or -1 for another gate mode.
 */
int gsdpa_oracle_gate_scores(const double* X, const double* Wg, double* scores, long rows, int d_model, int Hq,
                             int dk, int gate_mode)
{
    if (gate_mode != ORACLE_GATE_HEADWISE && gate_mode != ORACLE_GATE_ELEMENTWISE) return -1;
    if (rows < 0 || d_model < 1 || !X || !Wg || !scores) return -1;
    const long G = gate_width(gate_mode, Hq, dk);
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r)
        for (long col = 0; col < G; ++col) {
            double gl = 0.0;
            for (int m = 0; m < d_model; ++m) gl += X[r * d_model + m] * Wg[(long)m * G + col];
            scores[r * G + col] = sigmoid(gl);
        }
    return 0;
}

/* Number of threads an OpenMP region would use (1 without OpenMP). */
int gsdpa_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
