/*
 * kda_oracle.c -- plain FP64 CPU oracle for the KDA (Kimi Delta Attention) mixer step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library, its Python binding)
 * may link, load or call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the CUDA path.
 *
 * Sources (web pages; cited by title and section):
 *   [NVFP4-K3]  "vsabavat/TensorRT-LLM pull request 1: NVFP4 Kimi K3 targets", Description:
 *               "KDA fuses the f_b projection, convolution, FP32 recurrence and gated output
 *               normalization" (paraphrased); recurrent state stored as FP32 or BF16; FP32 recurrence
 *               and FP32 per-token draft records with either storage dtype.
 *   [K3-Rubin]  "NVIDIA/TensorRT-LLM pull request 21996: Kimi K3 NVFP4 on Rubin (SM107)", section 3
 *               (the SM107 target): the KDA mixer has prefill, MTP-decode and fused-projection kernels.
 *   [K3-V2]     "NVIDIA/TensorRT-LLM pull request 19841: Kimi K3 on modeling_v2", section 5 (Route B):
 *               KDA verify kernels write per-token KDA verify states.
 *
 * The pages never print the KDA equations.  Every formula below is the plainest reading of the
 * step list above in the public gated delta-rule form; each reading is marked READING.
 *
 * Notation (per sequence b, head h, token t):
 *   H heads, dk key dim, dv value dim, r = f_a rank, K conv taps.
 *   a1  f_b projection     graw[i] = sum_j W_fb[h*dk+i][j] * f_a[j]   (W_fb BF16, or FP8 E4M3 codes
 *                          times one scale per row: the FP8 input path, [NVFP4-K3] "FP8 projection
 *                          weights"; READING: the scale granularity)
 *   a2  decay gate         g[i] = -exp(A_log[h]) * softplus(graw[i] + dt_bias[h*dk+i]);  alpha = exp(g)
 *   a3  beta               beta = sigmoid(beta_logit[h])
 *   a4  short conv + SiLU  y[c] = SiLU( sum_{j<K-1} w[c][j]*win[j][c] + w[c][K-1]*x_t[c] ),
 *                          window shifts left by one and x_t enters at the newest tap
 *   a5  L2 norms           k <- k / sqrt(|k|^2 + l2_eps);  q <- q / sqrt(|q|^2 + l2_eps) / sqrt(dk)
 *   a6  recurrence         S <- Diag(alpha) S;  u = v - S^T k;  S <- S + beta k u^T;  o = S^T q
 *   a7  gated RMSNorm      y[j] = o[j] / sqrt(mean(o^2) + norm_eps) * norm_w[j] * sigmoid(gate[j])
 *
 * Parity pins: tests/test_oracle_pins.py.  The pages print no worked KDA values, so every function
 * is pinned by closed forms, library routines, invariants, brute force on tiny inputs and the
 * recurrent-equals-chunked identity instead.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDO_VERSION 2

/* Storage modes for the recurrent state between token steps. */
enum { KDO_STORE_F64 = 0, KDO_STORE_F32 = 1, KDO_STORE_BF16 = 2 };

typedef struct {
    int H, dk, dv, r, K;        /* heads, key dim, value dim, f_a rank, conv taps */
    const uint16_t *W_fb;       /* bf16 bits [H*dk][r] */
    const double *A_log;        /* [H] */
    const double *dt_bias;      /* [H*dk] */
    const uint16_t *conv_w;     /* bf16 bits: q [H*dk][K], then k [H*dk][K], then v [H*dv][K] */
    const double *norm_w;       /* [dv] */
    double l2_eps, norm_eps;
    const uint8_t *W_fb8;       /* FP8 input path: E4M3 codes [H*dk][r], or NULL (BF16 W_fb) */
    const double *W_fb_scale;   /* FP8 input path: per-row scale [H*dk] */
} kdo_layer;

/* ---------------------------------------------------------------- scalar helpers */

/* BF16 is the upper half of an IEEE binary32; decoding is exact. */
static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 code -> value: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
 * is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities (largest value 448). */
double kdo_e4m3_to_f64(uint8_t b)
{
    const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(8.0 + m, e - 10);          /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Round a double to the nearest BF16 value (8 significant bits, binary32 exponent range),
 * ties to even, returned as a double.  Plain definition via the value's binade. */
static double round_to_bf16(double x)
{
    if (x == 0.0 || isnan(x) || isinf(x)) return x;
    int e;
    frexp(x, &e);                       /* |x| in [2^(e-1), 2^e) */
    int q = e - 8;                      /* spacing of 8-bit significands in that binade */
    if (q < -133) q = -133;             /* subnormal spacing of the binary32 exponent range */
    double scaled = ldexp(x, -q);
    double r = ldexp(nearbyint(scaled), q);   /* default rounding mode: nearest, ties to even */
    if (fabs(r) > 3.3895313892515355e38) r = copysign(INFINITY, x);
    return r;
}

/* float32 -> bf16 bits, round to nearest even; NaN stays NaN (quiet). */
uint16_t kdo_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) return (uint16_t)((u >> 16) | 0x0040u);
    double r = round_to_bf16((double)f);
    float rf = (float)r;
    uint32_t v;
    memcpy(&v, &rf, sizeof v);
    return (uint16_t)(v >> 16);
}

static double softplus(double x) { return x > 40.0 ? x : log1p(exp(x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigmoid(x); }

static double store_round(double x, int storage)
{
    if (storage == KDO_STORE_F32) return (double)(float)x;
    if (storage == KDO_STORE_BF16) return round_to_bf16(x);
    return x;
}

/* Length of one sequence's conv window: q and k windows of H*dk channels, v window of H*dv. */
static size_t window_len(const kdo_layer *L)
{
    return (size_t)(L->K - 1) * (size_t)(2 * L->H * L->dk + L->H * L->dv);
}

/* ---------------------------------------------------------------- a1..a5: per-token prep */

/* a1 + a2: per-key-channel decay alpha[i] of head h for one token. */
void kdo_decay(const kdo_layer *L, int h, const uint16_t *f_a, double *alpha)
{
    const double a = exp(L->A_log[h]);
    for (int i = 0; i < L->dk; i++) {
        const size_t row = (size_t)(h * L->dk + i);
        double graw = 0.0;
        if (L->W_fb8) {   /* FP8 input path: W = scale_row * E4M3 code, dequantised exactly */
            const uint8_t *w8 = L->W_fb8 + row * L->r;
            for (int j = 0; j < L->r; j++) graw += L->W_fb_scale[row] * kdo_e4m3_to_f64(w8[j]) * bf16_to_f64(f_a[j]);
        } else {
            const uint16_t *w = L->W_fb + row * L->r;
            for (int j = 0; j < L->r; j++) graw += bf16_to_f64(w[j]) * bf16_to_f64(f_a[j]);
        }
        double g = -a * softplus(graw + L->dt_bias[h * L->dk + i]);
        alpha[i] = exp(g);
    }
}

/* a4 for one channel: causal depthwise conv over the window plus the current input, then SiLU.
 * win points at tap 0 of this channel, taps spaced by `stride`; w has K taps (oldest first). */
static double conv_channel(const double *win, size_t stride, int K, const uint16_t *w, double x)
{
    double acc = 0.0;
    for (int j = 0; j < K - 1; j++) acc += bf16_to_f64(w[j]) * win[(size_t)j * stride];
    acc += bf16_to_f64(w[K - 1]) * x;
    return silu(acc);
}

/* Shift one channel's window left by one tap and append x. */
static void conv_shift(double *win, size_t stride, int K, double x)
{
    for (int j = 0; j < K - 2; j++) win[(size_t)j * stride] = win[(size_t)(j + 1) * stride];
    win[(size_t)(K - 2) * stride] = x;
}

/* a4 for head h of one token: q,k (dk channels each) and v (dv channels).  Reads the window
 * `win_in` (may equal win_out) and writes the shifted window to `win_out`.  Channels of other
 * heads are not touched. */
static void conv_head(const kdo_layer *L, int h, const double *win_in, double *win_out,
                      const uint16_t *xq, const uint16_t *xk, const uint16_t *xv,
                      double *q, double *k, double *v)
{
    const int K = L->K, H = L->H, dk = L->dk, dv = L->dv;
    const size_t sq = (size_t)H * dk, sv = (size_t)H * dv;
    const size_t off_k = (size_t)(K - 1) * sq, off_v = 2 * (size_t)(K - 1) * sq;
    const uint16_t *wq = L->conv_w, *wk = L->conv_w + sq * K, *wv = L->conv_w + 2 * sq * K;
    for (int i = 0; i < dk; i++) {
        size_t c = (size_t)h * dk + i;
        double x = bf16_to_f64(xq[c]);
        q[i] = conv_channel(win_in + c, sq, K, wq + c * K, x);
        if (win_out != win_in) for (int j = 0; j < K - 1; j++) win_out[c + j * sq] = win_in[c + j * sq];
        conv_shift(win_out + c, sq, K, x);
        x = bf16_to_f64(xk[c]);
        k[i] = conv_channel(win_in + off_k + c, sq, K, wk + c * K, x);
        if (win_out != win_in) for (int j = 0; j < K - 1; j++) win_out[off_k + c + j * sq] = win_in[off_k + c + j * sq];
        conv_shift(win_out + off_k + c, sq, K, x);
    }
    for (int i = 0; i < dv; i++) {
        size_t c = (size_t)h * dv + i;
        double x = bf16_to_f64(xv[c]);
        v[i] = conv_channel(win_in + off_v + c, sv, K, wv + c * K, x);
        if (win_out != win_in) for (int j = 0; j < K - 1; j++) win_out[off_v + c + j * sv] = win_in[off_v + c + j * sv];
        conv_shift(win_out + off_v + c, sv, K, x);
    }
}

/* a5: k <- k/sqrt(|k|^2+eps); q <- q/sqrt(|q|^2+eps)/sqrt(dk). */
static void l2_norms(const kdo_layer *L, double *q, double *k)
{
    double sq = 0.0, sk = 0.0;
    for (int i = 0; i < L->dk; i++) { sq += q[i] * q[i]; sk += k[i] * k[i]; }
    const double rq = 1.0 / sqrt(sq + L->l2_eps) / sqrt((double)L->dk);
    const double rk = 1.0 / sqrt(sk + L->l2_eps);
    for (int i = 0; i < L->dk; i++) { q[i] *= rq; k[i] *= rk; }
}

/* ---------------------------------------------------------------- a6, a7 */

/* a6: one gated delta-rule step on S [dk][dv] (row i = key channel, column j = value channel).
 * Exported so that the pins can drive it with hand-picked vectors. */
void kdo_recurrence_step(int dk, int dv, double *S, const double *alpha, const double *k,
                         const double *v, const double *q, double beta, double *o)
{
    for (int i = 0; i < dk; i++)
        for (int j = 0; j < dv; j++) S[(size_t)i * dv + j] *= alpha[i];
    for (int j = 0; j < dv; j++) {
        double stk = 0.0;
        for (int i = 0; i < dk; i++) stk += S[(size_t)i * dv + j] * k[i];
        double u = v[j] - stk;
        for (int i = 0; i < dk; i++) S[(size_t)i * dv + j] += beta * k[i] * u;
    }
    for (int j = 0; j < dv; j++) {
        double acc = 0.0;
        for (int i = 0; i < dk; i++) acc += S[(size_t)i * dv + j] * q[i];
        o[j] = acc;
    }
}

/* a7: y = o / sqrt(mean(o^2)+eps) * w * sigmoid(gate). */
void kdo_gated_rmsnorm(int dv, const double *o, const double *norm_w, double eps,
                       const uint16_t *gate, double *y)
{
    double ss = 0.0;
    for (int j = 0; j < dv; j++) ss += o[j] * o[j];
    const double rinv = 1.0 / sqrt(ss / dv + eps);
    for (int j = 0; j < dv; j++) y[j] = o[j] * rinv * norm_w[j] * sigmoid(bf16_to_f64(gate[j]));
}

/* One token of one (sequence, head): a1..a7.  S [dk][dv] in/out (not storage-rounded here);
 * window read from win_in and written (shifted) to win_out; y [dv] receives the output. */
static void token_head(const kdo_layer *L, int h, double *S, const double *win_in, double *win_out,
                       const uint16_t *xq, const uint16_t *xk, const uint16_t *xv,
                       const uint16_t *f_a, const uint16_t *beta_logit, const uint16_t *gate,
                       double *y, double *scratch)
{
    const int dk = L->dk, dv = L->dv;
    double *alpha = scratch, *q = alpha + dk, *k = q + dk, *v = k + dk, *o = v + dv;
    kdo_decay(L, h, f_a, alpha);
    conv_head(L, h, win_in, win_out, xq, xk, xv, q, k, v);
    l2_norms(L, q, k);
    const double beta = sigmoid(bf16_to_f64(beta_logit[h]));
    kdo_recurrence_step(dk, dv, S, alpha, k, v, q, beta, o);
    kdo_gated_rmsnorm(dv, o, L->norm_w, L->norm_eps, gate + (size_t)h * dv, y);
}

static size_t scratch_len(const kdo_layer *L) { return 3 * (size_t)L->dk + 2 * (size_t)L->dv; }

static int check_layer(const kdo_layer *L)
{
    if (!L || L->H < 1 || L->dk < 1 || L->dv < 1 || L->r < 1 || L->K < 2) return 1;
    if ((!L->W_fb && !L->W_fb8) || !L->A_log || !L->dt_bias || !L->conv_w || !L->norm_w) return 1;
    if (L->W_fb8 && !L->W_fb_scale) return 1;
    return 0;
}

int kdo_version(void) { return KDO_VERSION; }

int kdo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void kdo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- decode
 * n_steps consecutive single-token steps for B sequences.
 *   state  [B][H][dk][dv]   in/out (the sequences' slot states, already gathered)
 *   window [B][window_len]  in/out
 *   inputs per step s, sequence b: q,k [s][b][H*dk], v [s][b][H*dv], f_a [s][b][r],
 *          beta_logit [s][b][H], gate [s][b][H*dv]   (bf16 bits)
 *   out    [s][b][H*dv]     unrounded outputs
 * `storage` rounds the state to the storage dtype after every token (FP32 recurrence, state
 * stored as FP32 or BF16 between steps, [NVFP4-K3] Description). */
int kdo_decode(const kdo_layer *L, int B, int n_steps, int storage, double *state, double *window,
               const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *f_a,
               const uint16_t *beta_logit, const uint16_t *gate, double *out)
{
    if (check_layer(L) || B < 0 || n_steps < 0) return 1;
    const int H = L->H, dk = L->dk, dv = L->dv;
    const size_t wl = window_len(L), sz = (size_t)dk * dv;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            double *scr = malloc(scratch_len(L) * sizeof(double));
            if (!scr) { bad = 1; continue; }
            double *S = state + ((size_t)b * H + h) * sz;
            double *win = window + (size_t)b * wl;
            for (int s = 0; s < n_steps; s++) {
                size_t tb = (size_t)s * B + b;
                token_head(L, h, S, win, win, q + tb * H * dk, k + tb * H * dk, v + tb * H * dv,
                           f_a + tb * L->r, beta_logit + tb * H, gate + tb * H * dv,
                           out + tb * H * dv + (size_t)h * dv, scr);
                for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);
            }
            free(scr);
        }
    return bad;
}

/* ---------------------------------------------------------------- verify
 * T draft tokens per sequence, in order, from the slot state.  The state stays in full
 * precision across the T tokens (FP32 per-token draft records with either storage dtype,
 * [NVFP4-K3] Description; per-token verify states, [K3-V2] section 5).
 *   state [B][H][dk][dv], window [B][window_len]: read only
 *   inputs [b][t][...]; records [b][t][H][dk][dv]; window records [b][t][window_len];
 *   out [b][t][H*dv] */
int kdo_verify(const kdo_layer *L, int B, int T, const double *state, const double *window,
               const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *f_a,
               const uint16_t *beta_logit, const uint16_t *gate, double *rec_state,
               double *rec_window, double *out)
{
    if (check_layer(L) || B < 0 || T < 0) return 1;
    const int H = L->H, dk = L->dk, dv = L->dv;
    const size_t wl = window_len(L), sz = (size_t)dk * dv;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            double *scr = malloc((scratch_len(L) + sz) * sizeof(double));
            if (!scr) { bad = 1; continue; }
            double *S = scr + scratch_len(L);
            memcpy(S, state + ((size_t)b * H + h) * sz, sz * sizeof(double));
            const double *win_prev = window + (size_t)b * wl;
            for (int t = 0; t < T; t++) {
                size_t bt = (size_t)b * T + t;
                double *win_t = rec_window + bt * wl;
                token_head(L, h, S, win_prev, win_t, q + bt * H * dk, k + bt * H * dk,
                           v + bt * H * dv, f_a + bt * L->r, beta_logit + bt * H, gate + bt * H * dv,
                           out + bt * H * dv + (size_t)h * dv, scr);
                memcpy(rec_state + (bt * H + h) * sz, S, sz * sizeof(double));
                win_prev = win_t;
            }
            free(scr);
        }
    return bad;
}

/* ---------------------------------------------------------------- commit
 * For each sequence b with n = accepted[b] >= 1: slot state <- storage cast of record[b][n-1],
 * slot conv window <- window record[b][n-1].  n == 0 leaves the slot untouched.
 * Operates on raw pool bytes exactly as stored:
 *   pool_state  float32 or bf16 bits [num_slots][H][dk][dv] (storage 1 or 2)
 *   pool_window bf16 bits [num_slots][window_len]
 *   rec_state   float32 [B][T][H][dk][dv];  rec_window bf16 bits [B][T][window_len]
 * Returns 2 when an id or length is out of range (nothing is written for that sequence). */
int kdo_commit(int B, int T, int H, int dk, int dv, int K, int storage, int num_slots,
               void *pool_state, uint16_t *pool_window, const int32_t *slot_ids,
               const int32_t *accepted, const float *rec_state, const uint16_t *rec_window)
{
    const size_t sz = (size_t)H * dk * dv, wl = (size_t)(K - 1) * (2 * H * dk + H * dv);
    int rc = 0;
    for (int b = 0; b < B; b++) {
        int n = accepted[b], s = slot_ids[b];
        if (n < 0 || n > T || s < 0 || s >= num_slots) { rc = 2; continue; }
        if (n == 0) continue;
        const float *src = rec_state + ((size_t)b * T + (n - 1)) * sz;
        if (storage == KDO_STORE_F32) {
            memcpy((float *)pool_state + (size_t)s * sz, src, sz * sizeof(float));
        } else {
            uint16_t *dst = (uint16_t *)pool_state + (size_t)s * sz;
            for (size_t e = 0; e < sz; e++) dst[e] = kdo_f32_to_bf16(src[e]);
        }
        memcpy(pool_window + (size_t)s * wl, rec_window + ((size_t)b * T + (n - 1)) * wl,
               wl * sizeof(uint16_t));
    }
    return rc;
}

/* ---------------------------------------------------------------- prefill (token by token)
 * L_tok tokens per sequence from the given state and window (in/out), one token at a time:
 * the reference the chunked prefill is checked against.  The state is kept in full precision
 * across the tokens and rounded to the storage dtype once at the end.
 *   inputs [b][t][...], out [b][t][H*dv]. */
int kdo_prefill(const kdo_layer *L, int B, int L_tok, int storage, double *state, double *window,
                const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *f_a,
                const uint16_t *beta_logit, const uint16_t *gate, double *out)
{
    if (check_layer(L) || B < 0 || L_tok < 0) return 1;
    const int H = L->H, dk = L->dk, dv = L->dv;
    const size_t wl = window_len(L), sz = (size_t)dk * dv;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            double *scr = malloc(scratch_len(L) * sizeof(double));
            if (!scr) { bad = 1; continue; }
            double *S = state + ((size_t)b * H + h) * sz;
            double *win = window + (size_t)b * wl;
            for (int t = 0; t < L_tok; t++) {
                size_t bt = (size_t)b * L_tok + t;
                token_head(L, h, S, win, win, q + bt * H * dk, k + bt * H * dk, v + bt * H * dv,
                           f_a + bt * L->r, beta_logit + bt * H, gate + bt * H * dv,
                           out + bt * H * dv + (size_t)h * dv, scr);
            }
            for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);
            free(scr);
        }
    return bad;
}

/* ---------------------------------------------------------------- prefill (chunk form)
 * The same recurrence written chunk by chunk (the WY / UT form that chunked prefill kernels
 * use, [K3-Rubin] section 3).  Within a chunk of C tokens with entry state S0, let Gam_t be the
 * inclusive cumulative log-decay per key channel and kt_s = beta_s * u_s.  Then
 *   M[t][s]  = beta_t * sum_c k_t[c] k_s[c] exp(Gam_t[c] - Gam_s[c])        (s < t)
 *   (I + M) Ut = diag(beta) V - diag(beta) Ktil S0,   Ktil_t = k_t * exp(Gam_t)
 *   O[t]     = S0^T (q_t * exp(Gam_t)) + sum_{s<=t} P[t][s] Ut_s,
 *              P[t][s] = sum_c q_t[c] k_s[c] exp(Gam_t[c] - Gam_s[c])
 *   S_end    = Diag(exp(Gam_last)) S0 + sum_s (k_s * exp(Gam_last - Gam_s)) Ut_s^T
 * The exponent differences are formed directly (no factorisation), so nothing overflows.
 * Used only to pin the identity "recurrent = chunked"; the conv / gate / norm prep is the same
 * per-token code as above. */
int kdo_prefill_chunked(const kdo_layer *L, int B, int L_tok, int chunk, int storage,
                        double *state, double *window, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const uint16_t *f_a, const uint16_t *beta_logit,
                        const uint16_t *gate, double *out)
{
    if (check_layer(L) || B < 0 || L_tok < 0 || chunk < 1) return 1;
    const int H = L->H, dk = L->dk, dv = L->dv, C = chunk;
    const size_t wl = window_len(L), sz = (size_t)dk * dv;
    int bad = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            /* per-chunk buffers */
            double *Q = malloc((size_t)C * dk * sizeof(double));
            double *Kc = malloc((size_t)C * dk * sizeof(double));
            double *V = malloc((size_t)C * dv * sizeof(double));
            double *Gm = malloc((size_t)C * dk * sizeof(double));
            double *bet = malloc((size_t)C * sizeof(double));
            double *M = malloc((size_t)C * C * sizeof(double));
            double *Ut = malloc((size_t)C * dv * sizeof(double));
            double *o = malloc((size_t)dv * sizeof(double));
            double *alpha = malloc((size_t)dk * sizeof(double));
            double *Snew = malloc(sz * sizeof(double));
            if (!Q || !Kc || !V || !Gm || !bet || !M || !Ut || !o || !alpha || !Snew) {
                bad = 1;
                goto done;
            }
            double *S = state + ((size_t)b * H + h) * sz;
            double *win = window + (size_t)b * wl;
            for (int t0 = 0; t0 < L_tok; t0 += C) {
                const int n = (L_tok - t0 < C) ? (L_tok - t0) : C;
                /* prep: conv, norms, gates, cumulative log-decay */
                for (int t = 0; t < n; t++) {
                    size_t bt = (size_t)b * L_tok + t0 + t;
                    conv_head(L, h, win, win, q + bt * H * dk, k + bt * H * dk, v + bt * H * dv,
                              Q + (size_t)t * dk, Kc + (size_t)t * dk, V + (size_t)t * dv);
                    l2_norms(L, Q + (size_t)t * dk, Kc + (size_t)t * dk);
                    kdo_decay(L, h, f_a + bt * L->r, alpha);
                    for (int c = 0; c < dk; c++)
                        Gm[(size_t)t * dk + c] = log(alpha[c]) + (t ? Gm[(size_t)(t - 1) * dk + c] : 0.0);
                    bet[t] = sigmoid(bf16_to_f64(beta_logit[bt * H + h]));
                }
                /* M (strictly lower) */
                for (int t = 0; t < n; t++)
                    for (int s = 0; s < t; s++) {
                        double acc = 0.0;
                        for (int c = 0; c < dk; c++)
                            acc += Kc[(size_t)t * dk + c] * Kc[(size_t)s * dk + c] *
                                   exp(Gm[(size_t)t * dk + c] - Gm[(size_t)s * dk + c]);
                        M[(size_t)t * C + s] = bet[t] * acc;
                    }
                /* right-hand side, then forward substitution with the unit lower matrix I + M */
                for (int t = 0; t < n; t++)
                    for (int j = 0; j < dv; j++) {
                        double ks0 = 0.0;
                        for (int c = 0; c < dk; c++)
                            ks0 += Kc[(size_t)t * dk + c] * exp(Gm[(size_t)t * dk + c]) * S[(size_t)c * dv + j];
                        double rhs = bet[t] * (V[(size_t)t * dv + j] - ks0);
                        for (int s = 0; s < t; s++) rhs -= M[(size_t)t * C + s] * Ut[(size_t)s * dv + j];
                        Ut[(size_t)t * dv + j] = rhs;
                    }
                /* outputs */
                for (int t = 0; t < n; t++) {
                    size_t bt = (size_t)b * L_tok + t0 + t;
                    for (int j = 0; j < dv; j++) {
                        double acc = 0.0;
                        for (int c = 0; c < dk; c++)
                            acc += Q[(size_t)t * dk + c] * exp(Gm[(size_t)t * dk + c]) * S[(size_t)c * dv + j];
                        o[j] = acc;
                    }
                    for (int s = 0; s <= t; s++) {
                        double p = 0.0;
                        for (int c = 0; c < dk; c++)
                            p += Q[(size_t)t * dk + c] * Kc[(size_t)s * dk + c] *
                                 exp(Gm[(size_t)t * dk + c] - Gm[(size_t)s * dk + c]);
                        for (int j = 0; j < dv; j++) o[j] += p * Ut[(size_t)s * dv + j];
                    }
                    kdo_gated_rmsnorm(dv, o, L->norm_w, L->norm_eps, gate + bt * H * dv + (size_t)h * dv,
                                      out + bt * H * dv + (size_t)h * dv);
                }
                /* state at the chunk end */
                const double *Gl = Gm + (size_t)(n - 1) * dk;
                for (int c = 0; c < dk; c++)
                    for (int j = 0; j < dv; j++) {
                        double acc = exp(Gl[c]) * S[(size_t)c * dv + j];
                        for (int s = 0; s < n; s++)
                            acc += Kc[(size_t)s * dk + c] * exp(Gl[c] - Gm[(size_t)s * dk + c]) * Ut[(size_t)s * dv + j];
                        Snew[(size_t)c * dv + j] = acc;
                    }
                memcpy(S, Snew, sz * sizeof(double));
            }
            for (size_t e = 0; e < sz; e++) S[e] = store_round(S[e], storage);
        done:
            free(Q); free(Kc); free(V); free(Gm); free(bet); free(M); free(Ut); free(o); free(alpha); free(Snew);
        }
    return bad;
}

/* ---------------------------------------------------------------- exported pieces for the pins */

/* a4 + shift for a single channel sequence: y[t] for x[0..n) starting from window w0 [K-1]. */
void kdo_conv_sequence(int K, const uint16_t *w, const double *w0, const uint16_t *x, int n, double *y,
                       double *w_end)
{
    double win[64];
    for (int j = 0; j < K - 1 && j < 64; j++) win[j] = w0[j];
    for (int t = 0; t < n; t++) {
        double xt = bf16_to_f64(x[t]);
        y[t] = conv_channel(win, 1, K, w, xt);
        conv_shift(win, 1, K, xt);
    }
    for (int j = 0; j < K - 1 && j < 64; j++) w_end[j] = win[j];
}

/* a5 on explicit vectors (q, k of length dk, in place). */
void kdo_l2_norms(int dk, double l2_eps, double *q, double *k)
{
    kdo_layer L;
    memset(&L, 0, sizeof L);
    L.dk = dk;
    L.l2_eps = l2_eps;
    l2_norms(&L, q, k);
}

/* Storage rounding on an array (for pins of the BF16 emulation). */
void kdo_store_round(double *x, size_t n, int storage)
{
    for (size_t i = 0; i < n; i++) x[i] = store_round(x[i], storage);
}
