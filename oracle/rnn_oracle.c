/*
 * rnn_oracle.c -- plain, slow, single-threaded CPU oracle for the ONNX RNN,
 * GRU and LSTM sequence operators.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the CPU
 * baseline leg of the benchmark may load this file.  The product path (the
 * CUDA library) never calls it, shares no code, header, table or constant
 * with it, and fails if its own extension is missing.
 *
 * What it computes (page "Recurrent operators: RNN, GRU, LSTM"):
 *   - Computation: per direction, XW = X.W^T with one fp32 accumulator per
 *     output, k increasing from +0; per step Rec = H.R^T the same way; for GRU
 *     with linear_before_reset = 0 the candidate product (r (.) H).Rh^T is
 *     formed after r is known.  Every '*' and '+' is one IEEE fp32 operation,
 *     rounded to nearest even; nothing is fused (build with -ffp-contract=off).
 *     pre = ((xw + rec) + Wb) + Rb, the bias adds skipped when B is absent;
 *     LSTM peepholes are added after the biases (Pi, Pf with the previous cell,
 *     Po with the new one); clip (when present and positive) then clamps every
 *     gate input to [-clip, clip], a NaN passing through.
 *   - Activations: f, g, h per direction, names case-insensitive, defaults,
 *     alpha/beta consumed by separate cursors in activation order.
 *   - Choices the specification leaves open: sequence_lens (a row runs its
 *     first len steps; reverse starts at len-1; Y = 0 at t >= len; Y_h/Y_c are
 *     the state after the last valid step, 0 for a length-0 row; a length
 *     outside [0, seq] is InvalidInput), input_forget (f = 1 - i), layout 1
 *     (the layout-0 case with every tensor transposed), omitted inputs are
 *     zeros, zero-size runs nothing, hidden_size 0 is an error.
 *   - Exact mode: every NaN written to Y, Y_h, Y_c is 0x7FC00000.
 *
 * The transcendental functions (exp, log, tanh, sigmoid) are this library's
 * own, built from IEEE +, -, *, / and bit operations only; their definition is
 * given at each function.  The page's own polynomials are not available, so
 * bit parity with that library is unpinned; accuracy is pinned by the tests
 * against double-precision math.
 *
 * oracle_rnn_cell computes the single RNN cell of page "RNNCell" (RNNCell-3)
 * in the same rounding order (its header gives the reading).
 *
 * Status codes: 0 ok, 1 invalid argument, 2 invalid input.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ bits */

static float o_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t o_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static int o_isnan(float x) { return x != x; }
static float o_fabs(float x) { return o_from_bits(o_to_bits(x) & 0x7FFFFFFFu); }
static float o_canon(float x) { return o_isnan(x) ? o_from_bits(0x7FC00000u) : x; }

/* ------------------------------------------------------ own exp/log/tanh */

/* exp(x): Cody-Waite reduction x = k*ln2 + r, |r| <= ln2/2, with ln2 split
 * into a 15-significant-bit head (so k*head is exact for |k| < 256) and a
 * tail; then the degree-7 Taylor polynomial of e^r in Horner form (each
 * multiply and add rounded); then scaling by 2^k as two exact powers of two
 * built from exponent bits, so only the last multiply can round (this also
 * gives correctly rounded underflow into subnormals and overflow to inf). */
float oracle_exp(float x)
{
    /* ln2 head: ln(2) rounded to 15 significant bits = 0.693145751953125 */
    const float LN2_HEAD = 0.693145751953125f;
    /* ln2 tail: float(ln(2) - head) */
    const float LN2_TAIL = 1.42860677e-06f;
    /* 1/ln(2) rounded to float */
    const float INV_LN2 = 1.44269502f;
    /* 1.5 * 2^23: adding and subtracting it rounds a float to an integer */
    const float ROUNDER = 12582912.0f;
    /* Taylor coefficients 1/n!, each the float nearest the rational */
    const float E2 = 0.5f;             /* 1/2    */
    const float E3 = 0.166666672f;     /* 1/6    */
    const float E4 = 0.0416666679f;    /* 1/24   */
    const float E5 = 0.00833333377f;   /* 1/120  */
    const float E6 = 0.00138888892f;   /* 1/720  */
    const float E7 = 0.000198412701f;  /* 1/5040 */

    if (o_isnan(x)) return x;
    if (x > 89.0f) return o_from_bits(0x7F800000u);
    if (x < -110.0f) return 0.0f;

    float t = x * INV_LN2;
    float kf = (t + ROUNDER) - ROUNDER;
    float r = (x - kf * LN2_HEAD) - kf * LN2_TAIL;

    float p = E7;
    p = p * r + E6;
    p = p * r + E5;
    p = p * r + E4;
    p = p * r + E3;
    p = p * r + E2;
    p = p * r + 1.0f;
    p = p * r + 1.0f;

    int k = (int)kf;
    int k1 = k / 2;
    int k2 = k - k1;
    float s1 = o_from_bits((uint32_t)(k1 + 127) << 23);
    float s2 = o_from_bits((uint32_t)(k2 + 127) << 23);
    return (p * s1) * s2;
}

/* log(x): x = m * 2^e with m in [sqrt(1/2), sqrt(2)); s = (m-1)/(m+1);
 * log(m) = 2*atanh(s) = 2s + 2s*(z/3 + z^2/5 + z^3/7 + z^4/9 + z^5/11),
 * z = s*s, Horner with each operation rounded; log(x) = e*head + (log(m) +
 * e*tail) with the same ln2 split as exp. */
float oracle_log(float x)
{
    const float LN2_HEAD = 0.693145751953125f;
    const float LN2_TAIL = 1.42860677e-06f;
    const float SQRT2 = 1.41421354f;   /* float nearest sqrt(2) */
    const float L3 = 0.333333343f;     /* 1/3  */
    const float L5 = 0.200000003f;     /* 1/5  */
    const float L7 = 0.142857149f;     /* 1/7  */
    const float L9 = 0.111111112f;     /* 1/9  */
    const float L11 = 0.0909090936f;   /* 1/11 */

    if (o_isnan(x)) return x;
    if (x < 0.0f) return o_from_bits(0x7FC00000u);
    if (x == 0.0f) return o_from_bits(0xFF800000u);
    if (x == o_from_bits(0x7F800000u)) return x;

    int eadj = 0;
    if (x < o_from_bits(0x00800000u)) {        /* subnormal: scale by 2^24 */
        x = x * 16777216.0f;
        eadj = -24;
    }
    uint32_t b = o_to_bits(x);
    int e = (int)((b >> 23) & 0xFFu) - 127 + eadj;
    float m = o_from_bits((b & 0x007FFFFFu) | 0x3F800000u);
    if (m > SQRT2) {
        m = m * 0.5f;
        e = e + 1;
    }
    float f = m - 1.0f;
    float s = f / (m + 1.0f);
    float z = s * s;
    float q = L11;
    q = q * z + L9;
    q = q * z + L7;
    q = q * z + L5;
    q = q * z + L3;
    float w = q * z;
    float s2 = s + s;
    float lm = s2 + s2 * w;
    float ef = (float)e;
    return ef * LN2_HEAD + (lm + ef * LN2_TAIL);
}

/* tanh(x): |x| > 9.1 gives +-1; |x| < 0.4 uses the odd Taylor series
 * a + a*z*(T3 + z*(T5 + ... + z*T13)), z = a*a, with the series' rational
 * coefficients -1/3, 2/15, -17/315, 62/2835, -1382/155925, 21844/6081075;
 * otherwise 1 - 2/(exp(2a) + 1).  The sign of x is restored at the end. */
float oracle_tanh(float x)
{
    const float T3 = -0.333333343f;      /* -1/3            */
    const float T5 = 0.13333334f;        /* 2/15            */
    const float T7 = -0.0539682545f;     /* -17/315         */
    const float T9 = 0.0218694881f;      /* 62/2835         */
    const float T11 = -0.00886323582f;   /* -1382/155925    */
    const float T13 = 0.00359212793f;    /* 21844/6081075   */

    if (o_isnan(x)) return x;
    uint32_t sign = o_to_bits(x) & 0x80000000u;
    float a = o_fabs(x);
    float y;
    if (a > 9.1f) {
        y = 1.0f;
    } else if (a < 0.4f) {
        float z = a * a;
        float q = T13;
        q = q * z + T11;
        q = q * z + T9;
        q = q * z + T7;
        q = q * z + T5;
        q = q * z + T3;
        float w = q * z;
        y = a + a * w;
    } else {
        float e = oracle_exp(a + a);
        y = 1.0f - 2.0f / (e + 1.0f);
    }
    return o_from_bits(o_to_bits(y) | sign);
}

/* sigmoid(x) = 1 / (1 + exp(-x)) */
float oracle_sigmoid(float x)
{
    return 1.0f / (1.0f + oracle_exp(-x));
}

/* ------------------------------------------------------------ activations */

enum {
    OA_RELU = 0, OA_TANH, OA_SIGMOID, OA_AFFINE, OA_LEAKYRELU,
    OA_THRESHOLDEDRELU, OA_SCALEDTANH, OA_HARDSIGMOID, OA_ELU,
    OA_SOFTSIGN, OA_SOFTPLUS, OA_COUNT
};

static const char* const o_act_names[OA_COUNT] = {
    "relu", "tanh", "sigmoid", "affine", "leakyrelu", "thresholdedrelu",
    "scaledtanh", "hardsigmoid", "elu", "softsign", "softplus"
};

typedef struct { int fn; float alpha; float beta; } OAct;

/* Definitions from the Activations section. */
float oracle_activation(int fn, float alpha, float beta, float x)
{
    switch (fn) {
    case OA_RELU:            return x < 0.0f ? 0.0f : x;
    case OA_TANH:            return oracle_tanh(x);
    case OA_SIGMOID:         return oracle_sigmoid(x);
    case OA_AFFINE:          return alpha * x + beta;
    case OA_LEAKYRELU:       return x < 0.0f ? alpha * x : x;
    case OA_THRESHOLDEDRELU: return x > alpha ? x : 0.0f;
    case OA_SCALEDTANH:      return alpha * oracle_tanh(beta * x);
    case OA_HARDSIGMOID: {
        float v = alpha * x + beta;
        /* min(1, max(0, v)) written with compares so that a NaN propagates */
        return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);
    }
    case OA_ELU:             return x >= 0.0f ? x : alpha * (oracle_exp(x) - 1.0f);
    case OA_SOFTSIGN:        return x / (1.0f + o_fabs(x));
    case OA_SOFTPLUS:        return x > 20.0f ? x : oracle_log(1.0f + oracle_exp(x));
    default:                 return o_from_bits(0x7FC00000u);
    }
}

static int o_takes_alpha(int fn)
{
    return fn == OA_AFFINE || fn == OA_LEAKYRELU || fn == OA_THRESHOLDEDRELU ||
           fn == OA_SCALEDTANH || fn == OA_HARDSIGMOID || fn == OA_ELU;
}

static int o_takes_beta(int fn)
{
    return fn == OA_AFFINE || fn == OA_SCALEDTANH || fn == OA_HARDSIGMOID;
}

static float o_default_alpha(int fn)
{
    switch (fn) {
    case OA_LEAKYRELU: return 0.01f;
    case OA_THRESHOLDEDRELU: return 1.0f;
    case OA_ELU: return 1.0f;
    case OA_HARDSIGMOID: return 0.2f;
    case OA_AFFINE: return 1.0f;
    case OA_SCALEDTANH: return 1.0f;
    default: return 0.0f;
    }
}

static float o_default_beta(int fn)
{
    switch (fn) {
    case OA_HARDSIGMOID: return 0.5f;
    default: return 0.0f;   /* Affine and ScaledTanh default beta is 0 */
    }
}

static int o_name_to_fn(const char* s)
{
    if (!s) return -1;
    for (int f = 0; f < OA_COUNT; ++f) {
        const char* a = o_act_names[f];
        size_t i = 0;
        for (;; ++i) {
            char c = s[i];
            if (c >= 'A' && c <= 'Z') c = (char)(c - 'A' + 'a');
            if (c != a[i]) break;
            if (c == '\0') return f;
        }
    }
    return -1;
}

static int o_gates(int op) { return op == 0 ? 1 : (op == 1 ? 3 : 4); }
static int o_acts_per_dir(int op) { return op == 0 ? 1 : (op == 1 ? 2 : 3); }

/* Resolve the activation list into [dirs][3] (fn, alpha, beta) triples.
 * Returns 0 or 1 (invalid argument). */
int oracle_resolve_activations(int op, int direction,
                               const char* const* acts, int n_acts,
                               const float* alpha, int n_alpha,
                               const float* beta, int n_beta,
                               int* fn_out, float* alpha_out, float* beta_out)
{
    if (op < 0 || op > 2 || direction < 0 || direction > 2) return 1;
    int k = o_acts_per_dir(op);
    int dirs = direction == 2 ? 2 : 1;
    OAct list[6];
    int n_list;
    if (n_acts == 0) {
        /* defaults: LSTM Sigmoid, Tanh, Tanh; GRU Sigmoid, Tanh; RNN Tanh */
        if (op == 0) { list[0].fn = OA_TANH; }
        else if (op == 1) { list[0].fn = OA_SIGMOID; list[1].fn = OA_TANH; }
        else { list[0].fn = OA_SIGMOID; list[1].fn = OA_TANH; list[2].fn = OA_TANH; }
        n_list = k;
        for (int i = 0; i < n_list; ++i) {
            list[i].alpha = o_default_alpha(list[i].fn);
            list[i].beta = o_default_beta(list[i].fn);
        }
    } else {
        if (n_acts != k && n_acts != 2 * k) return 1;
        if (!acts) return 1;
        n_list = n_acts;
        int ca = 0, cb = 0;       /* separate alpha and beta cursors */
        for (int i = 0; i < n_list; ++i) {
            int fn = o_name_to_fn(acts[i]);
            if (fn < 0) return 1;
            list[i].fn = fn;
            list[i].alpha = o_default_alpha(fn);
            list[i].beta = o_default_beta(fn);
            if (o_takes_alpha(fn)) {
                if (alpha && ca < n_alpha) list[i].alpha = alpha[ca];
                ca++;
            }
            if (o_takes_beta(fn)) {
                if (beta && cb < n_beta) list[i].beta = beta[cb];
                cb++;
            }
        }
    }
    for (int d = 0; d < dirs; ++d) {
        int base = (n_list == 2 * k && d == 1) ? k : 0;
        for (int s = 0; s < 3; ++s) {
            int idx = d * 3 + s;
            if (s < k) {
                fn_out[idx] = list[base + s].fn;
                alpha_out[idx] = list[base + s].alpha;
                beta_out[idx] = list[base + s].beta;
            } else {
                fn_out[idx] = -1;
                alpha_out[idx] = 0.0f;
                beta_out[idx] = 0.0f;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------- operator */

typedef struct {
    int op, dirs, G, layout, lbr, input_forget, has_clip;
    long S, N, I, H;
    float clip;
    const float *X, *W, *R, *B, *h0, *c0, *P;
    const int32_t* lens;
    float *Y, *Yh, *Yc;
} OArgs;

static long o_xidx(const OArgs* a, long t, long n)
{
    return a->layout == 0 ? (t * a->N + n) * a->I : (n * a->S + t) * a->I;
}

static long o_yidx(const OArgs* a, long t, long d, long n)
{
    return a->layout == 0 ? ((t * a->dirs + d) * a->N + n) * a->H
                          : ((n * a->S + t) * a->dirs + d) * a->H;
}

static long o_sidx(const OArgs* a, long d, long n)   /* initial_h, Y_h, ... */
{
    return a->layout == 0 ? (d * a->N + n) * a->H : (n * a->dirs + d) * a->H;
}

/* One accumulator, k increasing from +0, each product and sum rounded. */
static float o_dot(const float* x, const float* w, long K)
{
    float acc = 0.0f;
    for (long k = 0; k < K; ++k) acc = acc + x[k] * w[k];
    return acc;
}

static float o_clip(const OArgs* a, float v)
{
    if (!a->has_clip) return v;
    if (v > a->clip) return a->clip;
    if (v < -a->clip) return -a->clip;
    return v;   /* also a NaN */
}

static float o_act(const OAct* f, float x)
{
    return oracle_activation(f->fn, f->alpha, f->beta, x);
}

/* XW for one (t, n): xw[j] = sum_k X[t,n,k] * W[d][j][k] over all G*H j. */
static void o_project(const OArgs* a, long d, long t, long n, float* xw)
{
    long GH = a->G * a->H;
    const float* x = a->X + o_xidx(a, t, n);
    for (long j = 0; j < GH; ++j)
        xw[j] = o_dot(x, a->W + (d * GH + j) * a->I, a->I);
}

static void o_run_row(const OArgs* a, long d, long n, int reverse,
                      const OAct* acts, float* buf)
{
    long H = a->H, GH = a->G * a->H;
    float* h = buf;
    float* c = h + H;
    float* hn = c + H;
    float* cn = hn + H;
    float* z = cn + H;
    float* r = z + H;
    float* rh = r + H;
    float* xw = rh + H;
    const float* Rd = a->R + d * GH * H;
    const float* Wb = a->B ? a->B + d * 2 * GH : NULL;
    const float* Rb = a->B ? a->B + d * 2 * GH + GH : NULL;
    const float* Pi = a->P ? a->P + d * 3 * H : NULL;
    const float* Po = a->P ? a->P + d * 3 * H + H : NULL;
    const float* Pf = a->P ? a->P + d * 3 * H + 2 * H : NULL;

    for (long u = 0; u < H; ++u) {
        h[u] = a->h0 ? a->h0[o_sidx(a, d, n) + u] : 0.0f;
        c[u] = a->c0 ? a->c0[o_sidx(a, d, n) + u] : 0.0f;
    }
    long L = a->lens ? (long)a->lens[n] : a->S;

    for (long s = 0; s < L; ++s) {
        long t = reverse ? L - 1 - s : s;
        o_project(a, d, t, n, xw);
        if (a->op == 0) {                                    /* RNN */
            for (long u = 0; u < H; ++u) {
                float pre = xw[u] + o_dot(h, Rd + u * H, H);
                if (a->B) { pre = pre + Wb[u]; pre = pre + Rb[u]; }
                hn[u] = o_act(&acts[0], o_clip(a, pre));
            }
        } else if (a->op == 1) {                             /* GRU z, r, h */
            for (long u = 0; u < H; ++u) {
                float pz = xw[u] + o_dot(h, Rd + u * H, H);
                float pr = xw[H + u] + o_dot(h, Rd + (H + u) * H, H);
                if (a->B) {
                    pz = pz + Wb[u]; pz = pz + Rb[u];
                    pr = pr + Wb[H + u]; pr = pr + Rb[H + u];
                }
                z[u] = o_act(&acts[0], o_clip(a, pz));
                r[u] = o_act(&acts[0], o_clip(a, pr));
            }
            if (a->lbr == 0) {
                for (long k = 0; k < H; ++k) rh[k] = r[k] * h[k];
            }
            for (long u = 0; u < H; ++u) {
                const float* Rh = Rd + (2 * H + u) * H;
                float ph;
                if (a->lbr == 0) {
                    ph = xw[2 * H + u] + o_dot(rh, Rh, H);
                    if (a->B) { ph = ph + Wb[2 * H + u]; ph = ph + Rb[2 * H + u]; }
                } else {
                    float rec = o_dot(h, Rh, H);
                    if (a->B) ph = (xw[2 * H + u] + r[u] * (rec + Rb[2 * H + u])) + Wb[2 * H + u];
                    else ph = xw[2 * H + u] + r[u] * rec;
                }
                float ht = o_act(&acts[1], o_clip(a, ph));
                hn[u] = (1.0f - z[u]) * ht + z[u] * h[u];
            }
        } else {                                             /* LSTM i, o, f, c */
            for (long u = 0; u < H; ++u) {
                float pi = xw[u] + o_dot(h, Rd + u * H, H);
                float po = xw[H + u] + o_dot(h, Rd + (H + u) * H, H);
                float pf = xw[2 * H + u] + o_dot(h, Rd + (2 * H + u) * H, H);
                float pc = xw[3 * H + u] + o_dot(h, Rd + (3 * H + u) * H, H);
                if (a->B) {
                    pi = pi + Wb[u];         pi = pi + Rb[u];
                    po = po + Wb[H + u];     po = po + Rb[H + u];
                    pf = pf + Wb[2 * H + u]; pf = pf + Rb[2 * H + u];
                    pc = pc + Wb[3 * H + u]; pc = pc + Rb[3 * H + u];
                }
                if (a->P) {
                    pi = pi + Pi[u] * c[u];
                    pf = pf + Pf[u] * c[u];
                }
                float ig = o_act(&acts[0], o_clip(a, pi));
                float fg = a->input_forget ? 1.0f - ig : o_act(&acts[0], o_clip(a, pf));
                float ct = o_act(&acts[1], o_clip(a, pc));
                cn[u] = fg * c[u] + ig * ct;
                if (a->P) po = po + Po[u] * cn[u];
                float og = o_act(&acts[0], o_clip(a, po));
                hn[u] = og * o_act(&acts[2], cn[u]);
            }
        }
        for (long u = 0; u < H; ++u) { h[u] = hn[u]; c[u] = cn[u]; }
        if (a->Y) {
            float* y = a->Y + o_yidx(a, t, d, n);
            for (long u = 0; u < H; ++u) y[u] = o_canon(h[u]);
        }
    }
    if (a->Y) {
        for (long t = L; t < a->S; ++t) {
            float* y = a->Y + o_yidx(a, t, d, n);
            for (long u = 0; u < H; ++u) y[u] = 0.0f;
        }
    }
    if (a->Yh) {
        float* yh = a->Yh + o_sidx(a, d, n);
        for (long u = 0; u < H; ++u) yh[u] = L > 0 ? o_canon(h[u]) : 0.0f;
    }
    if (a->Yc && a->op == 2) {
        float* yc = a->Yc + o_sidx(a, d, n);
        for (long u = 0; u < H; ++u) yc[u] = L > 0 ? o_canon(c[u]) : 0.0f;
    }
}

/* The whole operator.  Arrays are dense, in the shapes of the operator's
 * inputs and outputs for the given layout; B, lens, h0, c0, P, Y, Yh, Yc may
 * be NULL (absent).  Rows n_begin..n_end-1 of the batch are computed (the
 * rows of a batch are independent; the full range gives the whole result). */
int oracle_rnn_rows(int op, int direction, long hidden_size, long input_size,
                    const char* const* acts, int n_acts,
                    const float* alpha, int n_alpha, const float* beta, int n_beta,
                    float clip, int layout, int lbr, int input_forget,
                    long seq, long batch,
                    const float* X, const float* W, const float* R, const float* B,
                    const int32_t* lens, const float* h0, const float* c0, const float* P,
                    float* Y, float* Yh, float* Yc, long n_begin, long n_end)
{
    if (op < 0 || op > 2 || direction < 0 || direction > 2) return 1;
    if (hidden_size <= 0 || input_size < 0 || seq < 0 || batch < 0) return 1;
    if (layout != 0 && layout != 1) return 1;
    if (lbr != 0 && lbr != 1) return 1;
    if (input_forget != 0 && input_forget != 1) return 1;
    if (n_begin < 0 || n_end > batch || n_begin > n_end) return 1;

    OArgs a;
    a.op = op;
    a.dirs = direction == 2 ? 2 : 1;
    a.G = o_gates(op);
    a.layout = layout;
    a.lbr = op == 1 ? lbr : 0;
    a.input_forget = op == 2 ? input_forget : 0;
    a.has_clip = clip > 0.0f;     /* absent (NaN) or non-positive: no clip */
    a.clip = clip;
    a.S = seq; a.N = batch; a.I = input_size; a.H = hidden_size;
    a.X = X; a.W = W; a.R = R; a.B = B; a.lens = lens;
    a.h0 = h0; a.c0 = op == 2 ? c0 : NULL; a.P = op == 2 ? P : NULL;
    a.Y = Y; a.Yh = Yh; a.Yc = Yc;

    int fn[6]; float al[6]; float be[6];
    if (oracle_resolve_activations(op, direction, acts, n_acts, alpha, n_alpha,
                                   beta, n_beta, fn, al, be) != 0)
        return 1;

    /* zero-size: nothing runs; final states are the initial states or 0 */
    if (seq == 0 || batch == 0) {
        for (long d = 0; d < a.dirs; ++d)
            for (long n = n_begin; n < n_end; ++n)
                for (long u = 0; u < a.H; ++u) {
                    long i = o_sidx(&a, d, n) + u;
                    if (Yh) Yh[i] = h0 ? h0[i] : 0.0f;
                    if (Yc && op == 2) Yc[i] = a.c0 ? a.c0[i] : 0.0f;
                }
        return 0;
    }

    if (lens) {
        for (long n = 0; n < batch; ++n)
            if (lens[n] < 0 || (long)lens[n] > seq) return 2;
    }

    float* buf = (float*)malloc(sizeof(float) * (size_t)(7 * a.H + a.G * a.H));
    if (!buf) return 1;
    for (long d = 0; d < a.dirs; ++d) {
        int reverse = direction == 1 || (direction == 2 && d == 1);
        OAct da[3];
        for (int s = 0; s < 3; ++s) {
            da[s].fn = fn[d * 3 + s];
            da[s].alpha = al[d * 3 + s];
            da[s].beta = be[d * 3 + s];
        }
        for (long n = n_begin; n < n_end; ++n) o_run_row(&a, d, n, reverse, da, buf);
    }
    free(buf);
    return 0;
}

int oracle_rnn(int op, int direction, long hidden_size, long input_size,
               const char* const* acts, int n_acts,
               const float* alpha, int n_alpha, const float* beta, int n_beta,
               float clip, int layout, int lbr, int input_forget,
               long seq, long batch,
               const float* X, const float* W, const float* R, const float* B,
               const int32_t* lens, const float* h0, const float* c0, const float* P,
               float* Y, float* Yh, float* Yc)
{
    return oracle_rnn_rows(op, direction, hidden_size, input_size, acts, n_acts,
                           alpha, n_alpha, beta, n_beta, clip, layout, lbr,
                           input_forget, seq, batch, X, W, R, B, lens, h0, c0, P,
                           Y, Yh, Yc, 0, batch);
}

/* ------------------------------------------------------------ single cell */

/* One RNN cell (page "RNNCell", RNNCell-3: Detailed description, Attributes,
 * Inputs, Outputs): Ho = f(X.W^T + H.R^T + B), where B is the sum of the
 * input and recurrence biases, given once, and clip (when not +infinity, its
 * default) clamps f's input to [-clip, clip].  The page fixes no rounding
 * order; this follows the sequence operator's: each product with one
 * accumulator, k increasing from +0, then pre = (xw + rec) + B.
 * X [batch, I], H [batch, hidden], W [hidden, I], R [hidden, hidden],
 * B [hidden], Ho [batch, hidden]; f is relu, sigmoid or tanh (any case,
 * NULL = tanh); clip must be positive (NaN, 0 and negative values are
 * invalid).  Every NaN written to Ho is 0x7FC00000.  All arrays are
 * required.  Returns 0, or 1 for an invalid argument. */
int oracle_rnn_cell(long hidden_size, long input_size, const char* activation, float clip,
                    long batch, const float* X, const float* Hprev, const float* W,
                    const float* R, const float* B, float* Ho)
{
    if (hidden_size <= 0 || input_size < 0 || batch < 0) return 1;
    int fn = activation ? o_name_to_fn(activation) : OA_TANH;
    if (fn != OA_RELU && fn != OA_SIGMOID && fn != OA_TANH) return 1;
    if (!(clip > 0.0f)) return 1;
    if (batch > 0 && (!Hprev || !W || !R || !B || !Ho || (input_size > 0 && !X))) return 1;
    const long H = hidden_size, I = input_size;
    for (long n = 0; n < batch; ++n) {
        for (long j = 0; j < H; ++j) {
            float xw = o_dot(X + n * I, W + j * I, I);
            float rec = o_dot(Hprev + n * H, R + j * H, H);
            float pre = (xw + rec) + B[j];
            if (pre > clip) pre = clip;
            else if (pre < -clip) pre = -clip;
            Ho[n * H + j] = o_canon(oracle_activation(fn, 0.0f, 0.0f, pre));
        }
    }
    return 0;
}

/* Array forms of the transcendental and activation functions, for tests. */
void oracle_exp_n(const float* x, float* y, long n) { for (long i = 0; i < n; ++i) y[i] = oracle_exp(x[i]); }
void oracle_log_n(const float* x, float* y, long n) { for (long i = 0; i < n; ++i) y[i] = oracle_log(x[i]); }
void oracle_tanh_n(const float* x, float* y, long n) { for (long i = 0; i < n; ++i) y[i] = oracle_tanh(x[i]); }
void oracle_sigmoid_n(const float* x, float* y, long n) { for (long i = 0; i < n; ++i) y[i] = oracle_sigmoid(x[i]); }
void oracle_activation_n(int fn, float alpha, float beta, const float* x, float* y, long n)
{
    for (long i = 0; i < n; ++i) y[i] = oracle_activation(fn, alpha, beta, x[i]);
}
