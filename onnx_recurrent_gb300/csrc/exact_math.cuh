// Device activation functions.
//
// Exact mode (page "Recurrent operators: RNN, GRU, LSTM", Activations and
// Exact mode): every function is built from IEEE-rounded +, -, *, / (the
// __f*_rn intrinsics, which the compiler never contracts into FMA) and bit
// operations, so its result is the same on every machine that follows the
// same steps.  The steps are this library's own definition:
//   exp(x)   Cody-Waite reduction x = k*ln2 + r with ln2 split into a
//            15-significant-bit head and a tail, degree-7 Taylor polynomial of
//            e^r in Horner form, scaling by 2^k as two exact powers of two.
//   log(x)   x = m*2^e, m in [sqrt(1/2), sqrt(2)), s = (m-1)/(m+1),
//            log m = 2s + 2s*(z/3 + z^2/5 + z^3/7 + z^4/9 + z^5/11), z = s^2.
//   tanh(x)  |x| > 9.1: +-1; |x| < 0.4: odd Taylor series to x^13;
//            otherwise 1 - 2/(exp(2|x|) + 1); sign restored.
//   sigmoid  1 / (1 + exp(-x)).
// Fast mode (Fast mode section) uses CUDA's expf / tanhf / logf instead.
#pragma once

#include <cuda_runtime.h>

namespace rnngb {

__device__ __forceinline__ float fadd(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float fsub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float fmul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float fdiv(float a, float b) { return __fdiv_rn(a, b); }

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// The special cases are selected after the fact rather than branched to, so
// that independent calls can be interleaved; inside [-110, 89] the clamp is
// the identity and the result is the polynomial path's.
__device__ __forceinline__ float dx_exp(float x)
{
    const float xc = fminf(fmaxf(x, -110.0f), 89.0f);
    const float t = fmul(xc, 0x1.715476p+0f);                          // x / ln 2
    const float kf = fsub(fadd(t, 0x1.8p+23f), 0x1.8p+23f);            // round to integer
    const float r = fsub(fsub(xc, fmul(kf, 0x1.62e4p-1f)), fmul(kf, 0x1.7f7d1cp-20f));
    float p = 0x1.a01a02p-13f;                                         // 1/5040
    p = fadd(fmul(p, r), 0x1.6c16c2p-10f);                             // 1/720
    p = fadd(fmul(p, r), 0x1.111112p-7f);                              // 1/120
    p = fadd(fmul(p, r), 0x1.555556p-5f);                              // 1/24
    p = fadd(fmul(p, r), 0x1.555556p-3f);                              // 1/6
    p = fadd(fmul(p, r), 0.5f);
    p = fadd(fmul(p, r), 1.0f);
    p = fadd(fmul(p, r), 1.0f);
    const int k = (int)kf;
    const int k1 = k / 2;
    const int k2 = k - k1;
    float v = fmul(fmul(p, pow2i(k1)), pow2i(k2));
    v = x > 89.0f ? __int_as_float(0x7f800000) : v;
    v = x < -110.0f ? 0.0f : v;
    return x != x ? x : v;
}

__device__ __forceinline__ float dx_log(float x)
{
    if (x != x) return x;
    if (x < 0.0f) return __int_as_float(0x7fc00000);
    if (x == 0.0f) return __int_as_float(0xff800000);
    if (x == __int_as_float(0x7f800000)) return x;
    int eadj = 0;
    if (x < 0x1p-126f) {
        x = fmul(x, 0x1p+24f);
        eadj = -24;
    }
    const unsigned b = __float_as_uint(x);
    int e = (int)((b >> 23) & 0xffu) - 127 + eadj;
    float m = __uint_as_float((b & 0x007fffffu) | 0x3f800000u);
    if (m > 0x1.6a09e6p+0f) {                                          // sqrt(2)
        m = fmul(m, 0.5f);
        e += 1;
    }
    const float s = fdiv(fsub(m, 1.0f), fadd(m, 1.0f));
    const float z = fmul(s, s);
    float q = 0x1.745d18p-4f;                                          // 1/11
    q = fadd(fmul(q, z), 0x1.c71c72p-4f);                              // 1/9
    q = fadd(fmul(q, z), 0x1.24924ap-3f);                              // 1/7
    q = fadd(fmul(q, z), 0x1.99999ap-3f);                              // 1/5
    q = fadd(fmul(q, z), 0x1.555556p-2f);                              // 1/3
    const float w = fmul(q, z);
    const float s2 = fadd(s, s);
    const float lm = fadd(s2, fmul(s2, w));
    const float ef = (float)e;
    return fadd(fmul(ef, 0x1.62e4p-1f), fadd(lm, fmul(ef, 0x1.7f7d1cp-20f)));
}

// Both series are evaluated and the one for |x|'s range selected (no
// divergent branches); each range's value is the same expression as above.
__device__ __forceinline__ float dx_tanh(float x)
{
    const unsigned sign = __float_as_uint(x) & 0x80000000u;
    const float a = __uint_as_float(__float_as_uint(x) & 0x7fffffffu);
    const float z = fmul(a, a);
    float q = 0x1.d6d3d0p-9f;                                          // 21844/6081075
    q = fadd(fmul(q, z), -0x1.226e36p-7f);                             // -1382/155925
    q = fadd(fmul(q, z), 0x1.664f48p-6f);                              // 62/2835
    q = fadd(fmul(q, z), -0x1.ba1ba2p-5f);                             // -17/315
    q = fadd(fmul(q, z), 0x1.111112p-3f);                              // 2/15
    q = fadd(fmul(q, z), -0x1.555556p-2f);                             // -1/3
    const float ys = fadd(a, fmul(a, fmul(q, z)));                     // |x| < 0.4
    const float e = dx_exp(fadd(a, a));
    const float yl = fsub(1.0f, fdiv(2.0f, fadd(e, 1.0f)));            // 0.4 <= |x| <= 9.1
    const float y = a > 9.1f ? 1.0f : (a < 0.4f ? ys : yl);
    return x != x ? x : __uint_as_float(__float_as_uint(y) | sign);
}

__device__ __forceinline__ float dx_sigmoid(float x) { return fdiv(1.0f, fadd(1.0f, dx_exp(-x))); }

// Fast-mode transcendentals: CUDA's accurate (non-intrinsic) functions.
__device__ __forceinline__ float df_exp(float x) { return expf(x); }
__device__ __forceinline__ float df_log(float x) { return logf(x); }
__device__ __forceinline__ float df_tanh(float x) { return tanhf(x); }
__device__ __forceinline__ float df_sigmoid(float x) { return fdiv(1.0f, fadd(1.0f, expf(-x))); }

// One activation (ids as RNN_ACT_* in the public header).
template <bool EXACT>
__device__ __forceinline__ float activation(int fn, float alpha, float beta, float x)
{
    switch (fn) {
    case 0: return x < 0.0f ? 0.0f : x;                                         // Relu
    case 1: return EXACT ? dx_tanh(x) : df_tanh(x);                             // Tanh
    case 2: return EXACT ? dx_sigmoid(x) : df_sigmoid(x);                       // Sigmoid
    case 3: return fadd(fmul(alpha, x), beta);                                  // Affine
    case 4: return x < 0.0f ? fmul(alpha, x) : x;                               // LeakyRelu
    case 5: return x > alpha ? x : 0.0f;                                        // ThresholdedRelu
    case 6: return fmul(alpha, EXACT ? dx_tanh(fmul(beta, x)) : df_tanh(fmul(beta, x)));
    case 7: {                                                                   // HardSigmoid
        const float v = fadd(fmul(alpha, x), beta);
        return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);
    }
    case 8:                                                                     // Elu
        return x >= 0.0f ? x : fmul(alpha, fsub(EXACT ? dx_exp(x) : df_exp(x), 1.0f));
    case 9: return fdiv(x, fadd(1.0f, fabsf(x)));                               // Softsign
    case 10:                                                                    // Softplus
        return x > 20.0f ? x
                         : (EXACT ? dx_log(fadd(1.0f, dx_exp(x))) : df_log(fadd(1.0f, df_exp(x))));
    default: return __int_as_float(0x7fc00000);
    }
}

__device__ __forceinline__ float canon_nan(float v) { return v != v ? __int_as_float(0x7fc00000) : v; }

}  // namespace rnngb
