// Single RNN cell, one fused kernel (page "RNNCell", RNNCell-3: Detailed
// description, Attributes, Inputs, Outputs):
//     Ho[n, j] = f(clip((xw + rec) + B[j]))
//     xw  = sum_k X[n, k] * W[j, k]    k = 0 .. I-1, one accumulator from +0
//     rec = sum_k H[n, k] * R[j, k]    k = 0 .. H-1, one accumulator from +0
// in the sequence operator's rounding order (exact mode: every product and
// sum rounded separately; fast mode: fused multiply-add, same order).
//
// The cells of a call are independent, so there is no recurrence and no
// barrier: an output tile per CTA (32 rows x 64 units, 128 threads, 4 x 4
// outputs per thread), both operands staged through shared memory in
// k-major chunks of 16 by asynchronous copies, five chunks in flight ahead
// of the one being multiplied.  Entries past I, H, the batch or the units are
// staged as zeros on both sides: the extra products are 0 * 0 = +0, and an
// accumulator that starts at +0 is never -0, so adding them changes no bit.
#include "exact_math.cuh"
#include "rnn_internal.h"

namespace rnngb {
namespace {

constexpr int CT_M = 32;    // batch rows per CTA
constexpr int CT_N = 64;    // units per CTA
constexpr int CT_K = 16;    // k chunk
constexpr int CT_RM = 4;    // rows per thread (and 4 units)
constexpr int CT_THREADS = (CT_M / CT_RM) * (CT_N / 4);

template <bool EXACT>
__device__ __forceinline__ float mac(float acc, float a, float b)
{
    return EXACT ? fadd(acc, fmul(a, b)) : __fmaf_rn(a, b, acc);
}

constexpr int CT_STAGES = 6;   // k chunks in flight
static_assert(CT_RM == 4 && CT_N / 4 == 16, "thread layout: ty = t / 16, tx = t % 16; 4 rows per thread");

__device__ __forceinline__ void cp4(float* dst, const float* src, bool valid)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

struct CellStage {
    float a[CT_K][CT_M];
    float b[CT_K][CT_N + 4];
};

// Stage chunk `c` of the k sequence (the I chunks of X.W^T, then the H
// chunks of H.R^T) into `st`, transposed to k-major: A rows n0.., B rows j0..
// (both row-major, k contiguous).  Out-of-range entries are zero-filled.
__device__ __forceinline__ void cell_issue(CellStage& st, int64_t c, int64_t nI, const float* X, const float* W,
                                           const float* Hp, const float* R, int64_t N, int64_t U, int64_t I,
                                           int64_t H, int64_t n0, int64_t j0)
{
    const bool first = c < nI;
    const float* A = first ? X : Hp;
    const float* Bm = first ? W : R;
    const int64_t K = first ? I : H;
    const int64_t k0 = (first ? c : c - nI) * CT_K;
    const int t = threadIdx.x;
    constexpr int AK = CT_M * CT_K / CT_THREADS, BK = CT_N * CT_K / CT_THREADS;
    const int ar = t / (CT_K / AK), ak = (t % (CT_K / AK)) * AK;     // A: AK consecutive k of one row
    const int bu = t / (CT_K / BK), bk = (t % (CT_K / BK)) * BK;     // B: BK consecutive k of one unit
    const int64_t an = n0 + ar, bj = j0 + bu;
#pragma unroll
    for (int i = 0; i < AK; ++i) {
        const int64_t k = k0 + ak + i;
        const bool v = an < N && k < K;
        cp4(&st.a[ak + i][ar], v ? A + an * K + k : A, v);
    }
#pragma unroll
    for (int i = 0; i < BK; ++i) {
        const int64_t k = k0 + bk + i;
        const bool v = bj < U && k < K;
        cp4(&st.b[bk + i][bu], v ? Bm + bj * K + k : Bm, v);
    }
}

template <bool EXACT>
__device__ __forceinline__ void cell_chunk(const CellStage& st, float (&acc)[CT_RM][4])
{
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int kk = 0; kk < CT_K; ++kk) {
        const float4 a = *reinterpret_cast<const float4*>(&st.a[kk][ty * CT_RM]);
        const float4 b = *reinterpret_cast<const float4*>(&st.b[kk][tx * 4]);
        const float av[CT_RM] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int r = 0; r < CT_RM; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = mac<EXACT>(acc[r][c], av[r], bv[c]);
    }
}

template <bool EXACT, int FN>
__device__ __forceinline__ float cell_act(float v)
{
    if constexpr (FN == 0) return v < 0.0f ? 0.0f : v;                       // Relu
    else if constexpr (FN == 1) return EXACT ? dx_tanh(v) : df_tanh(v);      // Tanh
    else return EXACT ? dx_sigmoid(v) : df_sigmoid(v);                       // Sigmoid
}

template <bool EXACT, int FN>
__global__ void __launch_bounds__(CT_THREADS) rnn_cell_kernel(const float* __restrict__ X,
                                                              const float* __restrict__ Hp,
                                                              const float* __restrict__ W,
                                                              const float* __restrict__ R,
                                                              const float* __restrict__ B, float* __restrict__ Ho,
                                                              int64_t N, int64_t I, int64_t H, int has_clip,
                                                              float clip)
{
    __shared__ __align__(16) CellStage ring[CT_STAGES];
    const int64_t j0 = (int64_t)blockIdx.x * CT_N, n0 = (int64_t)blockIdx.y * CT_M;
    float xw[CT_RM][4], rec[CT_RM][4];
#pragma unroll
    for (int r = 0; r < CT_RM; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) xw[r][c] = rec[r][c] = 0.0f;
    // one k sequence: X.W^T's chunks, then H.R^T's, CT_STAGES - 1 in flight
    const int64_t nI = (I + CT_K - 1) / CT_K, nC = nI + (H + CT_K - 1) / CT_K;
#pragma unroll
    for (int s = 0; s < CT_STAGES - 1; ++s) {
        if (s < nC) cell_issue(ring[s], s, nI, X, W, Hp, R, N, H, I, H, n0, j0);
        cp_commit();
    }
    for (int64_t c = 0; c < nC; ++c) {
        cp_wait<CT_STAGES - 2>();     // chunk c has landed (this thread's copies)
        __syncthreads();              // everyone's copies; and chunk c-1's slot is free
        const int64_t nx = c + CT_STAGES - 1;
        if (nx < nC) cell_issue(ring[nx % CT_STAGES], nx, nI, X, W, Hp, R, N, H, I, H, n0, j0);
        cp_commit();
        if (c < nI) cell_chunk<EXACT>(ring[c % CT_STAGES], xw);
        else cell_chunk<EXACT>(ring[c % CT_STAGES], rec);
    }
    cp_wait<0>();

    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int r = 0; r < CT_RM; ++r) {
        const int64_t n = n0 + ty * CT_RM + r;
        if (n >= N) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t j = j0 + tx * 4 + c;
            if (j >= H) continue;
            float pre = fadd(fadd(xw[r][c], rec[r][c]), B[j]);
            if (has_clip) pre = pre > clip ? clip : (pre < -clip ? -clip : pre);   // a NaN passes
            Ho[n * H + j] = canon_nan(cell_act<EXACT, FN>(pre));
        }
    }
}

template <bool EXACT>
cudaError_t launch_cell_fn(int fn, dim3 grid, const float* X, const float* Hp, const float* W, const float* R,
                           const float* B, float* Ho, int64_t N, int64_t I, int64_t H, int has_clip, float clip,
                           cudaStream_t s)
{
    if (fn == 0) rnn_cell_kernel<EXACT, 0><<<grid, CT_THREADS, 0, s>>>(X, Hp, W, R, B, Ho, N, I, H, has_clip, clip);
    else if (fn == 1) rnn_cell_kernel<EXACT, 1><<<grid, CT_THREADS, 0, s>>>(X, Hp, W, R, B, Ho, N, I, H, has_clip, clip);
    else rnn_cell_kernel<EXACT, 2><<<grid, CT_THREADS, 0, s>>>(X, Hp, W, R, B, Ho, N, I, H, has_clip, clip);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cell(const float* X, const float* Hp, const float* W, const float* R, const float* B, float* Ho,
                        int64_t N, int64_t I, int64_t H, int fn, int has_clip, float clip, bool exact,
                        cudaStream_t stream)
{
    if (N <= 0) return cudaSuccess;
    if (fn < 0 || fn > 2) return cudaErrorInvalidValue;
    const int64_t gx = (H + CT_N - 1) / CT_N, gy = (N + CT_M - 1) / CT_M;
    if (gx > 0x7fffffff || gy > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)gx, (unsigned)gy);
    return exact ? launch_cell_fn<true>(fn, grid, X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, stream)
                 : launch_cell_fn<false>(fn, grid, X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, stream);
}

}  // namespace rnngb
