// Single RNN cell, one fused kernel (page "RNNCell", RNNCell-3: Detailed
// description, Attributes, Inputs, Outputs):
//     Ho[n, j] = f(clip((xw + rec) + B[j]))
//     xw  = sum_k X[n, k] * W[j, k]    k = 0 .. I-1, one accumulator from +0
//     rec = sum_k H[n, k] * R[j, k]    k = 0 .. H-1, one accumulator from +0
// in the sequence operator's rounding order (exact mode: every product and
// sum rounded separately; fast mode: fused multiply-add, same order).
//
// The cells of a call are independent, so there is no recurrence and no
// barrier: an output tile per CTA (32 rows x 64 units, 128 threads, 4 rows x
// 4 units per thread), both operands staged through shared memory in chunks
// of 16 k by asynchronous copies (16-byte copies where rows are aligned),
// five chunks in flight ahead of the one being multiplied.  Entries past I, H, the batch or the units are
// staged as zeros on both sides: the extra products are 0 * 0 = +0, and an
// accumulator that starts at +0 is never -0, so adding them changes no bit.
#include "exact_math.cuh"
#include "rnn_internal.h"

namespace rnngb {
namespace {

constexpr int CT_M = 32;    // batch rows per CTA
constexpr int CT_N = 64;    // units per CTA
constexpr int CT_K = 16;    // k chunk: four 16-byte pieces per row
constexpr int CT_THREADS = 128;
constexpr int CT_STAGES = 6;   // k chunks in flight
// thread t: rows ty*4 .. ty*4+3 (ty = t / 16), units tx + 16c, c = 0..3 (tx = t % 16)

template <bool EXACT>
__device__ __forceinline__ float mac(float acc, float a, float b)
{
    return EXACT ? fadd(acc, fmul(a, b)) : __fmaf_rn(a, b, acc);
}

// Rows are stored row-major, 16 floats each, with the four 16-byte pieces of
// row r permuted by r's bits 1-2: eight consecutive rows then cover all 32
// banks for any one piece, so the 16-byte reads of the k loop and the
// 16-byte copies that fill a stage are free of bank conflicts.
__device__ __forceinline__ int piece_at(int row, int piece) { return (piece ^ ((row >> 1) & 3)) * 4; }

struct CellStage {
    float a[CT_M][CT_K];
    float b[CT_N][CT_K];
};

__device__ __forceinline__ void cp16(float* dst, const float* src, int bytes)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(d), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp4(float* dst, const float* src, bool valid)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(d), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// One 16-byte piece (k0 + 4p .. +3) of row `row` of a [rows, K] matrix into
// dst; past the last row or K it is zero-filled.  vec: K % 4 == 0 and the
// matrix 16-byte aligned, so a row's pieces are aligned 16-byte copies.
__device__ __forceinline__ void stage_piece(float* dst, const float* M, int64_t row, int64_t rows, int64_t K,
                                            int64_t k, bool vec)
{
    if (vec) {
        const int64_t left = (row < rows) ? K - k : 0;
        const int bytes = left >= 4 ? 16 : (left > 0 ? (int)left * 4 : 0);
        cp16(dst, bytes ? M + row * K + k : M, bytes);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const bool v = row < rows && k + e < K;
            cp4(dst + e, v ? M + row * K + k + e : M, v);
        }
    }
}

// Stage chunk `c` of the k sequence (the chunks of X.W^T, then those of
// H.R^T): A rows n0 .. n0+31 (one piece per thread), B rows j0 .. j0+63 (two).
__device__ __forceinline__ void cell_issue(CellStage& st, int64_t c, int64_t nI, const float* X, const float* W,
                                           const float* Hp, const float* R, int64_t N, int64_t U, int64_t I,
                                           int64_t H, int64_t n0, int64_t j0, bool vec_x, bool vec_h)
{
    const bool first = c < nI;
    const float* A = first ? X : Hp;
    const float* Bm = first ? W : R;
    const int64_t K = first ? I : H;
    const bool vec = first ? vec_x : vec_h;
    const int64_t k0 = (first ? c : c - nI) * CT_K;
    const int t = threadIdx.x;
    const int r = t / 4, p = t % 4;
    const int64_t k = k0 + 4 * p;
    stage_piece(&st.a[r][piece_at(r, p)], A, n0 + r, N, K, k, vec);
    stage_piece(&st.b[r][piece_at(r, p)], Bm, j0 + r, U, K, k, vec);
    stage_piece(&st.b[r + 32][piece_at(r + 32, p)], Bm, j0 + r + 32, U, K, k, vec);
}

template <bool EXACT>
__device__ __forceinline__ void cell_chunk(const CellStage& st, float (&acc)[4][4])
{
    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float4 a[4], b[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = ty * 4 + r;
            a[r] = *reinterpret_cast<const float4*>(&st.a[row][piece_at(row, p)]);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int u = tx + 16 * c;
            b[c] = *reinterpret_cast<const float4*>(&st.b[u][piece_at(u, p)]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float av = e == 0 ? a[r].x : e == 1 ? a[r].y : e == 2 ? a[r].z : a[r].w;
                    const float bv = e == 0 ? b[c].x : e == 1 ? b[c].y : e == 2 ? b[c].z : b[c].w;
                    acc[r][c] = mac<EXACT>(acc[r][c], av, bv);
                }
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
                                                              float clip, int vec_x, int vec_h)
{
    __shared__ __align__(16) CellStage ring[CT_STAGES];
    const int64_t j0 = (int64_t)blockIdx.x * CT_N, n0 = (int64_t)blockIdx.y * CT_M;
    float xw[4][4], rec[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) xw[r][c] = rec[r][c] = 0.0f;
    // one k sequence: X.W^T's chunks, then H.R^T's, CT_STAGES - 1 in flight
    const int64_t nI = (I + CT_K - 1) / CT_K, nC = nI + (H + CT_K - 1) / CT_K;
#pragma unroll
    for (int s = 0; s < CT_STAGES - 1; ++s) {
        if (s < nC) cell_issue(ring[s], s, nI, X, W, Hp, R, N, H, I, H, n0, j0, vec_x, vec_h);
        cp_commit();
    }
    for (int64_t c = 0; c < nC; ++c) {
        cp_wait<CT_STAGES - 2>();     // chunk c has landed (this thread's copies)
        __syncthreads();              // everyone's copies; and chunk c-1's slot is free
        const int64_t nx = c + CT_STAGES - 1;
        if (nx < nC) cell_issue(ring[nx % CT_STAGES], nx, nI, X, W, Hp, R, N, H, I, H, n0, j0, vec_x, vec_h);
        cp_commit();
        if (c < nI) cell_chunk<EXACT>(ring[c % CT_STAGES], xw);
        else cell_chunk<EXACT>(ring[c % CT_STAGES], rec);
    }
    cp_wait<0>();

    const int ty = threadIdx.x / 16, tx = threadIdx.x % 16;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t n = n0 + ty * 4 + r;
        if (n >= N) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t j = j0 + tx + 16 * c;
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
                           int vx, int vh, cudaStream_t s)
{
    if (fn == 0)
        rnn_cell_kernel<EXACT, 0><<<grid, CT_THREADS, 0, s>>>(X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, vx, vh);
    else if (fn == 1)
        rnn_cell_kernel<EXACT, 1><<<grid, CT_THREADS, 0, s>>>(X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, vx, vh);
    else
        rnn_cell_kernel<EXACT, 2><<<grid, CT_THREADS, 0, s>>>(X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, vx, vh);
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
    auto a16 = [](const void* p) { return ((uintptr_t)p & 15) == 0; };
    const int vx = I % 4 == 0 && a16(X) && a16(W);     // 16-byte copies of X and W rows
    const int vh = H % 4 == 0 && a16(Hp) && a16(R);
    return exact ? launch_cell_fn<true>(fn, grid, X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, vx, vh, stream)
                 : launch_cell_fn<false>(fn, grid, X, Hp, W, R, B, Ho, N, I, H, has_clip, clip, vx, vh, stream);
}

}  // namespace rnngb
