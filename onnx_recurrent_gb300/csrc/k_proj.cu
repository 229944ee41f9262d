// Input projection XW = X . W^T for every time step at once (page "Recurrent
// operators: RNN, GRU, LSTM", Computation: one matrix product of shape
// [seq*batch, G*H] per direction, one accumulator per output, increasing k
// from +0).
//
// SIMT register-tiled GEMM: C[M][ncols] = A[M][K] . Bt[K][ncols], with A the
// input rows (row-major, K contiguous), Bt the packed transposed weights of
// all directions side by side, C the projection scratch.  A 128x128 output
// tile per CTA of 256 threads, each thread an 8x8 register tile (two 4x4
// quadrants 64 apart, so shared-memory reads are conflict-free float4s),
// k-tiles of 8 double-buffered through shared memory with the next tile held
// in registers while the current one is consumed.  Each accumulator walks k
// in increasing order.  Exact mode multiplies and adds with separate
// roundings; fast mode uses fused multiply-add.  Out-of-range rows, columns
// and k are read as +0: adding +0*+0 never changes an accumulator that
// started at +0 (round-to-nearest cannot produce -0 from +0), so the padding
// is invisible in the result.
#include "exact_math.cuh"
#include "rnn_internal.h"

namespace rnngb {

namespace {

constexpr int BM = 128, BN = 128, BK = 8;

template <bool EXACT, bool VEC>
__global__ void __launch_bounds__(256, 2)
proj_gemm_kernel(const float* __restrict__ A, const float* __restrict__ Bt, float* __restrict__ C,
                 int64_t M, int64_t K, int64_t NC)
{
    __shared__ __align__(16) float As[2][BK][BM];
    __shared__ __align__(16) float Bs[2][BK][BN];

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int64_t m0 = (int64_t)blockIdx.y * BM;
    const int64_t n0 = (int64_t)blockIdx.x * BN;

    // global -> register mapping
    const int a_row = tid >> 1, a_kq = (tid & 1) * 4;   // A: 128 rows x 8 k
    const int b_k = tid >> 5, b_c = (tid & 31) * 4;     // B: 8 k x 128 cols

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    float ar[4], br[4];
    auto gload = [&](int64_t k0) {
        const int64_t m = m0 + a_row;
        const int64_t ka = k0 + a_kq;
        if (VEC && m < M && ka + 3 < K) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(A + m * K + ka));
            ar[0] = v.x; ar[1] = v.y; ar[2] = v.z; ar[3] = v.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) ar[q] = (m < M && ka + q < K) ? __ldg(A + m * K + ka + q) : 0.0f;
        }
        const int64_t kb = k0 + b_k;
        const int64_t nb = n0 + b_c;
        if (VEC && kb < K && nb + 3 < NC) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(Bt + kb * NC + nb));
            br[0] = v.x; br[1] = v.y; br[2] = v.z; br[3] = v.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) br[q] = (kb < K && nb + q < NC) ? __ldg(Bt + kb * NC + nb + q) : 0.0f;
        }
    };
    auto sstore = [&](int buf) {
#pragma unroll
        for (int q = 0; q < 4; ++q) As[buf][a_kq + q][a_row] = ar[q];
        *reinterpret_cast<float4*>(&Bs[buf][b_k][b_c]) = make_float4(br[0], br[1], br[2], br[3]);
    };

    const int64_t ntiles = (K + BK - 1) / BK;
    if (ntiles > 0) {
        gload(0);
        sstore(0);
    }
    __syncthreads();
    for (int64_t t = 0; t < ntiles; ++t) {
        const int buf = (int)(t & 1);
        if (t + 1 < ntiles) gload((t + 1) * BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4 + 64]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    acc[i][j] = EXACT ? fadd(acc[i][j], fmul(a[i], b[j])) : __fmaf_rn(a[i], b[j], acc[i][j]);
        }
        if (t + 1 < ntiles) sstore(buf ^ 1);
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= M) continue;
        float* crow = C + m * NC;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + h * 64 + tx * 4;
            if (VEC && n + 3 < NC) {
                *reinterpret_cast<float4*>(crow + n) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (n + q < NC) crow[n + q] = acc[i][4 * h + q];
            }
        }
    }
}

}  // namespace

cudaError_t launch_projection(const float* X, const float* Bt, float* XW, int64_t M, int64_t K,
                              int64_t ncols, bool exact, cudaStream_t stream)
{
    if (M <= 0 || ncols <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((ncols + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    const bool vec = (K % 4 == 0) && (ncols % 4 == 0) && ((uintptr_t)X % 16 == 0) &&
                     ((uintptr_t)Bt % 16 == 0) && ((uintptr_t)XW % 16 == 0);
    if (exact) {
        if (vec) proj_gemm_kernel<true, true><<<grid, 256, 0, stream>>>(X, Bt, XW, M, K, ncols);
        else proj_gemm_kernel<true, false><<<grid, 256, 0, stream>>>(X, Bt, XW, M, K, ncols);
    } else {
        if (vec) proj_gemm_kernel<false, true><<<grid, 256, 0, stream>>>(X, Bt, XW, M, K, ncols);
        else proj_gemm_kernel<false, false><<<grid, 256, 0, stream>>>(X, Bt, XW, M, K, ncols);
    }
    return cudaGetLastError();
}

}  // namespace rnngb
