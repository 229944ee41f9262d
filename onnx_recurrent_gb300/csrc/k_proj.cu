// Input projection XW = X . W^T for every time step at once (page "Recurrent
// operators: RNN, GRU, LSTM", Computation: one matrix product of shape
// [seq*batch, G*H] per direction, one accumulator per output, increasing k
// from +0).
//
// SIMT register-tiled GEMM: C[M][ncols] = A[M][K] . Bt[K][ncols], with A the
// input rows (row-major, K contiguous), Bt the packed transposed weights of
// all directions side by side, C the projection scratch.  A 128x128 output
// tile per CTA of 256 threads, each thread an 8x8 register tile (two 4x4
// quadrants 64 apart, so shared-memory reads are conflict-free float4s).
// Each accumulator walks k in increasing order.  Exact mode multiplies and
// adds with separate roundings; fast mode uses fused multiply-add.
// Out-of-range rows, columns and k are read as +0: adding +0*+0 never
// changes an accumulator that started at +0 (round-to-nearest cannot produce
// -0 from +0), so the padding is invisible in the result.
//
// Two loaders feed the same arithmetic:
//   * tensor copies (TMA): the A tile [128 rows][TK k] and the Bt tile
//     [TK k][128 cols] of each k-step are each one cp.async.bulk.tensor.2d
//     copy into a ring (fast mode 32 k x 3 stages, exact 16 k x 4),
//     completing on the stage's mbarrier; the
//     threads read A row-major (the 8 threads of a quarter warp share their
//     rows, so each 16-byte read is a broadcast).  Used when rows of A and Bt
//     are 16-byte aligned.
//   * register staging: k-tiles of 8 double-buffered through shared memory,
//     the next tile held in registers while the current one is consumed.
//     Used for any alignment.
#include "exact_math.cuh"
#include "rnn_internal.h"
#include "tma.cuh"

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

// Ring shape per mode (measured on GB300): fast mode takes 32 k per stage in
// 3 stages (half the barriers per k; 4-5% faster than 16 k x 4), exact mode
// 16 k per stage in 4 stages (17% faster than 32 k x 3).
template <bool EXACT>
struct ProjRing {
    static constexpr int TK = EXACT ? 16 : 32;                          // k per stage
    static constexpr int STAGES = EXACT ? 4 : 3;
    static constexpr unsigned kTileBytes = (BM * TK + TK * BN) * 4;    // one stage: A tile + Bt tile
    static constexpr size_t kSmem = (size_t)STAGES * kTileBytes + 128;
};

struct ProjArgs {
    CUtensorMap amap;    // A [M][K]: dims {K, M}, box {TK, 128}
    CUtensorMap bmap;    // Bt [K][NC]: dims {NC, K}, box {128, TK}
    float* C;
    int64_t M, NC;
    int ntiles;          // k-steps of TK
    int* status;         // device status word (a wait that gives up writes RNN_ERR_TIMEOUT)
    long long limit_ns;
};

// Bounded wait for a ring stage (false once the limit has passed).
__device__ __forceinline__ bool stage_wait(uint64_t* bar, unsigned parity, long long limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    unsigned it = 0;
    while (!mbar_test(bar, parity)) {
        if ((++it & 255u) == 0u && (long long)(globaltimer_ns() - t0) > limit_ns) return false;
    }
    return true;
}

template <bool EXACT>
__global__ void __launch_bounds__(256, 2) proj_tma_kernel(const __grid_constant__ ProjArgs a)
{
    constexpr int TK = ProjRing<EXACT>::TK, TSTAGES = ProjRing<EXACT>::STAGES;
    constexpr unsigned kTileBytes = ProjRing<EXACT>::kTileBytes;
    extern __shared__ __align__(128) unsigned char proj_smem[];
    __shared__ __align__(8) uint64_t full[TSTAGES];
    unsigned char* base = proj_smem + ((128u - (smem_addr(proj_smem) & 127u)) & 127u);

    const int tid = threadIdx.x;
    const int tx = tid & 15, ty = tid >> 4;
    const int m0 = (int)blockIdx.y * BM;
    const int n0 = (int)blockIdx.x * BN;

    if (tid == 0) {
        for (int i = 0; i < TSTAGES; ++i) mbar_init(&full[i], 1);
        mbar_fence_init();
    }
    __syncthreads();
    auto issue = [&](int t) {
        const int st = t % TSTAGES;
        float* as = reinterpret_cast<float*>(base + (size_t)st * kTileBytes);
        float* bs = as + BM * TK;
        mbar_arrive_expect_tx(&full[st], kTileBytes);
        tma_load_2d(as, &a.amap, t * TK, m0, &full[st]);
        tma_load_2d(bs, &a.bmap, n0, t * TK, &full[st]);
    };
    if (tid == 0)
        for (int t = 0; t < TSTAGES && t < a.ntiles; ++t) issue(t);

    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    int issued = min(TSTAGES, a.ntiles);
    bool ok = true;
    for (int t = 0; t < a.ntiles; ++t) {
        const int st = t % TSTAGES;
        ok = stage_wait(&full[st], (unsigned)(t / TSTAGES) & 1u, a.limit_ns);
        if (__syncthreads_or(!ok)) {
            ok = false;
            break;
        }
        const float* as = reinterpret_cast<const float*>(base + (size_t)st * kTileBytes);
        const float* bs = as + BM * TK;
#pragma unroll
        for (int kq = 0; kq < TK; kq += 4) {
            float4 av[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int row = i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4);
                av[i] = *reinterpret_cast<const float4*>(as + row * TK + kq);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 b0 = *reinterpret_cast<const float4*>(bs + (kq + k) * BN + tx * 4);
                const float4 b1 = *reinterpret_cast<const float4*>(bs + (kq + k) * BN + 64 + tx * 4);
                const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float ai = k == 0 ? av[i].x : (k == 1 ? av[i].y : (k == 2 ? av[i].z : av[i].w));
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[i][j] = EXACT ? fadd(acc[i][j], fmul(ai, b[j])) : __fmaf_rn(ai, b[j], acc[i][j]);
                }
            }
        }
        __syncthreads();   // every thread is done with stage st
        if (tid == 0 && t + TSTAGES < a.ntiles) {
            issue(t + TSTAGES);
            ++issued;
        }
    }
    if (!ok) {
        // record the failure, then wait (bounded) for this CTA's copies in
        // flight before the shared memory they target is released
        if (tid == 0) {
            atomicCAS(a.status, 0, 6 /* RNN_ERR_TIMEOUT */);
            for (int t = max(0, issued - TSTAGES); t < issued; ++t)
                (void)stage_wait(&full[t % TSTAGES], (unsigned)(t / TSTAGES) & 1u, a.limit_ns);
        }
        return;
    }

#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t m = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
        if (m >= a.M) continue;
        float* crow = a.C + m * a.NC;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = n0 + h * 64 + tx * 4;
            if (n + 3 < a.NC) {
                *reinterpret_cast<float4*>(crow + n) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (n + q < a.NC) crow[n + q] = acc[i][4 * h + q];
            }
        }
    }
}

}  // namespace

cudaError_t launch_projection(const float* X, const float* Bt, float* XW, int64_t M, int64_t K,
                              int64_t ncols, bool exact, int* status, long long limit_ns, cudaStream_t stream)
{
    if (M <= 0 || ncols <= 0) return cudaSuccess;
    const dim3 grid((unsigned)((ncols + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    if (grid.y > 65535u) return cudaErrorInvalidConfiguration;
    const bool vec = (K % 4 == 0) && (ncols % 4 == 0) && ((uintptr_t)X % 16 == 0) &&
                     ((uintptr_t)Bt % 16 == 0) && ((uintptr_t)XW % 16 == 0);
    if (vec && K > 0 && M < (1ll << 31) && ncols < (1ll << 31) && K < (1ll << 31)) {
        ProjArgs pa;
        const int TK = exact ? ProjRing<true>::TK : ProjRing<false>::TK;
        const size_t smem = exact ? ProjRing<true>::kSmem : ProjRing<false>::kSmem;
        const cuuint64_t adims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t astr[1] = {(cuuint64_t)K * 4};
        const cuuint32_t abox[2] = {(cuuint32_t)TK, (cuuint32_t)BM};
        const cuuint64_t bdims[2] = {(cuuint64_t)ncols, (cuuint64_t)K};
        const cuuint64_t bstr[1] = {(cuuint64_t)ncols * 4};
        const cuuint32_t bbox[2] = {(cuuint32_t)BN, (cuuint32_t)TK};
        if (encode_tensor_map(&pa.amap, X, 2, adims, astr, abox) &&
            encode_tensor_map(&pa.bmap, Bt, 2, bdims, bstr, bbox)) {
            pa.C = XW;
            pa.M = M;
            pa.NC = ncols;
            pa.ntiles = (int)((K + TK - 1) / TK);
            pa.status = status;
            pa.limit_ns = limit_ns;
            const void* fn = exact ? (const void*)proj_tma_kernel<true> : (const void*)proj_tma_kernel<false>;
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            if (exact) proj_tma_kernel<true><<<grid, 256, smem, stream>>>(pa);
            else proj_tma_kernel<false><<<grid, 256, smem, stream>>>(pa);
            return cudaGetLastError();
        }
    }
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
