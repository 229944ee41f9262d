// Input projection on the tensor cores: XW[M][NC] = X[M][K] . Wk[NC][K]^T
// (page "Recurrent operators: RNN, GRU, LSTM", Computation: the projection
// of every step as one matrix product; Fast mode: the product need not keep
// the exact mode's rounding order).  Two operand kinds, sums in FP32 on the
// tensor cores:
//   * TF32: fp32 operands, products of their TF32 parts (10-bit mantissas),
//     tcgen05.mma kind::tf32, K 8 per instruction;
//   * BF16: operands converted to bf16 beforehand (round to nearest even),
//     tcgen05.mma kind::f16 with both A and B bf16, K 16 per instruction.
// Either way a k-block is 128 bytes of every row (32 fp32 or 64 bf16).
//
// One CTA per 128 x 128 output tile, 128 threads, two CTAs per SM (so one
// tile's read-out overlaps the other's MMAs):
//   * warp 0, one lane: tensor copies (TMA) of the A tile [128 rows][k-block]
//     and the Wk tile [128 cols][k-block] of each k-block into a 3-stage
//     ring, both with 128-byte swizzle (the layout the MMA descriptors
//     describe);
//   * warp 1, one lane: per k-block four tcgen05.mma (M 128, N 128)
//     accumulating in tensor memory, then tcgen05.commit to the stage's
//     "empty" mbarrier (the ring slot is free once those MMAs have read it)
//     and after the last k-block to the "done" mbarrier;
//   * warp 2 allocates (and at the end frees) 128 tensor-memory columns;
//   * all four warps then read the accumulators (warp w owns rows
//     32w .. 32w + 31, one tensor-memory lane per row) and write them out.
// Out-of-range rows, columns and k are read as zero by the copies.  Every
// wait is bounded; a wait that gives up records RNN_ERR_TIMEOUT in the
// status word, the roles stop issuing, and the CTA still waits (bounded) for
// its work in flight and frees its tensor memory before it returns.
#include <cstdint>

#include "rnn_internal.h"
#include "tma.cuh"

namespace rnngb {

namespace {

constexpr int TC_BM = 128, TC_BN = 128, TC_ROWB = 128, TC_ST = 3;   // TC_ROWB: bytes of a row per k-block
constexpr unsigned kTcTileA = TC_BM * TC_ROWB, kTcTileB = TC_BN * TC_ROWB;   // 16 KB each
constexpr unsigned kTcStage = kTcTileA + kTcTileB;
constexpr size_t kTcSmem = (size_t)TC_ST * kTcStage + 1024;   // + alignment slack (1024 for the swizzle)
constexpr unsigned kTmemCols = 128;

struct TcArgs {
    CUtensorMap amap;   // X  [M][K]:  dims {K, M},  box {k-block, 128}, 128-byte swizzle
    CUtensorMap bmap;   // Wk [NC][K]: dims {K, NC}, box {k-block, 128}, 128-byte swizzle
    float* C;
    int M, NC, nk;      // nk: k-blocks
    int* status;
    long long limit_ns;
};

// Shared-memory matrix descriptor of a K-major operand stored as 128-byte
// rows with 128-byte swizzle (8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_k_sw128(unsigned saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);     // start address
    d |= (uint64_t)1u << 16;                      // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;            // stride byte offset: next 8-row group
    d |= (uint64_t)1u << 46;                      // descriptor version
    d |= (uint64_t)2u << 61;                      // 128-byte swizzle
    return d;
}

// Instruction descriptors: D f32, both operands K-major, M 128, N 128;
// A and B tf32 (kind::tf32) or both bf16 (kind::f16).
constexpr uint32_t kIdescShape = ((uint32_t)(TC_BN >> 3) << 17) | ((uint32_t)(TC_BM >> 4) << 24);
constexpr uint32_t kIdescTf32 = (1u << 4) | (2u << 7) | (2u << 10) | kIdescShape;
constexpr uint32_t kIdescBf16 = (1u << 4) | (1u << 7) | (1u << 10) | kIdescShape;

template <bool BF16>
__device__ __forceinline__ void mma_issue(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate)
{
    if constexpr (BF16) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
            "l"(adesc), "l"(bdesc), "r"(kIdescBf16), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
            "l"(adesc), "l"(bdesc), "r"(kIdescTf32), "r"(accumulate)
            : "memory");
    }
}

__device__ __forceinline__ void mma_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive accumulator columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait on an mbarrier phase; gives up when the limit passes or (if
// abort_flag is given) another role of the CTA has given up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, unsigned parity, long long limit_ns,
                                        volatile int* abort_flag)
{
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    unsigned it = 0;
    while (!mbar_test(bar, parity)) {
        if ((++it & 255u) == 0u) {
            if (abort_flag && *abort_flag) return false;
            if ((long long)(globaltimer_ns() - t0) > limit_ns) return false;
        }
    }
    return true;
}

template <bool BF16>
__global__ void __launch_bounds__(128, 2) proj_tc_kernel(const __grid_constant__ TcArgs a)
{
    constexpr int BKE = BF16 ? 64 : 32;   // elements of a row per k-block
    extern __shared__ __align__(1024) unsigned char tc_smem[];
    __shared__ __align__(8) uint64_t full[TC_ST], empty[TC_ST], done;
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort;
    unsigned char* base = tc_smem + ((1024u - (smem_addr(tc_smem) & 1023u)) & 1023u);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = (int)blockIdx.y * TC_BM, n0 = (int)blockIdx.x * TC_BN;

    if (threadIdx.x == 0) {
        for (int i = 0; i < TC_ST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&done, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;

    int issued = 0;   // producer: k-blocks whose copies were issued
    if (warp == 0 && lane == 0) {
        // producer
        for (int kb = 0; kb < a.nk; ++kb) {
            const int s = kb % TC_ST;
            if (kb >= TC_ST && !tc_wait(&empty[s], (unsigned)((kb / TC_ST) - 1) & 1u, a.limit_ns, &s_abort)) {
                atomicCAS(a.status, 0, 6 /* RNN_ERR_TIMEOUT */);
                s_abort = 1;
                break;
            }
            unsigned char* st = base + (size_t)s * kTcStage;
            mbar_arrive_expect_tx(&full[s], kTcStage);
            tma_load_2d(st, &a.amap, kb * BKE, m0, &full[s]);
            tma_load_2d(st + kTcTileA, &a.bmap, kb * BKE, n0, &full[s]);
            ++issued;
        }
    } else if (warp == 1 && lane == 0) {
        // MMA issuer
        int kb = 0;
        for (; kb < a.nk; ++kb) {
            const int s = kb % TC_ST;
            if (!tc_wait(&full[s], (unsigned)(kb / TC_ST) & 1u, a.limit_ns, &s_abort)) {
                atomicCAS(a.status, 0, 6 /* RNN_ERR_TIMEOUT */);
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const unsigned sa = smem_addr(base + (size_t)s * kTcStage);
            const unsigned sb = sa + kTcTileA;
#pragma unroll
            for (int j = 0; j < 4; ++j)   // one MMA per 32 bytes along the swizzled row (K 8 tf32 / 16 bf16)
                mma_issue<BF16>(tmem, sdesc_k_sw128(sa + 32u * j), sdesc_k_sw128(sb + 32u * j),
                                (kb > 0 || j > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
        }
        mma_commit(&done);   // arrives once every MMA issued above has completed
    }
    __syncwarp();

    // epilogue: every warp reads its 32 lanes (rows) of the accumulators
    // (the tensor-memory loads are warp-collective: the decision is made
    // once for the whole CTA)
    const bool ok = __syncthreads_and(tc_wait(&done, 0u, a.limit_ns, &s_abort) && !s_abort);
    tc_fence_after();
    if (ok && a.nk > 0) {
        const int row = m0 + warp * 32 + lane;
#pragma unroll 1
        for (int c = 0; c < TC_BN; c += 32) {
            float v[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
            if (row < a.M) {
                float* crow = a.C + (size_t)row * a.NC + n0 + c;
                if (n0 + c + 32 <= a.NC) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        *reinterpret_cast<float4*>(crow + 4 * q) = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                } else {
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        if (n0 + c + q < a.NC) crow[q] = v[q];
                }
            }
        }
    } else if (!ok && threadIdx.x == 0) {
        atomicCAS(a.status, 0, 6 /* RNN_ERR_TIMEOUT */);
        // copies still in flight must land before the shared memory goes away
        for (int kb = max(0, issued - TC_ST); kb < issued; ++kb)
            (void)tc_wait(&full[kb % TC_ST], (unsigned)(kb / TC_ST) & 1u, a.limit_ns, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

bool projection_tc_supported(const void* X, const void* Wk, float* XW, int64_t M, int64_t K, int64_t ncols,
                             bool bf16)
{
    const int64_t kq = bf16 ? 8 : 4;   // 16-byte rows
    return K > 0 && K % kq == 0 && ncols % 4 == 0 && (uintptr_t)X % 16 == 0 && (uintptr_t)Wk % 16 == 0 &&
           (uintptr_t)XW % 16 == 0 && M < (1ll << 31) && ncols < (1ll << 31) && K < (1ll << 31) &&
           (M + TC_BM - 1) / TC_BM <= 65535;
}

cudaError_t launch_projection_tc(const void* X, const void* Wk, float* XW, int64_t M, int64_t K, int64_t ncols,
                                 bool bf16, int* status, long long limit_ns, cudaStream_t stream)
{
    if (M <= 0 || ncols <= 0) return cudaSuccess;
    if (!projection_tc_supported(X, Wk, XW, M, K, ncols, bf16)) return cudaErrorInvalidValue;
    const int es = bf16 ? 2 : 4, bke = TC_ROWB / es;
    TcArgs ta;
    const cuuint64_t adims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t astr[1] = {(cuuint64_t)K * es};
    const cuuint32_t box[2] = {(cuuint32_t)bke, (cuuint32_t)TC_BM};
    const cuuint64_t bdims[2] = {(cuuint64_t)K, (cuuint64_t)ncols};
    if (!encode_tensor_map(&ta.amap, X, 2, adims, astr, box, true, bf16) ||
        !encode_tensor_map(&ta.bmap, Wk, 2, bdims, astr, box, true, bf16))
        return cudaErrorInvalidValue;
    ta.C = XW;
    ta.M = (int)M;
    ta.NC = (int)ncols;
    ta.nk = (int)((K + bke - 1) / bke);
    ta.status = status;
    ta.limit_ns = limit_ns;
    const void* fn = bf16 ? (const void*)proj_tc_kernel<true> : (const void*)proj_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)((ncols + TC_BN - 1) / TC_BN), (unsigned)((M + TC_BM - 1) / TC_BM));
    if (bf16) proj_tc_kernel<true><<<grid, 128, kTcSmem, stream>>>(ta);
    else proj_tc_kernel<false><<<grid, 128, kTcSmem, stream>>>(ta);
    return cudaGetLastError();
}

}  // namespace rnngb
