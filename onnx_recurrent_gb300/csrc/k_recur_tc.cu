// Persistent recurrent kernel on the tensor cores (the TF32 and BF16 modes,
// batches of up to 128 rows).
//
// Page "Recurrent operators: RNN, GRU, LSTM", Computation: per step the
// recurrent product Rec = H . R^T, then the gate arithmetic per batch row in
// the written order (Fast mode: the product's order and rounding are free).
// Here the product runs on the tensor cores with fp16 operands (h and R
// rounded to nearest: 10-bit mantissas, as TF32) and FP32 sums.  The kernel
// is used only when every h it produces is bounded (see the planner), so h
// always fits fp16's range.
//
// One cooperative launch, one CTA per SM; CTA c of direction d owns hidden
// units [u0, u0 + U) and their G gate columns (column ul*G + g, padded to NP,
// a multiple of 16), for all batch rows (padded to 128: the MMA's M).
//   * its slice of R (fp16, K-major, NP rows x H) is loaded once into shared
//     memory by tensor copies (128-byte swizzle, one box per 64-k block) and
//     stays there as the MMA's B operand;
//   * warp 4 (one lane) waits each step for every CTA of the direction to
//     have published the step (a release-add / acquire-poll counter), then
//     moves h (fp16 [128 rows][H], the exchange buffer) through a ring of
//     64-k blocks (up to 4 stages of 16 KB, fewer if shared memory is short)
//     with tensor copies;
//   * warp 5 (one lane) issues four tcgen05.mma (kind::f16, M 128, N NP,
//     K 16) per block into tensor memory, commits each ring slot back to the
//     producer and, after the last block, the accumulators to the epilogue;
//   * warps 0-3 are the epilogue: thread t owns batch row t (tensor-memory
//     lane t), reads its NP accumulators, adds XW (its row's columns, 16
//     bytes per load where they are aligned) and the biases, runs the gate
//     arithmetic (FMA-based, hardware tanh) with its cell state kept in
//     registers (h kept in fp32 too), and stages its row of Y and of the
//     fp16 h in shared memory; the four warps then write the h tile with
//     consecutive threads on consecutive units (a thread per row would make
//     every store instruction touch 32 rows), the CTA publishes, and only
//     then is the Y tile written (no other CTA reads Y).
// Every wait is bounded; on a failure the CTA records RNN_ERR_TIMEOUT and
// its roles leave at the next uniform point, waiting (bounded) for their
// copies and MMAs in flight before the tensor memory is freed.
#include <cstdint>
#include <type_traits>

#include <cuda_fp16.h>

#include "k_recur.cuh"
#include "tma.cuh"

namespace rnngb {

namespace {

constexpr int TR_M = 128;                       // MMA rows (batch rows, padded)
constexpr int TR_KB = 64;                       // fp16 k per block (128-byte rows)
constexpr int TR_STMAX = 4;                     // most h ring stages (measured: deeper rings are slower)
constexpr unsigned kTrHStage = TR_M * 128;      // one h block: 16 KB
constexpr int TR_NPMAX = 64;                    // most gate columns per CTA
constexpr int TR_THREADS = 192;

__device__ __forceinline__ uint64_t tr_sdesc(unsigned saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);    // start address
    d |= (uint64_t)1u << 16;                     // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;           // stride byte offset: next 8-row group
    d |= (uint64_t)1u << 46;                     // descriptor version
    d |= (uint64_t)2u << 61;                     // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void tr_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tr_commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tr_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tr_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tr_bar(int id, int threads) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory"); }

// Columns J .. J+15 of this thread's tensor-memory lane into acc[J .. J+15].
template <int J>
__device__ __forceinline__ void tr_ld16(uint32_t taddr, float (&acc)[TR_NPMAX])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[J + i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tr_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Bounded wait on an mbarrier phase; gives up when the limit passes, the CTA
// is aborting, or another CTA reported a failure.
__device__ __forceinline__ bool tr_wait(uint64_t* bar, unsigned parity, const RecParams& p, volatile int* abort_flag)
{
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    unsigned it = 0;
    while (!mbar_test(bar, parity)) {
        if ((++it & 255u) == 0u) {
            if (abort_flag && *abort_flag) return false;
            if (ld_relaxed_s32(p.status) != 0) return false;
            if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tr_fail(const RecParams& p, volatile int* abort_flag)
{
    atomicCAS(p.status, 0, 6 /* RNN_ERR_TIMEOUT */);
    *abort_flag = 1;
}

// The tensor-core modes promise 5e-3, so their tanh and sigmoid use the
// hardware tanh (tanh.approx.f32, relative error about 2^-11, below the fp16
// rounding of h): tanh(x), sigmoid(x) = 1/2 + tanh(x/2)/2, alpha*tanh(beta*x).
__device__ __forceinline__ float tc_tanh(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float tc_sigmoid(float x) { return fmaf(0.5f, tc_tanh(0.5f * x), 0.5f); }

// v[k] = act(v[k]) over a whole array for one activation id known at compile
// time (the id's switch folds away: one formula per element).
template <int FN, int K>
__device__ __forceinline__ void tc_apply(const ActSpec& a, float (&v)[K])
{
#pragma unroll
    for (int k = 0; k < K; ++k) {
        if constexpr (FN == 1) v[k] = tc_tanh(v[k]);
        else if constexpr (FN == 2) v[k] = tc_sigmoid(v[k]);
        else if constexpr (FN == 6) v[k] = a.alpha * tc_tanh(a.beta * v[k]);
        else v[k] = activation<false>(FN, a.alpha, a.beta, v[k]);
    }
}

// KIND 1 and 2 call sigmoid and tanh directly; KIND 0 dispatches on the
// activation id once for the array.
template <int KIND, int K>
__device__ __forceinline__ void tc_act_array(const ActSpec& a, float (&v)[K], const RecParams& p, bool clip)
{
    if (clip && p.has_clip) {
#pragma unroll
        for (int k = 0; k < K; ++k) v[k] = v[k] > p.clip ? p.clip : (v[k] < -p.clip ? -p.clip : v[k]);
    }
    if constexpr (KIND == 1) {
        tc_apply<2, K>(a, v);
    } else if constexpr (KIND == 2) {
        tc_apply<1, K>(a, v);
    } else {
        switch (a.fn) {
        case 0: tc_apply<0, K>(a, v); break;
        case 1: tc_apply<1, K>(a, v); break;
        case 2: tc_apply<2, K>(a, v); break;
        case 3: tc_apply<3, K>(a, v); break;
        case 4: tc_apply<4, K>(a, v); break;
        case 5: tc_apply<5, K>(a, v); break;
        case 6: tc_apply<6, K>(a, v); break;
        case 7: tc_apply<7, K>(a, v); break;
        case 8: tc_apply<8, K>(a, v); break;
        case 9: tc_apply<9, K>(a, v); break;
        default: tc_apply<10, K>(a, v); break;
        }
    }
}

// A row's XW columns [0, n) into registers (zero past n): 16-byte loads when
// `vec` (start 16-byte aligned, n a multiple of 4), else 4-byte loads.
template <int NMAX>
__device__ __forceinline__ void tc_load_xw(float (&xw)[NMAX], const float* src, int n, bool vec)
{
    if (vec) {
#pragma unroll
        for (int j = 0; j < NMAX / 4; ++j) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (4 * j < n) v = __ldg(reinterpret_cast<const float4*>(src) + j);
            xw[4 * j] = v.x; xw[4 * j + 1] = v.y; xw[4 * j + 2] = v.z; xw[4 * j + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < NMAX; ++j) xw[j] = j < n ? __ldg(src + j) : 0.f;
    }
}

// TWO (GRU with linear_before_reset = 0): two products per step, z and r
// over h, then the candidate over r (.) h once every CTA has published its
// units' r (.) h; R's rows are packed z/r first, candidate rows after.
template <int OP, bool TWO>
__global__ void __launch_bounds__(TR_THREADS, 1) rnn_tc_kernel(const __grid_constant__ RecParams p)
{
    constexpr int G = OP == 0 ? 1 : (OP == 1 ? 3 : 4);
    constexpr int UMAX = G == 1 ? 32 : TR_NPMAX / G;   // most units per CTA (register arrays)
    extern __shared__ __align__(1024) unsigned char tr_smem[];
    __shared__ __align__(8) uint64_t full[TR_STMAX], empty[TR_STMAX], r_ready, acc_ready, acc_free, mma_done;
    __shared__ __align__(8) uint64_t acc2_ready, acc2_free;   // TWO: the candidate product's accumulators
    __shared__ uint32_t tmem_slot;
    __shared__ int s_abort;
    __shared__ float s_wb[TR_NPMAX], s_rb[TR_NPMAX], s_p[3][UMAX];

    unsigned char* base = tr_smem + ((1024u - (smem_addr(tr_smem) & 1023u)) & 1023u);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = p.ctas_per_dir;
    const int d = blockIdx.x / C, c = blockIdx.x - d * C;
    const int H = p.H, GH = G * H;
    const int u0 = (int)(((long long)c * H) / C);
    const int U = (int)(((long long)(c + 1) * H) / C) - u0;
    const int NP = p.npad;                                  // padded gate columns (MMA N)
    const int NP2 = TWO ? p.npad2 : 0;                      // TWO: padded candidate columns
    const int nkb = (H + TR_KB - 1) / TR_KB;
    unsigned char* rsm = base;                              // R slice: nkb blocks of [NP rows][128 B]
    unsigned char* rsm2 = base + (size_t)nkb * NP * 128;    // TWO: nkb blocks of [NP2 rows][128 B]
    const int nst = p.slots;                                // h ring stages
    unsigned char* hring = rsm2 + (size_t)nkb * NP2 * 128;  // nst blocks of [128 rows][128 B]
    // per-step staging of the CTA's output tiles: Y [128][umax] fp32, h [128][umax] fp16, t per row
    float* s_y = reinterpret_cast<float*>(hring + (size_t)nst * kTrHStage);
    __half* s_h = reinterpret_cast<__half*>(s_y + (size_t)TR_M * p.umax);
    int* s_t = reinterpret_cast<int*>(s_h + (size_t)TR_M * ((p.umax + 1) & ~1));
    const bool rev = p.dir_reverse[d] != 0;
    unsigned* counter = p.bar + d;
    unsigned* counter2 = p.flags + d;                       // TWO: r (.) h publications
    const uint32_t idesc = (1u << 4) | ((uint32_t)(NP >> 3) << 17) | ((uint32_t)(TR_M >> 4) << 24);
    const uint32_t idesc2 = (1u << 4) | ((uint32_t)(NP2 >> 3) << 17) | ((uint32_t)(TR_M >> 4) << 24);
    int tmem_cols = 32;
    while (tmem_cols < NP + NP2) tmem_cols *= 2;

    if (threadIdx.x == 0) {
        for (int i = 0; i < nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&r_ready, 1);
        mbar_init(&acc_ready, 1);
        mbar_init(&acc_free, 4);   // one arrival per epilogue warp
        mbar_init(&acc2_ready, 1);
        mbar_init(&acc2_free, 4);
        mbar_init(&mma_done, 1);
        s_abort = 0;
        mbar_fence_init();
    }
    // biases and peepholes of the CTA's columns (zero where absent)
    for (int j = threadIdx.x; j < TR_NPMAX; j += blockDim.x) {
        const int ul = j / G, g = j - ul * G;
        const bool in = ul < U;
        s_wb[j] = (in && p.has_B) ? p.B[(size_t)d * 2 * GH + (size_t)g * H + u0 + ul] : 0.f;
        s_rb[j] = (in && p.has_B) ? p.B[(size_t)d * 2 * GH + GH + (size_t)g * H + u0 + ul] : 0.f;
    }
    for (int j = threadIdx.x; j < 3 * UMAX; j += blockDim.x) {
        const int k = j / UMAX, ul = j - k * UMAX;
        s_p[k][ul] = (OP == 2 && p.has_P && ul < U) ? p.P[(size_t)d * 3 * H + (size_t)k * H + u0 + ul] : 0.f;
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                     "r"(tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // h blocks are copied for the batch's rows only (rounded up to 8): the
    // MMA's other rows stay zero in every ring slot (whole 128-byte rows, so
    // the swizzle does not matter); the tensor cores read them through the
    // async proxy
    const int hrows = (p.N + 7) & ~7;
    const unsigned hbytes = (unsigned)hrows * 128u;
    if (hrows < TR_M) {
        for (int st = 0; st < nst; ++st) {
            uint4* z = reinterpret_cast<uint4*>(hring + (size_t)st * kTrHStage + hbytes);
            for (int i = threadIdx.x; i < (int)((kTrHStage - hbytes) / 16); i += blockDim.x) z[i] = make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tr_fence_before();
    __syncthreads();
    tr_fence_after();
    const uint32_t tmem = tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            mbar_arrive_expect_tx(&r_ready, (unsigned)(nkb * (NP + NP2) * 128));
            for (int kb = 0; kb < nkb; ++kb) {
                if constexpr (TWO) {
                    tma_load_2d(rsm + (size_t)kb * NP * 128, &p.rmap, kb * TR_KB, d * GH + u0 * 2, &r_ready);
                    tma_load_2d(rsm2 + (size_t)kb * NP2 * 128, &p.rmap2, kb * TR_KB, d * GH + 2 * H + u0,
                                &r_ready);
                } else {
                    tma_load_2d(rsm + (size_t)kb * NP * 128, &p.rmap, kb * TR_KB, d * GH + u0 * G, &r_ready);
                }
            }
            unsigned q = 0;
            bool ok = true;
            for (int s = 0; s < p.max_len && ok; ++s) {
                if (s > 0) {
                    const unsigned need = (unsigned)s * (unsigned)C;
                    const unsigned long long t0 = globaltimer_ns();
                    unsigned it = 0;
                    while (ld_acquire_u32(counter) < need) {
                        if ((++it & 63u) == 0u) {
                            if (s_abort || ld_relaxed_s32(p.status) != 0) { ok = false; break; }
                            if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) {
                                tr_fail(p, &s_abort);
                                ok = false;
                                break;
                            }
                        }
                    }
                    if (!ok) break;
                    fence_proxy_async_global();
                }
                const int z = (s & 1) * p.D + d;
                for (int part = 0; part < (TWO ? 2 : 1) && ok; ++part) {
                    if (part == 1) {
                        // every CTA of the direction has published r (.) h of this step
                        const unsigned need = (unsigned)(s + 1) * (unsigned)C;
                        const unsigned long long t0 = globaltimer_ns();
                        unsigned it = 0;
                        while (ld_acquire_u32(counter2) < need) {
                            if ((++it & 63u) == 0u) {
                                if (s_abort || ld_relaxed_s32(p.status) != 0) { ok = false; break; }
                                if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) {
                                    tr_fail(p, &s_abort);
                                    ok = false;
                                    break;
                                }
                            }
                        }
                        if (!ok) break;
                        fence_proxy_async_global();
                    }
                    const CUtensorMap* src = part == 0 ? &p.hmap : &p.rhmap;
                    for (int kb = 0; kb < nkb; ++kb, ++q) {
                        const int slot = (int)(q % nst);
                        if (q >= (unsigned)nst && !tr_wait(&empty[slot], ((q / nst) - 1u) & 1u, p, &s_abort)) {
                            tr_fail(p, &s_abort);
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[slot], hbytes);
                        tma_load_3d(hring + (size_t)slot * kTrHStage, src, kb * TR_KB, 0, z, &full[slot]);
                    }
                }
            }
            // copies still in flight land before the CTA can leave
            (void)tr_wait(&r_ready, 0u, p, nullptr);
            for (unsigned k = (q > (unsigned)nst ? q - nst : 0u); k < q; ++k)
                (void)tr_wait(&full[k % nst], (k / nst) & 1u, p, nullptr);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool ok = tr_wait(&r_ready, 0u, p, &s_abort);
            if (!ok) tr_fail(p, &s_abort);
            unsigned q = 0;
            for (int s = 0; s < p.max_len && ok; ++s) {
                if (s > 0 && !tr_wait(&acc_free, (unsigned)(s - 1) & 1u, p, &s_abort)) {
                    tr_fail(p, &s_abort);
                    break;
                }
                tr_fence_after();
                for (int part = 0; part < (TWO ? 2 : 1) && ok; ++part) {
                    if (part == 1) {
                        // the candidate accumulators of the previous step have been read
                        if (s > 0 && !tr_wait(&acc2_free, (unsigned)(s - 1) & 1u, p, &s_abort)) {
                            tr_fail(p, &s_abort);
                            ok = false;
                            break;
                        }
                        tr_fence_after();
                    }
                    unsigned char* rb = part == 0 ? rsm : rsm2;
                    const int np = part == 0 ? NP : NP2;
                    const uint32_t id = part == 0 ? idesc : idesc2;
                    const uint32_t td = tmem + (part == 0 ? 0u : (uint32_t)NP);
                    for (int kb = 0; kb < nkb; ++kb, ++q) {
                        const int slot = (int)(q % nst);
                        if (!tr_wait(&full[slot], (q / nst) & 1u, p, &s_abort)) {
                            tr_fail(p, &s_abort);
                            ok = false;
                            break;
                        }
                        tr_fence_after();
                        const unsigned sa = smem_addr(hring + (size_t)slot * kTrHStage);
                        const unsigned sb = smem_addr(rb + (size_t)kb * np * 128);
#pragma unroll
                        for (int j = 0; j < 4; ++j)   // K 16 per MMA = 32 bytes along the swizzled rows
                            tr_mma_f16(td, tr_sdesc(sa + 32u * j), tr_sdesc(sb + 32u * j), id,
                                       (kb > 0 || j > 0) ? 1u : 0u);
                        tr_commit(&empty[slot]);
                    }
                    if (!ok) break;
                    tr_commit(part == 0 ? &acc_ready : &acc2_ready);
                }
                if (!ok) break;
            }
            // completes once every MMA issued above has: waited for before the
            // tensor memory is freed
            tr_commit(&mma_done);
            (void)tr_wait(&mma_done, 0u, p, nullptr);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int n = warp * 32 + lane;                      // batch row = tensor-memory lane
        const bool row = n < p.N;
        const int len = row ? (p.has_lens ? p.lens[n] : p.S) : 0;
        const ActSpec fA = p.act[d][0], gA = p.act[d][1], hA = p.act[d][2];
        // the operator's default activations (RNN Tanh; GRU Sigmoid, Tanh; LSTM
        // Sigmoid, Tanh, Tanh) are called directly
        const bool fixed_acts = OP == 0 ? fA.fn == 1
                                        : (OP == 1 ? fA.fn == 2 && gA.fn == 1 : fA.fn == 2 && gA.fn == 1 && hA.fn == 1);
        float hown[UMAX], cown[UMAX];
#pragma unroll
        for (int ul = 0; ul < UMAX; ++ul) {
            hown[ul] = (row && ul < U && p.has_h0) ? io_load(p.h0, s_index(p, d, n, u0 + ul), p.io) : 0.f;
            cown[ul] = (row && ul < U && OP == 2 && p.has_c0) ? io_load(p.c0, s_index(p, d, n, u0 + ul), p.io) : 0.f;
        }
        const size_t xw_ld = (size_t)p.D * GH;
        const size_t xw_col = (size_t)d * GH + (size_t)u0 * G;
        // a row's columns are one contiguous run: 16-byte loads where it is
        // aligned (each lane reads another row, so fewer, wider requests)
        const bool xw_vec = OP == 2 && ((xw_ld | xw_col | (size_t)(U * G)) % 4 == 0) &&
                            (reinterpret_cast<uintptr_t>(p.XW) % 16 == 0);
        __half* hx = reinterpret_cast<__half*>(p.hbuf);
        const bool skip_first = p.debug_skip_cta == (int)blockIdx.x;
        bool alive = true;
        if constexpr (TWO) {
            __half* rx = reinterpret_cast<__half*>(p.rhbuf);
            for (int s = 0; s < p.max_len; ++s) {
                float xw[TR_NPMAX];
                const bool live = row && s < len;
                const int t = live ? (rev ? len - 1 - s : s) : 0;
                if (live) {
                    const size_t xrow = p.layout == 0 ? (size_t)t * p.N + n : (size_t)n * p.S + t;
                    const float* src = p.XW + xrow * xw_ld + xw_col;
                    tc_load_xw<TR_NPMAX>(xw, src, U * G, xw_vec);
                }
                // ---- z and r: accumulators j = 2 ul + g in columns 0 .. NP-1
                const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
                const bool got = __all_sync(0xffffffffu, alive && tr_wait(&acc_ready, (unsigned)s & 1u, p, &s_abort));
                float acc[TR_NPMAX];
                if (got) {
                    tr_fence_after();
                    tr_ld16<0>(taddr, acc);
                    if (NP > 16) tr_ld16<16>(taddr + 16u, acc);
                    if (NP > 32) tr_ld16<32>(taddr + 32u, acc);
                    if (NP > 48) tr_ld16<48>(taddr + 48u, acc);
                    tr_ld_wait();
                    tr_fence_before();
                } else if (alive && lane == 0) {
                    tr_fail(p, &s_abort);
                }
                __syncwarp();
                if (lane == 0 && got) mbar_arrive(&acc_free);
                float z[UMAX], rr[UMAX];
                if (got && live) {
#pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul) {
                        const int j = 3 * ul;
                        z[ul] = (xw[j] + acc[2 * ul]) + s_wb[j] + s_rb[j];
                        rr[ul] = (xw[j + 1] + acc[2 * ul + 1]) + s_wb[j + 1] + s_rb[j + 1];
                    }
                    if (fixed_acts) {
                        tc_act_array<1, UMAX>(fA, z, p, true);
                        tc_act_array<1, UMAX>(fA, rr, p, true);
                    } else {
                        tc_act_array<0, UMAX>(fA, z, p, true);
                        tc_act_array<0, UMAX>(fA, rr, p, true);
                    }
                }
                // r (.) h of the CTA's units, staged and written units-fastest
                if (got && row) {
#pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul)
                        if (ul < U) s_h[n * p.umax + ul] = __float2half_rn(live ? rr[ul] * hown[ul] : 0.f);
                }
                tr_bar(1, 128);
                bool abort_now = s_abort != 0 || !got;
                if (!abort_now) {
                    __half* rdst = rx + ((size_t)(s & 1) * p.D + d) * TR_M * H + u0;
                    const int tot = p.N * U;
                    for (int i = threadIdx.x; i < tot; i += 128) {
                        const int rn = i / U, ul = i - rn * U;
                        rdst[(size_t)rn * H + ul] = s_h[rn * p.umax + ul];
                    }
                }
                tr_bar(1, 128);
                if (abort_now) {
                    alive = false;
                    break;
                }
                if (threadIdx.x == 0) {
                    fence_proxy_async_global();
                    red_release_add_u32(counter2, 1u);
                }
                // ---- candidate: accumulators j = ul in columns NP .. NP+NP2-1
                const bool got2 =
                    __all_sync(0xffffffffu, alive && tr_wait(&acc2_ready, (unsigned)s & 1u, p, &s_abort));
                if (got2) {
                    tr_fence_after();
                    tr_ld16<0>(taddr + (uint32_t)NP, acc);
                    if (NP2 > 16) tr_ld16<16>(taddr + (uint32_t)NP + 16u, acc);
                    tr_ld_wait();
                    tr_fence_before();
                } else if (alive && lane == 0) {
                    tr_fail(p, &s_abort);
                }
                __syncwarp();
                if (lane == 0 && got2) mbar_arrive(&acc2_free);
                if (got2 && live) {
                    float hc[UMAX];
#pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul) {
                        const int j = 3 * ul + 2;
                        hc[ul] = p.has_B ? ((xw[j] + acc[ul]) + s_wb[j]) + s_rb[j] : xw[j] + acc[ul];
                    }
                    if (fixed_acts) tc_act_array<2, UMAX>(gA, hc, p, true);
                    else tc_act_array<0, UMAX>(gA, hc, p, true);
#pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul) {
                        if (ul < U) {
                            hown[ul] = (1.0f - z[ul]) * hc[ul] + z[ul] * hown[ul];
                            s_y[n * p.umax + ul] = canon_nan(hown[ul]);
                        }
                    }
                } else if (got2 && row) {
#pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul)
                        if (ul < U) s_y[n * p.umax + ul] = 0.f;   // Y is +0 past the row's length
                }
                if (got2 && row) {
                    s_t[n] = live ? t : s;
#pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul)
                        if (ul < U) s_h[n * p.umax + ul] = __float2half_rn(hown[ul]);
                }
                tr_bar(1, 128);
                abort_now = s_abort != 0 || !got2;
                if (!abort_now) {
                    __half* hdst = hx + ((size_t)((s + 1) & 1) * p.D + d) * TR_M * H + u0;
                    const int tot = p.N * U;
                    for (int i = threadIdx.x; i < tot; i += 128) {
                        const int rn = i / U, ul = i - rn * U;
                        hdst[(size_t)rn * H + ul] = s_h[rn * p.umax + ul];
                    }
                }
                tr_bar(1, 128);
                if (abort_now) {
                    alive = false;
                    break;
                }
                if (threadIdx.x == 0 && !(skip_first && s == 0)) {
                    fence_proxy_async_global();
                    red_release_add_u32(counter, 1u);
                }
                // Y is read by no other CTA: its stores follow the publication,
                // off the exchange's critical path; the staged tiles are reused
                // only after every epilogue thread has read them
                if (p.Y) {
                    const int tot = p.N * U;
                    for (int i = threadIdx.x; i < tot; i += 128) {
                        const int rn = i / U, ul = i - rn * U;
                        io_store(p.Y, y_index(p, s_t[rn], d, rn, u0 + ul), s_y[rn * p.umax + ul], p.io);
                    }
                    tr_bar(1, 128);
                }
            }
        } else {
            for (int s = 0; s < p.max_len; ++s) {
                // this step's XW row (independent of the product: loaded first)
                float xw[TR_NPMAX];
                const bool live = row && s < len;
                const int t = live ? (rev ? len - 1 - s : s) : 0;
                if (live) {
                    const size_t xrow = p.layout == 0 ? (size_t)t * p.N + n : (size_t)n * p.S + t;
                    const float* src = p.XW + xrow * xw_ld + xw_col;
                    tc_load_xw<TR_NPMAX>(xw, src, U * G, xw_vec);
                }
                // accumulators (warp-collective loads: the decision is warp-uniform)
                const bool got = __all_sync(0xffffffffu, alive && tr_wait(&acc_ready, (unsigned)s & 1u, p, &s_abort));
                float acc[TR_NPMAX];
                if (got) {
                    tr_fence_after();
                    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
                    tr_ld16<0>(taddr, acc);
                    if (NP > 16) tr_ld16<16>(taddr + 16u, acc);
                    if (NP > 32) tr_ld16<32>(taddr + 32u, acc);
                    if (NP > 48) tr_ld16<48>(taddr + 48u, acc);
                    tr_ld_wait();
                    tr_fence_before();
                } else if (alive && lane == 0) {
                    tr_fail(p, &s_abort);
                }
                __syncwarp();
                if (lane == 0 && got) mbar_arrive(&acc_free);
                // pre-activations in place: acc = ((xw + rec) + Wb) + Rb, except the
                // GRU candidate's column, whose xw is kept apart (it is added after
                // r (.) (rec + Rb))
                float xh[OP == 1 ? UMAX : 1];
                if (got && live) {
    #pragma unroll
                    for (int j = 0; j < TR_NPMAX; ++j) {
                        if (OP == 1 && j % 3 == 2) {
                            if (j / 3 < UMAX) xh[j / 3] = xw[j];
                        } else {
                            acc[j] = (xw[j] + acc[j]) + s_wb[j] + s_rb[j];
                        }
                    }
                }
                if (got && live) {
                    // gate arithmetic gate-by-gate over the CTA's units: each
                    // activation is applied to a whole array, so its dispatch is
                    // paid once per gate and the units' chains run side by side
                    auto cells = [&](auto fx) {
                        constexpr int KIND_F = decltype(fx)::value ? (OP == 0 ? 2 : 1) : 0;   // 1 sigmoid, 2 tanh
                        constexpr int KIND_T = decltype(fx)::value ? 2 : 0;
                        (void)KIND_T;
                        if constexpr (OP == 0) {
                            float a[UMAX];
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul) a[ul] = acc[ul];
                            tc_act_array<KIND_F, UMAX>(fA, a, p, true);
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul) hown[ul] = ul < U ? a[ul] : hown[ul];
                        } else if constexpr (OP == 1) {
                            float z[UMAX], r[UMAX];
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul) {
                                z[ul] = acc[3 * ul];
                                r[ul] = acc[3 * ul + 1];
                            }
                            tc_act_array<KIND_F, UMAX>(fA, z, p, true);
                            tc_act_array<KIND_F, UMAX>(fA, r, p, true);
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul) {
                                const int j = 3 * ul + 2;
                                r[ul] = p.has_B ? (xh[ul] + r[ul] * (acc[j] + s_rb[j])) + s_wb[j] : xh[ul] + r[ul] * acc[j];
                            }
                            tc_act_array<KIND_T, UMAX>(gA, r, p, true);   // r now holds the candidate
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul)
                                if (ul < U) hown[ul] = (1.0f - z[ul]) * r[ul] + z[ul] * hown[ul];
                        } else {
                            float gi[UMAX], gf[UMAX], gc[UMAX], go[UMAX];
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul) {
                                const int j = 4 * ul;
                                gi[ul] = acc[j];
                                go[ul] = acc[j + 1];
                                gf[ul] = acc[j + 2];
                                gc[ul] = acc[j + 3];
                                if (p.has_P) {
                                    gi[ul] += s_p[0][ul] * cown[ul];
                                    gf[ul] += s_p[2][ul] * cown[ul];
                                }
                            }
                            tc_act_array<KIND_F, UMAX>(fA, gi, p, true);
                            if (p.input_forget) {
    #pragma unroll
                                for (int ul = 0; ul < UMAX; ++ul) gf[ul] = 1.0f - gi[ul];
                            } else {
                                tc_act_array<KIND_F, UMAX>(fA, gf, p, true);
                            }
                            tc_act_array<KIND_T, UMAX>(gA, gc, p, true);
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul) {
                                const float cn = gf[ul] * cown[ul] + gi[ul] * gc[ul];
                                if (ul < U) cown[ul] = cn;
                                gc[ul] = cn;
                                if (p.has_P) go[ul] += s_p[1][ul] * cn;
                            }
                            tc_act_array<KIND_F, UMAX>(fA, go, p, true);
                            tc_act_array<KIND_T, UMAX>(hA, gc, p, false);   // the cell state is not clipped
    #pragma unroll
                            for (int ul = 0; ul < UMAX; ++ul)
                                if (ul < U) hown[ul] = go[ul] * gc[ul];
                        }
    #pragma unroll
                        for (int ul = 0; ul < UMAX; ++ul)
                            if (ul < U) s_y[n * p.umax + ul] = canon_nan(hown[ul]);
                    };
                    if (fixed_acts) cells(std::true_type{});
                    else cells(std::false_type{});
                } else if (got && row) {
    #pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul)
                        if (ul < U) s_y[n * p.umax + ul] = 0.f;   // Y is +0 past the row's length
                }
                if (got && row) {
                    s_t[n] = live ? t : s;
    #pragma unroll
                    for (int ul = 0; ul < UMAX; ++ul)
                        if (ul < U) s_h[n * p.umax + ul] = __float2half_rn(hown[ul]);
                }
                tr_bar(1, 128);
                const bool abort_now = s_abort != 0 || !got;
                if (!abort_now) {
                    // the staged tiles, units fastest: a warp's stores cover a few
                    // contiguous row segments
                    __half* hdst = hx + ((size_t)((s + 1) & 1) * p.D + d) * TR_M * H + u0;
                    const int tot = p.N * U;
                    for (int i = threadIdx.x; i < tot; i += 128) {
                        const int rn = i / U, ul = i - rn * U;
                        hdst[(size_t)rn * H + ul] = s_h[rn * p.umax + ul];
                    }
                }
                // publish: every epilogue thread's writes are done; leave together on a failure
                tr_bar(1, 128);
                if (abort_now) {
                    alive = false;
                    break;
                }
                if (threadIdx.x == 0 && !(skip_first && s == 0)) {
                    fence_proxy_async_global();
                    red_release_add_u32(counter, 1u);
                }
                // Y is read by no other CTA: its stores follow the publication,
                // off the exchange's critical path; the staged tiles are reused
                // only after every epilogue thread has read them
                if (p.Y) {
                    const int tot = p.N * U;
                    for (int i = threadIdx.x; i < tot; i += 128) {
                        const int rn = i / U, ul = i - rn * U;
                        io_store(p.Y, y_index(p, s_t[rn], d, rn, u0 + ul), s_y[rn * p.umax + ul], p.io);
                    }
                    tr_bar(1, 128);
                }
            }
        }
        if (alive && row) {
#pragma unroll
            for (int ul = 0; ul < UMAX; ++ul) {
                if (ul >= U) break;
                const size_t si = s_index(p, d, n, u0 + ul);
                if (p.Yh) io_store(p.Yh, si, len > 0 ? canon_nan(hown[ul]) : 0.f, p.io);
                if (OP == 2 && p.Yc) io_store(p.Yc, si, len > 0 ? canon_nan(cown[ul]) : 0.f, p.io);
            }
        }
    }

    tr_fence_before();
    __syncthreads();
    if (warp == 5) {
        tr_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(tmem_cols) : "memory");
    }
}

template <int OP, bool TWO>
const void* tc_kernel_ptr()
{
    return (const void*)rnn_tc_kernel<OP, TWO>;
}

const void* tc_kernel_for(int op, bool two)
{
    if (op == 0) return tc_kernel_ptr<0, false>();
    if (op == 1) return two ? tc_kernel_ptr<1, true>() : tc_kernel_ptr<1, false>();
    return tc_kernel_ptr<2, false>();
}

}  // namespace

size_t tc_recurrent_smem(int H, int npad, int umax, int stages)   // npad: R rows per CTA (both products)
{
    return 1024 + (size_t)((H + TR_KB - 1) / TR_KB) * npad * 128 + (size_t)stages * kTrHStage +
           (size_t)TR_M * umax * 4 + (size_t)TR_M * ((umax + 1) & ~1) * 2 + (size_t)TR_M * 4;
}

int tc_recurrent_max_stages() { return TR_STMAX; }

int tc_recurrent_threads() { return TR_THREADS; }

int tc_recurrent_max_columns() { return TR_NPMAX; }

int tc_recurrent_max_units(int op) { return op == 0 ? 32 : TR_NPMAX / (op == 1 ? 3 : 4); }

cudaError_t tc_recurrent_occupancy(int op, bool two, size_t smem, int* blocks)
{
    const void* fn = tc_kernel_for(op, two);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, TR_THREADS, smem);
}

cudaError_t launch_tc_recurrent(const RecParams& p, size_t smem, cudaStream_t stream)
{
    const void* fn = tc_kernel_for(p.op, p.op == 1 && p.lbr == 0);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {(void*)&p};
    return cudaLaunchCooperativeKernel(fn, dim3(p.D * p.ctas_per_dir), dim3(TR_THREADS), args, smem, stream);
}

}  // namespace rnngb
