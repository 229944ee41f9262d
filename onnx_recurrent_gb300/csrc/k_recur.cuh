// Persistent recurrent kernel: every time step of every direction in one
// cooperative launch.
//
// Page "Recurrent operators: RNN, GRU, LSTM", Computation: per step s the
// recurrent product Rec = H.R^T (one accumulator per output, k increasing
// from +0; for GRU with linear_before_reset = 0 only the z and r columns,
// followed by the candidate's product (r (.) H).Rh^T once r is known), then
// the gate arithmetic per batch row in the written order; Choices the
// specification leaves open: sequence_lens (a row runs its first len steps,
// the reverse direction starting at len - 1; Y = 0 past a row's length;
// Y_h / Y_c are the state after the row's last valid step, 0 for length 0);
// Exact mode: NaN outputs written as 0x7FC00000.
//
// Work split.  CTA c of direction d owns hidden units [u0, u1) and all G gate
// columns of each, so the cell update of a (row, unit) pair needs no data from
// other CTAs.  Thread (rb, ul) owns unit u0 + ul for batch rows
// rb*TN .. rb*TN + TN - 1: its gate pre-activations accumulate in registers
// and its cell state c never leaves them.  Only h crosses CTAs: each step
// writes its units' h into a global ping-pong buffer hbuf[d][2][H][npad]
// (k-major, so a k-chunk of it is one contiguous block), a device-wide
// barrier among the direction's CTAs publishes it, and every CTA streams the
// whole of it back through a cp.async ring in shared memory while it
// accumulates.  The CTA's slice of R (k-major [H][U*G]) stays resident in
// shared memory when it fits, else it is streamed through the same ring.
//
// The barrier is a monotonic arrival counter per direction (release add /
// acquire poll at GPU scope).  Every wait is bounded: past the limit the CTA
// records RNN_ERR_TIMEOUT in the status word and returns, and CTAs that see a
// non-zero status stop waiting too, so the grid always finishes.
#pragma once

#include "exact_math.cuh"
#include "io_types.cuh"
#include "rnn_internal.h"
#include "tma.cuh"

namespace rnngb {

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_add_u32(unsigned* p, unsigned v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_relaxed_s32(const int* p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async16_cg(void* smem, const void* gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async4_ca(void* smem, const void* gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Device-wide barrier among the `ctas` CTAs of one direction.  Returns false
// if the run is being abandoned (timeout here or elsewhere).
__device__ __forceinline__ bool step_barrier(unsigned* ctr, unsigned target, int* status,
                                             long long limit_ns, bool arrive, int ctas)
{
    __shared__ int s_ok;
    __syncthreads();
    if (ctas == 1 && arrive) return true;   // one CTA: __syncthreads is the barrier
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        if (arrive) red_release_add_u32(ctr, 1u);
        const unsigned long long t0 = globaltimer_ns();
        unsigned it = 0;
        while (ld_acquire_u32(ctr) < target) {
            if ((++it & 31u) == 0u) {
                if (ld_relaxed_s32(status) != 0) { ok = 0; break; }
                if ((long long)(globaltimer_ns() - t0) > limit_ns) {
                    atomicCAS(status, 0, 6 /* RNN_ERR_TIMEOUT */);
                    ok = 0;
                    break;
                }
            }
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

template <bool EXACT>
__device__ __forceinline__ float mac(float acc, float a, float b)
{
    return EXACT ? fadd(acc, fmul(a, b)) : __fmaf_rn(a, b, acc);
}

template <int TN>
__device__ __forceinline__ void load_rows(float (&hv)[TN], const float* p)
{
    if constexpr (TN == 1) {
        hv[0] = p[0];
    } else if constexpr (TN == 2) {
        const float2 v = *reinterpret_cast<const float2*>(p);
        hv[0] = v.x; hv[1] = v.y;
    } else {
#pragma unroll
        for (int q = 0; q < TN / 4; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(p + 4 * q);
            hv[4 * q] = v.x; hv[4 * q + 1] = v.y; hv[4 * q + 2] = v.z; hv[4 * q + 3] = v.w;
        }
    }
}

template <int NC>
__device__ __forceinline__ void load_cols(float (&rv)[NC], const float* p)
{
    if constexpr (NC == 4) {
        const float4 v = *reinterpret_cast<const float4*>(p);
        rv[0] = v.x; rv[1] = v.y; rv[2] = v.z; rv[3] = v.w;
    } else {
#pragma unroll
        for (int j = 0; j < NC; ++j) rv[j] = p[j];
    }
}

// One full k-chunk (kRecKC rows) of the product for a thread's TN rows and NC
// gate columns: acc[i][j] += h[k][i] * r[k][j], k ascending.  The shared-memory
// operands go through registers in blocks of KB k-rows, block b+1 loaded
// while block b is multiplied.
template <int TN, int NC, bool EXACT>
__device__ __forceinline__ void chunk_full(const float* hk, int hstride, const float* rk, int rstride,
                                           float (&acc)[TN][NC])
{
    constexpr int KB = (TN * NC >= 16) ? 4 : 8;
    constexpr int NB = kRecKC / KB;
    float hv[2][KB][TN], rv[2][KB][NC];
#pragma unroll
    for (int j = 0; j < KB; ++j) {
        load_rows<TN>(hv[0][j], hk + (size_t)j * hstride);
        load_cols<NC>(rv[0][j], rk + (size_t)j * rstride);
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
        const int cur = b & 1;
        if (b + 1 < NB) {
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                load_rows<TN>(hv[cur ^ 1][j], hk + (size_t)((b + 1) * KB + j) * hstride);
                load_cols<NC>(rv[cur ^ 1][j], rk + (size_t)((b + 1) * KB + j) * rstride);
            }
        }
#pragma unroll
        for (int j = 0; j < KB; ++j)
#pragma unroll
            for (int i = 0; i < TN; ++i)
#pragma unroll
                for (int g = 0; g < NC; ++g) acc[i][g] = mac<EXACT>(acc[i][g], hv[cur][j][i], rv[cur][j][g]);
    }
}

// A partial chunk (the last one when H is not a multiple of kRecKC).
template <int TN, int NC, bool EXACT>
__device__ __forceinline__ void chunk_part(const float* hk, int hstride, const float* rk, int rstride, int kc,
                                           float (&acc)[TN][NC])
{
    for (int kk = 0; kk < kc; ++kk) {
        float hv[TN], rv[NC];
        load_rows<TN>(hv, hk + (size_t)kk * hstride);
        load_cols<NC>(rv, rk + (size_t)kk * rstride);
#pragma unroll
        for (int i = 0; i < TN; ++i)
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[i][j] = mac<EXACT>(acc[i][j], hv[i], rv[j]);
    }
}

// Shared per-CTA context of the kernel.
struct RecCtx {
    int d, H, npad, G, GH, u0, UG, ugp, tid, nthreads, ul, rb;
    int res;     // resident 32-k chunks of the R slice (the rest streams)
    bool r16;    // the streamed R rows are whole 16-byte pieces (copied 16 bytes at a time)
    bool active;
    bool live;   // this step: some row of the thread's tile has not finished
    float* Rs;   // resident [res * KC (or H)][ugp]
    float* Rring;// streamed chunks: ring [stages][KC][ugp]
    float* Hs;   // ring [stages][KC][npad]
};

// Issue the cp.async copies of k-chunk `chunk` into ring slot `slot`:
// src rows k0 .. k0+kc-1 of a [H][npad] matrix, and (if that chunk of R is
// not resident) the CTA's R columns for those rows.
__device__ __forceinline__ void issue_chunk(const RecParams& p, const RecCtx& x, const float* src,
                                            int chunk, int slot)
{
    const int k0 = chunk * kRecKC;
    const int kc = min(kRecKC, x.H - k0);
    const float* s = src + (size_t)k0 * x.npad;
    float* dst = x.Hs + (size_t)slot * kRecKC * x.npad;
    const int n4 = kc * x.npad / 4;
    for (int i = x.tid; i < n4; i += x.nthreads) cp_async16_cg(dst + 4 * i, s + 4 * i);
    if (chunk >= x.res) {
        const float* rs = p.Rt + ((size_t)x.d * x.H + k0) * x.GH + (size_t)x.u0 * x.G;
        float* rd = x.Rring + (size_t)slot * kRecKC * x.ugp;
        if (x.r16) {
            const int q = x.UG / 4;                 // 16-byte pieces per k-row
            const int tot = kc * q;
            for (int i = x.tid; i < tot; i += x.nthreads) {
                const int kk = i / q, j = i - kk * q;
                cp_async16_cg(rd + (size_t)kk * x.ugp + 4 * j, rs + (size_t)kk * x.GH + 4 * j);
            }
        } else {
            const int tot = kc * x.UG;
            for (int i = x.tid; i < tot; i += x.nthreads) {
                const int kk = i / x.UG, j = i - kk * x.UG;
                cp_async4_ca(rd + (size_t)kk * x.ugp + j, rs + (size_t)kk * x.GH + j);
            }
        }
    }
}

// acc[i][j] += sum_k src[k][row_i] * R[k][ul*G + col_off + j], k ascending,
// one accumulator per output; src is a [H][npad] matrix in global memory.
template <int TN, int NC, bool EXACT>
__device__ __forceinline__ void accumulate(const RecParams& p, const RecCtx& x, const float* src,
                                           int col_off, float (&acc)[TN][NC])
{
    const int nchunks = (x.H + kRecKC - 1) / kRecKC;
#pragma unroll
    for (int c = 0; c < kRecStages - 1; ++c) {
        if (c < nchunks) issue_chunk(p, x, src, c, c);
        cp_async_commit();
    }
    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<kRecStages - 2>();
        __syncthreads();
        const int nxt = c + kRecStages - 1;
        if (nxt < nchunks) issue_chunk(p, x, src, nxt, nxt % kRecStages);
        cp_async_commit();
        const int slot = c % kRecStages;
        const int k0 = c * kRecKC;
        const int kc = min(kRecKC, x.H - k0);
        if (x.active && x.live) {
            const float* hk = x.Hs + (size_t)slot * kRecKC * x.npad + x.rb * TN;
            const float* rk = (c < x.res ? x.Rs + (size_t)k0 * x.ugp
                                         : x.Rring + (size_t)slot * kRecKC * x.ugp) +
                              x.ul * x.G + col_off;
            if (kc == kRecKC) chunk_full<TN, NC, EXACT>(hk, x.npad, rk, x.ugp, acc);
            else chunk_part<TN, NC, EXACT>(hk, x.npad, rk, x.ugp, kc, acc);
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // ring slots free for the next product
}

template <bool EXACT>
__device__ __forceinline__ float act(const ActSpec& a, float v)
{
    return activation<EXACT>(a.fn, a.alpha, a.beta, v);
}

__device__ __forceinline__ float clipv(const RecParams& p, float v)
{
    if (!p.has_clip) return v;
    return v > p.clip ? p.clip : (v < -p.clip ? -p.clip : v);
}

__device__ __forceinline__ size_t y_index(const RecParams& p, int t, int d, int n, int u)
{
    return p.layout == 0 ? (((size_t)t * p.D + d) * p.N + n) * p.H + u
                         : (((size_t)n * p.S + t) * p.D + d) * p.H + u;
}

__device__ __forceinline__ size_t s_index(const RecParams& p, int d, int n, int u)
{
    return p.layout == 0 ? ((size_t)d * p.N + n) * p.H + u : ((size_t)n * p.D + d) * p.H + u;
}

// Eight rows per thread hold 32 LSTM accumulators plus two blocks of
// operands: up to 255 registers, so at most 256 threads per CTA.
template <int TN>
struct StagedBounds {
    static constexpr int threads = TN == 8 ? 256 : 512;
};

template <int OP, int TN, bool EXACT>
__global__ void __launch_bounds__(StagedBounds<TN>::threads, 1) rnn_recurrent_kernel(const RecParams p)
{
    constexpr int G = OP == 0 ? 1 : (OP == 1 ? 3 : 4);
    extern __shared__ __align__(16) float smem[];

    RecCtx x;
    const int C = p.ctas_per_dir;
    x.d = blockIdx.x / C;
    const int c = blockIdx.x - x.d * C;
    x.H = p.H;
    x.npad = p.npad;
    x.G = G;
    x.GH = G * p.H;
    x.u0 = (int)(((long long)c * p.H) / C);
    const int u1 = (int)(((long long)(c + 1) * p.H) / C);
    const int U = u1 - x.u0;
    x.UG = U * G;
    x.ugp = rec_ugp(p.umax, G);
    x.tid = threadIdx.x;
    x.nthreads = blockDim.x;
    x.ul = x.tid % p.umax;
    x.rb = x.tid / p.umax;
    x.active = (x.ul < U) && (x.rb * TN < p.N);
    x.live = true;
    const int nchunks = (p.H + kRecKC - 1) / kRecKC;
    x.res = p.r_resident ? nchunks : min(p.res_chunks, nchunks);
    x.r16 = ((x.u0 * G) % 4 == 0) && (x.UG % 4 == 0) && (x.GH % 4 == 0);
    x.Rs = smem;
    x.Rring = smem + (x.res >= nchunks ? (size_t)p.H * x.ugp : (size_t)x.res * kRecKC * x.ugp);
    x.Hs = x.Rring + (x.res >= nchunks ? 0 : (size_t)kRecStages * kRecKC * x.ugp);

    const int d = x.d;
    const int u = x.u0 + x.ul;
    const int N = p.N;
    const bool rev = p.dir_reverse[d] != 0;
    unsigned* bar = p.bar + d;

    if (x.res > 0) {
        const float* src = p.Rt + (size_t)d * p.H * x.GH + (size_t)x.u0 * G;
        const int tot = min(p.H, x.res * kRecKC) * x.UG;
        for (int i = x.tid; i < tot; i += x.nthreads) {
            const int k = i / x.UG, j = i - k * x.UG;
            x.Rs[(size_t)k * x.ugp + j] = src[(size_t)k * x.GH + j];
        }
        // made visible by the __syncthreads inside accumulate()
    }

    // Per-thread constants and state.
    const ActSpec fA = p.act[d][0], gA = p.act[d][1], hA = p.act[d][2];
    float wb[G], rbv[G];
    float pI = 0.f, pO = 0.f, pF = 0.f;
    float hown[TN], cown[TN], xw[TN][G];
    int len[TN];
#pragma unroll
    for (int g = 0; g < G; ++g) { wb[g] = 0.f; rbv[g] = 0.f; }
    if (x.active) {
        if (p.has_B) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                wb[g] = p.B[(size_t)d * 2 * x.GH + (size_t)g * p.H + u];
                rbv[g] = p.B[(size_t)d * 2 * x.GH + x.GH + (size_t)g * p.H + u];
            }
        }
        if (OP == 2 && p.has_P) {
            pI = p.P[(size_t)d * 3 * p.H + u];
            pO = p.P[(size_t)d * 3 * p.H + p.H + u];
            pF = p.P[(size_t)d * 3 * p.H + 2 * p.H + u];
        }
    }
    // Rows: the exchange buffers use the internal row index r = rb*TN + i;
    // with sequence_lens the rows are sorted by length (longest first, so a
    // tile whose first row has finished has finished altogether) and rown[i]
    // is the caller's row behind r.
    int rown[TN];
    int tile_len = 0;
#pragma unroll
    for (int i = 0; i < TN; ++i) {
        const int r = x.rb * TN + i;
        const bool ok = x.active && r < N;
        rown[i] = ok ? (p.perm ? p.perm[r] : r) : 0;
        len[i] = ok ? (p.has_lens ? p.lens[rown[i]] : p.S) : 0;
        tile_len = len[i] > tile_len ? len[i] : tile_len;
        hown[i] = (ok && p.has_h0) ? io_load(p.h0, s_index(p, d, rown[i], u), p.io) : 0.f;
        cown[i] = (ok && OP == 2 && p.has_c0) ? io_load(p.c0, s_index(p, d, rown[i], u), p.io) : 0.f;
    }

    const size_t xw_ld = (size_t)p.D * x.GH;
    const size_t xw_col = (size_t)d * x.GH + (size_t)u * G;
    auto load_xw = [&](int s) {
#pragma unroll
        for (int i = 0; i < TN; ++i) {
            const int n = rown[i];
            if (x.active && x.rb * TN + i < N && s < len[i]) {
                const int t = rev ? len[i] - 1 - s : s;
                const size_t row = p.layout == 0 ? (size_t)t * N + n : (size_t)n * p.S + t;
                const float* q = p.XW + row * xw_ld + xw_col;
#pragma unroll
                for (int g = 0; g < G; ++g) xw[i][g] = __ldg(q + g);
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) xw[i][g] = 0.f;
            }
        }
    };

    unsigned episode = 0;
    load_xw(0);
    for (int s = 0; s < p.max_len; ++s) {
        const float* hsrc = p.hbuf + ((size_t)(d * 2 + (s & 1)) * p.H) * x.npad;
        float* hdst = p.hbuf + ((size_t)(d * 2 + ((s + 1) & 1)) * p.H) * x.npad;
        float xc[TN][G];
#pragma unroll
        for (int i = 0; i < TN; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g) xc[i][g] = xw[i][g];
        x.live = s < tile_len;   // a finished tile skips its products (its rows stay frozen)

        if constexpr (OP == 1) {
            if (p.lbr == 0) {
                // z and r from H.R^T, then the candidate's product over r (.) H.
                float az[TN][2];
#pragma unroll
                for (int i = 0; i < TN; ++i) { az[i][0] = 0.f; az[i][1] = 0.f; }
                accumulate<TN, 2, EXACT>(p, x, hsrc, 0, az);
                if (s + 1 < p.max_len) load_xw(s + 1);
                float zg[TN];
                float* rh = p.rhbuf + (size_t)d * 2 * p.H * x.npad;
#pragma unroll
                for (int i = 0; i < TN; ++i) {
                    const int n = x.rb * TN + i;   // internal row (exchange buffers)
                    zg[i] = 0.f;
                    if (!(x.active && n < N)) continue;
                    float rhv = 0.f;
                    if (s < len[i]) {
                        float pz = fadd(xc[i][0], az[i][0]);
                        float pr = fadd(xc[i][1], az[i][1]);
                        if (p.has_B) {
                            pz = fadd(pz, wb[0]); pz = fadd(pz, rbv[0]);
                            pr = fadd(pr, wb[1]); pr = fadd(pr, rbv[1]);
                        }
                        zg[i] = act<EXACT>(fA, clipv(p, pz));
                        const float r = act<EXACT>(fA, clipv(p, pr));
                        rhv = fmul(r, hown[i]);
                    }
                    rh[(size_t)u * x.npad + n] = rhv;
                }
                ++episode;
                if (!step_barrier(bar, episode * C, p.status, p.spin_limit_ns,
                                  !(episode == 1 && p.debug_skip_cta == (int)blockIdx.x), C))
                    return;
                float ah[TN][1];
#pragma unroll
                for (int i = 0; i < TN; ++i) ah[i][0] = 0.f;
                accumulate<TN, 1, EXACT>(p, x, rh, 2, ah);
#pragma unroll
                for (int i = 0; i < TN; ++i) {
                    const int n = x.rb * TN + i;   // internal row (exchange buffers)
                    const int nr = rown[i];        // the caller's row
                    if (!(x.active && n < N)) continue;
                    if (s < len[i]) {
                        const int t = rev ? len[i] - 1 - s : s;
                        float ph = fadd(xc[i][2], ah[i][0]);
                        if (p.has_B) { ph = fadd(ph, wb[2]); ph = fadd(ph, rbv[2]); }
                        const float ht = act<EXACT>(gA, clipv(p, ph));
                        const float hn = fadd(fmul(fsub(1.0f, zg[i]), ht), fmul(zg[i], hown[i]));
                        hown[i] = hn;
                        if (p.Y) io_store(p.Y, y_index(p, t, d, nr, u), canon_nan(hn), p.io);
                    } else if (p.Y) {
                        io_store(p.Y, y_index(p, s, d, nr, u), 0.f, p.io);
                    }
                    hdst[(size_t)u * x.npad + n] = hown[i];
                }
                ++episode;
                if (!step_barrier(bar, episode * C, p.status, p.spin_limit_ns, true, C)) return;
                continue;
            }
        }

        float acc[TN][G];
#pragma unroll
        for (int i = 0; i < TN; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g) acc[i][g] = 0.f;
        accumulate<TN, G, EXACT>(p, x, hsrc, 0, acc);
        if (s + 1 < p.max_len) load_xw(s + 1);

#pragma unroll
        for (int i = 0; i < TN; ++i) {
            const int n = x.rb * TN + i;   // internal row (exchange buffers)
            const int nr = rown[i];        // the caller's row
            if (!(x.active && n < N)) continue;
            if (s < len[i]) {
                const int t = rev ? len[i] - 1 - s : s;
                float hn;
                float pre[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    pre[g] = fadd(xc[i][g], acc[i][g]);
                    if (p.has_B) { pre[g] = fadd(pre[g], wb[g]); pre[g] = fadd(pre[g], rbv[g]); }
                }
                if constexpr (OP == 0) {
                    hn = act<EXACT>(fA, clipv(p, pre[0]));
                } else if constexpr (OP == 1) {
                    // linear_before_reset = 1: pre_h = (xw_h + r*(rec_h + Rbh)) + Wbh
                    const float z = act<EXACT>(fA, clipv(p, pre[0]));
                    const float r = act<EXACT>(fA, clipv(p, pre[1]));
                    float ph;
                    if (p.has_B) ph = fadd(fadd(xc[i][2], fmul(r, fadd(acc[i][2], rbv[2]))), wb[2]);
                    else ph = fadd(xc[i][2], fmul(r, acc[i][2]));
                    const float ht = act<EXACT>(gA, clipv(p, ph));
                    hn = fadd(fmul(fsub(1.0f, z), ht), fmul(z, hown[i]));
                } else {
                    // LSTM gate columns i, o, f, c
                    float pi = pre[0], po = pre[1], pf = pre[2];
                    const float pc = pre[3];
                    if (p.has_P) {
                        pi = fadd(pi, fmul(pI, cown[i]));
                        pf = fadd(pf, fmul(pF, cown[i]));
                    }
                    const float ig = act<EXACT>(fA, clipv(p, pi));
                    const float fg = p.input_forget ? fsub(1.0f, ig) : act<EXACT>(fA, clipv(p, pf));
                    const float ct = act<EXACT>(gA, clipv(p, pc));
                    const float cn = fadd(fmul(fg, cown[i]), fmul(ig, ct));
                    if (p.has_P) po = fadd(po, fmul(pO, cn));
                    const float og = act<EXACT>(fA, clipv(p, po));
                    hn = fmul(og, act<EXACT>(hA, cn));
                    cown[i] = cn;
                }
                hown[i] = hn;
                if (p.Y) io_store(p.Y, y_index(p, t, d, nr, u), canon_nan(hn), p.io);
            } else if (p.Y) {
                io_store(p.Y, y_index(p, s, d, nr, u), 0.f, p.io);
            }
            hdst[(size_t)u * x.npad + n] = hown[i];
        }
        ++episode;
        if (!step_barrier(bar, episode * C, p.status, p.spin_limit_ns,
                          !(episode == 1 && p.debug_skip_cta == (int)blockIdx.x), C))
            return;
    }

#pragma unroll
    for (int i = 0; i < TN; ++i) {
        const int n = x.rb * TN + i;
        if (!(x.active && n < N)) continue;
        const size_t si = s_index(p, d, rown[i], u);
        if (p.Yh) io_store(p.Yh, si, len[i] > 0 ? canon_nan(hown[i]) : 0.f, p.io);
        if (OP == 2 && p.Yc) io_store(p.Yc, si, len[i] > 0 ? canon_nan(cown[i]) : 0.f, p.io);
    }
}

// Select the instance for rows-per-thread and mode, set its shared-memory
// limit and launch it cooperatively (all CTAs co-resident).
template <int OP>
cudaError_t launch_recurrent_op(const RecParams& p, bool exact, int threads, size_t smem,
                                cudaStream_t stream)
{
    const void* fn = nullptr;
    switch (p.rows_per_thread * 2 + (exact ? 1 : 0)) {
    case 2: fn = (const void*)rnn_recurrent_kernel<OP, 1, false>; break;
    case 3: fn = (const void*)rnn_recurrent_kernel<OP, 1, true>; break;
    case 4: fn = (const void*)rnn_recurrent_kernel<OP, 2, false>; break;
    case 5: fn = (const void*)rnn_recurrent_kernel<OP, 2, true>; break;
    case 8: fn = (const void*)rnn_recurrent_kernel<OP, 4, false>; break;
    case 9: fn = (const void*)rnn_recurrent_kernel<OP, 4, true>; break;
    case 16: fn = (const void*)rnn_recurrent_kernel<OP, 8, false>; break;
    case 17: fn = (const void*)rnn_recurrent_kernel<OP, 8, true>; break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {(void*)&p};
    return cudaLaunchCooperativeKernel(fn, dim3(p.D * p.ctas_per_dir), dim3(threads), args, smem,
                                       stream);
}

template <int OP>
cudaError_t recurrent_occupancy_op(int rows_per_thread, bool exact, int threads, size_t smem,
                                   int* blocks)
{
    const void* fn = nullptr;
    switch (rows_per_thread * 2 + (exact ? 1 : 0)) {
    case 2: fn = (const void*)rnn_recurrent_kernel<OP, 1, false>; break;
    case 3: fn = (const void*)rnn_recurrent_kernel<OP, 1, true>; break;
    case 4: fn = (const void*)rnn_recurrent_kernel<OP, 2, false>; break;
    case 5: fn = (const void*)rnn_recurrent_kernel<OP, 2, true>; break;
    case 8: fn = (const void*)rnn_recurrent_kernel<OP, 4, false>; break;
    case 9: fn = (const void*)rnn_recurrent_kernel<OP, 4, true>; break;
    case 16: fn = (const void*)rnn_recurrent_kernel<OP, 8, false>; break;
    case 17: fn = (const void*)rnn_recurrent_kernel<OP, 8, true>; break;
    default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, smem);
}

}  // namespace rnngb
