// Stacked layers in one persistent launch: the wavefront.
//
// Page "Recurrent operators: RNN, GRU, LSTM", Computation: a layer is the
// input projection XW = X.W^T over all steps followed by the per-step
// recurrent product and the gate arithmetic.  In a stack of unidirectional
// layers that walk time the same way, layer l+1's input at its step s is
// layer l's h after layer l's step s (X_{l+1}[t] = Y_l[t] for the row's
// t of step s), so layer l+1 can take step s as soon as layer l has, while
// layer l goes on with step s+1.  This kernel runs every layer of such a
// stack at once: the SMs are split between the layers, and a CTA of layer
// l >= 1 computes its input product for the step itself (one accumulator
// per output, k increasing from +0: the same sum, rounded the same way, as
// the projection GEMM gives), so the layers overlap step by step instead of
// running one after another.  Layer 0's input product is the projection
// GEMM, computed for all steps before this launch.
//
// Work split inside a layer: the staged kernel's (k_recur.cuh).  CTA c of
// layer l owns hidden units [u0, u1) and all G gate columns of each, for
// every batch row; thread (rb, ul) owns unit u0 + ul of rows rb*TN ..
// rb*TN + TN - 1, keeps its gate sums and its cell state in registers, and
// the layer's slices of R (and, from layer 1 on, of W) stay resident in
// shared memory.  h moves through a ring of kWaveRing k-major buffers
// hbuf[ring][H][npad] per layer (rows ranked by length when sequence_lens
// is given): the next layer reads its input from the same buffers.
//
// Synchronisation: one monotonic arrival counter per layer; a CTA adds 1
// (release, after a CTA barrier) when its h of a step is written, twice per
// step for GRU with linear_before_reset = 0 (r (.) h, then h).  Layer l at
// step s waits (acquire polls, all bounded by the global timer) for
//   - its own layer's step s-1 (every CTA has written h(s-1));
//   - layer l-1's step s (its input), before the input product;
//   - layer l+1's step s+1-kWaveRing, before overwriting the ring buffer
//     that step read.
// Every wait is bounded: a CTA that gives up records RNN_ERR_TIMEOUT in the
// status word; CTAs that see a non-zero status leave at their next wait.
#pragma once

#include "k_recur.cuh"

namespace rnngb {

// Bounded wait until *ctr >= target (thread 0 polls, the CTA waits at a
// barrier).  Returns false when the run is being abandoned.
__device__ __forceinline__ bool wave_wait(const unsigned* ctr, unsigned target, int* status, long long limit_ns)
{
    __shared__ int s_ok;
    __syncthreads();   // every thread has read the previous wait's flag
    if (threadIdx.x == 0) {
        int ok = 1;
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

// Every thread of the CTA has written its part; one release add publishes it.
__device__ __forceinline__ void wave_arrive(unsigned* ctr, bool skip)
{
    __syncthreads();
    if (threadIdx.x == 0 && !skip) {
        __threadfence();
        red_release_add_u32(ctr, 1u);
    }
}

// acc[i][j] += sum_k src[k][row_i] * Rs[k][ul*G + col + j], k ascending, one
// accumulator per output: src is a k-major [K][npad] matrix in global memory,
// streamed through the CTA's cp.async ring Hs; Rs is a resident k-major
// [K][ugp] slice in shared memory.
template <int TN, int NC, bool EXACT>
__device__ __forceinline__ void wave_product(const float* src, int K, int npad, const float* Rs, int ugp, int G,
                                             int col, float* Hs, int rb, int ul, bool compute,
                                             float (&acc)[TN][NC])
{
    const int nchunks = (K + kRecKC - 1) / kRecKC;
    const int tid = threadIdx.x, nthreads = blockDim.x;
    auto issue = [&](int c, int slot) {
        const int k0 = c * kRecKC;
        const int kc = min(kRecKC, K - k0);
        const float* s = src + (size_t)k0 * npad;
        float* dst = Hs + (size_t)slot * kRecKC * npad;
        const int n4 = kc * npad / 4;
        for (int i = tid; i < n4; i += nthreads) cp_async16_cg(dst + 4 * i, s + 4 * i);
    };
#pragma unroll
    for (int c = 0; c < kRecStages - 1; ++c) {
        if (c < nchunks) issue(c, c);
        cp_async_commit();
    }
    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<kRecStages - 2>();
        __syncthreads();
        const int nxt = c + kRecStages - 1;
        if (nxt < nchunks) issue(nxt, nxt % kRecStages);
        cp_async_commit();
        const int slot = c % kRecStages;
        const int k0 = c * kRecKC;
        const int kc = min(kRecKC, K - k0);
        if (compute) {
            const float* hk = Hs + (size_t)slot * kRecKC * npad + rb * TN;
            const float* rk = Rs + (size_t)k0 * ugp + ul * G + col;
            if (kc == kRecKC) chunk_full<TN, NC, EXACT>(hk, npad, rk, ugp, acc);
            else chunk_part<TN, NC, EXACT>(hk, npad, rk, ugp, kc, acc);
        }
    }
    cp_async_wait<0>();
    __syncthreads();   // ring slots free for the next product
}

template <int OP, int TN, bool EXACT>
__global__ void __launch_bounds__(512, 1) rnn_wavefront_kernel(const __grid_constant__ WaveParams p)
{
    constexpr int G = OP == 0 ? 1 : (OP == 1 ? 3 : 4);
    extern __shared__ __align__(16) float smem[];

    int l = 0;
    while (l + 1 < p.L && (int)blockIdx.x >= p.layer[l + 1].cta0) ++l;
    const WaveLayer& ly = p.layer[l];
    const int C = ly.C;
    const int c = (int)blockIdx.x - ly.cta0;
    const int H = p.H, N = p.N, npad = p.npad;
    const int GH = G * H;
    const int u0 = (int)(((long long)c * H) / C);
    const int U = (int)(((long long)(c + 1) * H) / C) - u0;
    const int UG = U * G;
    const int ugp = ly.ugp;
    const int tid = threadIdx.x;
    const int ul = tid % ly.umax;
    const int rb = tid / ly.umax;
    const bool active = ul < U && rb * TN < N;
    const int u = u0 + ul;
    const bool rev = p.reverse != 0;
    const bool two = OP == 1 && ly.lbr == 0;           // GRU: r (.) h published mid-step
    const int K_in = ly.I;                              // layers >= 1: the previous layer's hidden size

    // shared memory: R slice [H][ugp], W slice [K_in][ugp], h ring
    float* Rs = smem;
    float* Ws = Rs + (size_t)H * ugp;
    float* Hs = Ws + (size_t)K_in * ugp;
    {
        const float* rsrc = ly.Rt + (size_t)u0 * G;
        for (int i = tid; i < H * UG; i += blockDim.x) {
            const int k = i / UG, j = i - k * UG;
            Rs[(size_t)k * ugp + j] = rsrc[(size_t)k * GH + j];
        }
        if (K_in > 0) {
            const float* wsrc = ly.Wt + (size_t)u0 * G;
            for (int i = tid; i < K_in * UG; i += blockDim.x) {
                const int k = i / UG, j = i - k * UG;
                Ws[(size_t)k * ugp + j] = wsrc[(size_t)k * GH + j];
            }
        }
        // made visible by the barriers inside wave_product
    }

    const ActSpec fA = ly.act[0], gA = ly.act[1], hA = ly.act[2];
    float wb[G], rbv[G];
    float pI = 0.f, pO = 0.f, pF = 0.f;
#pragma unroll
    for (int g = 0; g < G; ++g) { wb[g] = 0.f; rbv[g] = 0.f; }
    if (active) {
        if (ly.has_B) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                wb[g] = ly.B[(size_t)g * H + u];
                rbv[g] = ly.B[(size_t)GH + (size_t)g * H + u];
            }
        }
        if (OP == 2 && ly.has_P) {
            pI = ly.P[u];
            pO = ly.P[(size_t)H + u];
            pF = ly.P[(size_t)2 * H + u];
        }
    }
    // rows: internal row r = rb*TN + i in the exchange buffers, the caller's
    // row rown[i] = perm[r] (rows by length, longest first) everywhere else
    float hown[TN], cown[TN];
    int len[TN], rown[TN];
    int tile_len = 0;
#pragma unroll
    for (int i = 0; i < TN; ++i) {
        const int r = rb * TN + i;
        const bool ok = active && r < N;
        rown[i] = ok ? (p.perm ? p.perm[r] : r) : 0;
        len[i] = ok ? (p.has_lens ? p.lens[rown[i]] : p.S) : 0;
        tile_len = len[i] > tile_len ? len[i] : tile_len;
        const size_t si = (size_t)rown[i] * H + u;        // [1, N, H] and [N, 1, H] alike
        hown[i] = (ok && ly.has_h0) ? ly.h0[si] : 0.f;
        cown[i] = (ok && OP == 2 && ly.has_c0) ? ly.c0[si] : 0.f;
    }
    auto step_time = [&](int s, int i) { return rev ? len[i] - 1 - s : s; };
    // clip (when present: gate inputs to [-clip, clip], a NaN passing), then the activation
    const bool has_clip = ly.has_clip != 0;
    const float cl = ly.clip;
    auto clip = [&](float v) { return has_clip ? (v > cl ? cl : (v < -cl ? -cl : v)) : v; };
    auto act = [&](const ActSpec& a, float v) { return activation<EXACT>(a.fn, a.alpha, a.beta, v); };
    auto y_at = [&](int t, int n) {
        return p.layout == 0 ? ((size_t)t * N + n) * H + u : ((size_t)n * p.S + t) * H + u;
    };

    const size_t ring = (size_t)H * npad;
    const unsigned A = two ? 2u : 1u;                   // arrivals per step of this layer
    auto arrivals = [&](int layer) { return (OP == 1 && p.layer[layer].lbr == 0) ? 2u : 1u; };
    unsigned* bar = p.bar + l;
    const bool skip_first = p.debug_skip_cta == (int)blockIdx.x;

    for (int s = 0; s < p.max_len; ++s) {
        const bool live = s < tile_len;                 // a finished row tile skips its products
        const float* hsrc = ly.hbuf + (size_t)(s % kWaveRing) * ring;
        float* hdst = ly.hbuf + (size_t)((s + 1) % kWaveRing) * ring;
        // this layer's step s-1 is complete (h(s-1) written by every CTA; a
        // layer of one CTA has its own barrier behind it already)
        if (s > 0 && C > 1 && !wave_wait(bar, A * (unsigned)C * (unsigned)s, p.status, p.spin_limit_ns)) return;

        // the input part of the gate sums: XW (layer 0) or the product over
        // the previous layer's h after its step s (layers >= 1)
        float xg[TN][G];
#pragma unroll
        for (int i = 0; i < TN; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g) xg[i][g] = 0.f;
        // (GRU lbr = 0: z and r first, then the candidate after r (.) h)
        float acc[TN][G];
#pragma unroll
        for (int i = 0; i < TN; ++i)
#pragma unroll
            for (int g = 0; g < G; ++g) acc[i][g] = 0.f;
        if (two) {
            float az[TN][2];
#pragma unroll
            for (int i = 0; i < TN; ++i) { az[i][0] = 0.f; az[i][1] = 0.f; }
            wave_product<TN, 2, EXACT>(hsrc, H, npad, Rs, ugp, G, 0, Hs, rb, ul, active && live, az);
#pragma unroll
            for (int i = 0; i < TN; ++i) { acc[i][0] = az[i][0]; acc[i][1] = az[i][1]; }
        } else {
            wave_product<TN, G, EXACT>(hsrc, H, npad, Rs, ugp, G, 0, Hs, rb, ul, active && live, acc);
        }
        if (l > 0) {
            const WaveLayer& prev = p.layer[l - 1];
            const unsigned need = arrivals(l - 1) * (unsigned)prev.C * (unsigned)(s + 1);
            if (!wave_wait(p.bar + l - 1, need, p.status, p.spin_limit_ns)) return;
            const float* xsrc = prev.hbuf + (size_t)((s + 1) % kWaveRing) * ((size_t)K_in * npad);
            wave_product<TN, G, EXACT>(xsrc, K_in, npad, Ws, ugp, G, 0, Hs, rb, ul, active && live, xg);
        } else {
#pragma unroll
            for (int i = 0; i < TN; ++i) {
                if (active && rb * TN + i < N && s < len[i]) {
                    const int t = step_time(s, i);
                    const size_t row = p.layout == 0 ? (size_t)t * N + rown[i] : (size_t)rown[i] * p.S + t;
                    const float* q = ly.XW + row * GH + (size_t)u * G;
#pragma unroll
                    for (int g = 0; g < G; ++g) xg[i][g] = __ldg(q + g);
                }
            }
        }
        // the next layer has read the ring buffer this step overwrites
        if (l + 1 < p.L && s + 2 - kWaveRing > 0) {
            const WaveLayer& next = p.layer[l + 1];
            const unsigned need = arrivals(l + 1) * (unsigned)next.C * (unsigned)(s + 2 - kWaveRing);
            if (!wave_wait(p.bar + l + 1, need, p.status, p.spin_limit_ns)) return;
        }

        if (two) {
            // z and r, then r (.) h for every unit of the layer before the
            // candidate's product (page: Computation, GRU with
            // linear_before_reset = 0)
            float zg[TN];
#pragma unroll
            for (int i = 0; i < TN; ++i) {
                const int r = rb * TN + i;
                zg[i] = 0.f;
                if (!(active && r < N)) continue;
                float rhv = 0.f;
                if (s < len[i]) {
                    float pz = fadd(xg[i][0], acc[i][0]);
                    float pr = fadd(xg[i][1], acc[i][1]);
                    if (ly.has_B) {
                        pz = fadd(pz, wb[0]); pz = fadd(pz, rbv[0]);
                        pr = fadd(pr, wb[1]); pr = fadd(pr, rbv[1]);
                    }
                    zg[i] = act(fA, clip(pz));
                    const float rg = act(fA, clip(pr));
                    rhv = fmul(rg, hown[i]);
                }
                ly.rhbuf[(size_t)u * npad + r] = rhv;
            }
            wave_arrive(bar, skip_first && s == 0);
            if (C > 1 && !wave_wait(bar, A * (unsigned)C * (unsigned)s + (unsigned)C, p.status, p.spin_limit_ns))
                return;
            if (C == 1) __syncthreads();
            float ah[TN][1];
#pragma unroll
            for (int i = 0; i < TN; ++i) ah[i][0] = 0.f;
            wave_product<TN, 1, EXACT>(ly.rhbuf, H, npad, Rs, ugp, G, 2, Hs, rb, ul, active && live, ah);
#pragma unroll
            for (int i = 0; i < TN; ++i) {
                const int r = rb * TN + i;
                if (!(active && r < N)) continue;
                if (s < len[i]) {
                    const int t = step_time(s, i);
                    float ph = fadd(xg[i][2], ah[i][0]);
                    if (ly.has_B) { ph = fadd(ph, wb[2]); ph = fadd(ph, rbv[2]); }
                    const float ht = act(gA, clip(ph));
                    const float hn = fadd(fmul(fsub(1.0f, zg[i]), ht), fmul(zg[i], hown[i]));
                    hown[i] = hn;
                    if (ly.Y) ly.Y[y_at(t, rown[i])] = canon_nan(hn);
                } else if (ly.Y) {
                    ly.Y[y_at(s, rown[i])] = 0.f;
                }
                hdst[(size_t)u * npad + r] = hown[i];
            }
            wave_arrive(bar, false);
            continue;
        }

#pragma unroll
        for (int i = 0; i < TN; ++i) {
            const int r = rb * TN + i;
            if (!(active && r < N)) continue;
            if (s < len[i]) {
                const int t = step_time(s, i);
                float pre[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    pre[g] = fadd(xg[i][g], acc[i][g]);
                    if (ly.has_B) { pre[g] = fadd(pre[g], wb[g]); pre[g] = fadd(pre[g], rbv[g]); }
                }
                float hn;
                if constexpr (OP == 0) {
                    hn = act(fA, clip(pre[0]));
                } else if constexpr (OP == 1) {
                    // linear_before_reset = 1: pre_h = (xw_h + r*(rec_h + Rbh)) + Wbh
                    const float z = act(fA, clip(pre[0]));
                    const float rg = act(fA, clip(pre[1]));
                    float ph;
                    if (ly.has_B) ph = fadd(fadd(xg[i][2], fmul(rg, fadd(acc[i][2], rbv[2]))), wb[2]);
                    else ph = fadd(xg[i][2], fmul(rg, acc[i][2]));
                    const float ht = act(gA, clip(ph));
                    hn = fadd(fmul(fsub(1.0f, z), ht), fmul(z, hown[i]));
                } else {
                    // LSTM gate columns i, o, f, c
                    float pi = pre[0], po = pre[1], pf = pre[2];
                    const float pc = pre[3];
                    if (ly.has_P) {
                        pi = fadd(pi, fmul(pI, cown[i]));
                        pf = fadd(pf, fmul(pF, cown[i]));
                    }
                    const float ig = act(fA, clip(pi));
                    const float fg = ly.input_forget ? fsub(1.0f, ig) : act(fA, clip(pf));
                    const float ct = act(gA, clip(pc));
                    const float cn = fadd(fmul(fg, cown[i]), fmul(ig, ct));
                    if (ly.has_P) po = fadd(po, fmul(pO, cn));
                    const float og = act(fA, clip(po));
                    hn = fmul(og, act(hA, cn));
                    cown[i] = cn;
                }
                hown[i] = hn;
                if (ly.Y) ly.Y[y_at(t, rown[i])] = canon_nan(hn);
            } else if (ly.Y) {
                ly.Y[y_at(s, rown[i])] = 0.f;
            }
            hdst[(size_t)u * npad + r] = hown[i];
        }
        wave_arrive(bar, skip_first && s == 0);
    }

#pragma unroll
    for (int i = 0; i < TN; ++i) {
        const int r = rb * TN + i;
        if (!(active && r < N)) continue;
        const size_t si = (size_t)rown[i] * H + u;
        if (ly.Yh) ly.Yh[si] = len[i] > 0 ? canon_nan(hown[i]) : 0.f;
        if (OP == 2 && ly.Yc) ly.Yc[si] = len[i] > 0 ? canon_nan(cown[i]) : 0.f;
    }
}

template <int OP>
const void* wavefront_kernel_ptr(int tn, bool exact)
{
    switch (tn * 2 + (exact ? 1 : 0)) {
    case 2: return (const void*)rnn_wavefront_kernel<OP, 1, false>;
    case 3: return (const void*)rnn_wavefront_kernel<OP, 1, true>;
    case 4: return (const void*)rnn_wavefront_kernel<OP, 2, false>;
    case 5: return (const void*)rnn_wavefront_kernel<OP, 2, true>;
    case 8: return (const void*)rnn_wavefront_kernel<OP, 4, false>;
    case 9: return (const void*)rnn_wavefront_kernel<OP, 4, true>;
    default: return nullptr;
    }
}

template <int OP>
cudaError_t launch_wavefront_op(const WaveParams& p, bool exact, int tn, int ctas, int threads, size_t smem,
                                cudaStream_t stream)
{
    const void* fn = wavefront_kernel_ptr<OP>(tn, exact);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {(void*)&p};
    return cudaLaunchCooperativeKernel(fn, dim3(ctas), dim3(threads), args, smem, stream);
}

template <int OP>
cudaError_t wavefront_occupancy_op(int tn, bool exact, int threads, size_t smem, int* blocks)
{
    const void* fn = wavefront_kernel_ptr<OP>(tn, exact);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, smem);
}

}  // namespace rnngb
