// Small bandwidth-bound kernels around the two products.
//   pack        W and R transposed to k-major with gate-interleaved columns
//               (page "Recurrent operators: RNN, GRU, LSTM", Computation:
//               weights are transposed once per plan when constant, otherwise
//               on each run into scratch);
//   state_init  the first h exchange buffer from initial_h (omitted inputs
//               are zeros: Choices the specification leaves open);
//   mask_tail   Y = 0 at the steps no row reaches (sequence_lens: Y is zero
//               at t >= len).
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "io_types.cuh"
#include "rnn_internal.h"

namespace rnngb {

namespace {

// dst[k][dst_col0 + u*G + g] = src[g*H + u][k] for one direction.
__global__ void pack_kernel(const float* __restrict__ src, float* __restrict__ dst, int G, int64_t H,
                            int64_t K, int64_t dst_ld, int64_t dst_col0)
{
    __shared__ float tile[32][33];
    const int64_t GH = (int64_t)G * H;
    const int64_t c0 = (int64_t)blockIdx.x * 32;   // packed column tile
    const int64_t k0 = (int64_t)blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    for (int j = ty; j < 32; j += 8) {
        const int64_t cp = c0 + j;
        const int64_t k = k0 + tx;
        if (cp < GH && k < K) {
            const int64_t u = cp / G, g = cp - u * G;
            tile[j][tx] = src[(g * H + u) * K + k];
        }
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int64_t k = k0 + j;
        const int64_t cp = c0 + tx;
        if (k < K && cp < GH) dst[k * dst_ld + dst_col0 + cp] = tile[tx][j];
    }
}

// Exchange buffers at the start of a run.  Staged kernel: hbuf[d][b][u][n]
// (k-major).  Dataflow kernel: hbuf[d][b][cr][u / 32][rl][u % 32] with rows
// of 36 floats (row n = cr*npad + rl).  Buffer 0 starts as initial_h (or 0);
// buffer 1, padding rows and columns and rhbuf start as 0; barrier counters
// and flags 0.
__global__ void state_init_kernel(const RecParams p)
{
    const bool df = p.kernel == 2;
    const int64_t CR = p.row_groups;
    const int64_t W = df ? (int64_t)p.hpad / kRecKC * kDfPitch : p.H;   // floats per row (all chunks)
    const int64_t blk = (int64_t)p.npad * W;              // one row group's block
    const int64_t total = (int64_t)p.D * CR * blk;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t u, rl;
        if (df) {
            const int64_t e = i % blk, chunk = e / ((int64_t)p.npad * kDfPitch);
            const int64_t r = e % ((int64_t)p.npad * kDfPitch);
            rl = r / kDfPitch;
            const int64_t col = r % kDfPitch;
            u = col < kRecKC ? chunk * kRecKC + col : p.H;   // pitch padding: never a unit
        }
        else { rl = i % p.npad; u = (i / p.npad) % p.H; }
        const int64_t cr = (i / blk) % CR;
        const int64_t d = i / (blk * CR);
        const int64_t n = cr * p.npad + rl;
        float v = 0.0f;
        if (n < p.N && u < p.H && p.h0) {
            const int64_t nr = p.perm ? p.perm[n] : n;    // the caller's row behind internal row n
            const int64_t si = p.layout == 0 ? (d * p.N + nr) * p.H + u : (nr * p.D + d) * p.H + u;
            v = io_load(p.h0, si, p.io);
        }
        const int64_t off = i - d * CR * blk;             // offset inside direction d
        p.hbuf[(d * 2) * CR * blk + off] = v;
        p.hbuf[(d * 2 + 1) * CR * blk + off] = 0.0f;
        if (p.rhbuf) {
            p.rhbuf[(d * 2) * CR * blk + off] = 0.0f;
            p.rhbuf[(d * 2 + 1) * CR * blk + off] = 0.0f;
        }
    }
    if (blockIdx.x == 0) {
        if (threadIdx.x < p.D) p.bar[threadIdx.x] = 0u;
        const int nflags = p.D * p.row_groups;
        for (int j = threadIdx.x; j < nflags && p.flags; j += blockDim.x) p.flags[j] = 0u;
    }
}

// Wavefront kernel: every layer's ring buffer 0 = initial_h (rows through
// perm) or 0, the other ring buffers and r (.) h 0; the arrival counters 0.
__global__ void wave_state_init_kernel(const WaveParams p)
{
    const int64_t blk = (int64_t)p.H * p.npad;           // one [H][npad] buffer
    const int64_t per_layer = (int64_t)kWaveRing * blk;
    const int64_t total = (int64_t)p.L * per_layer;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int l = (int)(i / per_layer);
        const int64_t off = i - (int64_t)l * per_layer;
        const int64_t buf = off / blk;
        const int64_t e = off - buf * blk;
        const int64_t u = e / p.npad, n = e % p.npad;
        const WaveLayer& ly = p.layer[l];
        float v = 0.0f;
        if (buf == 0 && n < p.N && ly.h0) {
            const int64_t nr = p.perm ? p.perm[n] : n;
            v = ly.h0[nr * p.H + u];
        }
        ly.hbuf[off] = v;
        if (buf == 0 && ly.rhbuf) ly.rhbuf[e] = 0.0f;
    }
    if (blockIdx.x == 0 && threadIdx.x < p.L) p.bar[threadIdx.x] = 0u;
}

__global__ void mask_tail_kernel(float* __restrict__ Y, int layout, int64_t S, int64_t D, int64_t N,
                                 int64_t H, int64_t t0, int io)
{
    const int64_t DH = D * H;
    if (layout == 0) {
        const int64_t begin = t0 * D * N * H, end = S * D * N * H;
        for (int64_t i = begin + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < end;
             i += (int64_t)gridDim.x * blockDim.x)
            io_store(Y, (size_t)i, 0.0f, io);
    } else {
        const int64_t per_row = (S - t0) * DH;
        const int64_t total = N * per_row;
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
             i += (int64_t)gridDim.x * blockDim.x) {
            const int64_t n = i / per_row, r = i - n * per_row;
            io_store(Y, (size_t)((n * S + t0) * DH + r), 0.0f, io);
        }
    }
}

// Wk[r][k] = W[d*GH + g*H + u][k] for r = d*GH + u*G + g: whole rows of W,
// reordered to the projection's interleaved column order (fp32 copy or bf16).
template <typename T>
__global__ void pack_kmajor_kernel(const float* __restrict__ W, T* __restrict__ Wk, int G, int64_t H, int64_t I,
                                   int64_t rows)
{
    const int64_t GH = (int64_t)G * H;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const int64_t d = r / GH, rem = r - d * GH, u = rem / G, g = rem - u * G;
        const float* src = W + (d * GH + g * H + u) * I;
        T* dst = Wk + r * I;
        for (int64_t k = threadIdx.x; k < I; k += blockDim.x) {
            if constexpr (sizeof(T) == 4) dst[k] = src[k];
            else if constexpr (std::is_same<T, __half>::value) dst[k] = __float2half_rn(src[k]);
            else dst[k] = __float2bfloat16_rn(src[k]);
        }
    }
}

// dst[i] = src[i] between fp32 (0), fp16 (1) and bf16 (2); widening is exact,
// narrowing rounds to nearest even.
__global__ void convert_kernel(const void* __restrict__ src, int st, void* __restrict__ dst, int dt, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const float v = io_load(reinterpret_cast<const float*>(src), (size_t)i, st);
        if (dt == 2) reinterpret_cast<__nv_bfloat16*>(dst)[i] = __float2bfloat16_rn(v);
        else if (dt == 1) reinterpret_cast<__half*>(dst)[i] = __float2half_rn(v);
        else reinterpret_cast<float*>(dst)[i] = v;
    }
}

__global__ void to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n)
{
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        dst[i] = __float2bfloat16_rn(src[i]);
}

}  // namespace

cudaError_t launch_pack_kmajor(const float* W, void* Wk, int D, int G, int64_t H, int64_t I, int dtype,
                               cudaStream_t stream)
{
    const int64_t rows = (int64_t)D * G * H;
    if (rows <= 0 || I <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>(rows, 8192);
    if (dtype == 1) pack_kmajor_kernel<<<blocks, 128, 0, stream>>>(W, (__nv_bfloat16*)Wk, G, H, I, rows);
    else if (dtype == 2) pack_kmajor_kernel<<<blocks, 128, 0, stream>>>(W, (__half*)Wk, G, H, I, rows);
    else pack_kmajor_kernel<<<blocks, 128, 0, stream>>>(W, (float*)Wk, G, H, I, rows);
    return cudaGetLastError();
}

cudaError_t launch_convert(const void* src, int src_type, void* dst, int dst_type, int64_t n, cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 16);
    convert_kernel<<<blocks, 256, 0, stream>>>(src, src_type, dst, dst_type, n);
    return cudaGetLastError();
}

cudaError_t launch_to_bf16(const float* src, void* dst, int64_t n, cudaStream_t stream)
{
    if (n <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, 152 * 16);
    to_bf16_kernel<<<blocks, 256, 0, stream>>>(src, (__nv_bfloat16*)dst, n);
    return cudaGetLastError();
}

cudaError_t launch_pack(const float* W, const float* R, float* Wt, float* Rt, int D, int G, int64_t H,
                        int64_t I, cudaStream_t stream)
{
    const int64_t GH = (int64_t)G * H;
    const dim3 block(32, 8);
    for (int d = 0; d < D; ++d) {
        if (W && Wt && I > 0) {
            const dim3 grid((unsigned)((GH + 31) / 32), (unsigned)((I + 31) / 32));
            pack_kernel<<<grid, block, 0, stream>>>(W + (size_t)d * GH * I, Wt, G, H, I, (int64_t)D * GH,
                                                    (int64_t)d * GH);
        }
        if (R && Rt) {
            const dim3 grid((unsigned)((GH + 31) / 32), (unsigned)((H + 31) / 32));
            pack_kernel<<<grid, block, 0, stream>>>(R + (size_t)d * GH * H, Rt + (size_t)d * H * GH, G, H, H,
                                                    GH, 0);
        }
    }
    return cudaGetLastError();
}

namespace {

__global__ void rank_rows_kernel(const int32_t* __restrict__ lens, int32_t* __restrict__ perm, int N)
{
    for (int n = blockIdx.x * blockDim.x + threadIdx.x; n < N; n += gridDim.x * blockDim.x) {
        const int ln = lens[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int lm = lens[m];
            rank += (lm > ln || (lm == ln && m < n)) ? 1 : 0;
        }
        perm[rank] = n;
    }
}

__global__ void pack_r_split_kernel(const float* __restrict__ R, __half* __restrict__ Rp, int64_t H, int64_t rows)
{
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        const int64_t d = r / (3 * H), rem = r - d * 3 * H;
        const int64_t u = rem < 2 * H ? rem / 2 : rem - 2 * H;
        const int64_t g = rem < 2 * H ? rem % 2 : 2;
        const float* src = R + (d * 3 * H + g * H + u) * H;
        __half* dst = Rp + r * H;
        for (int64_t k = threadIdx.x; k < H; k += blockDim.x) dst[k] = __float2half_rn(src[k]);
    }
}

// Stacked layers, layout 0, bidirectional layer below: x[t][n][d*H + u] =
// y[t][d][n][u] (element size 4 or 2 bytes; moved as bits).
template <typename T>
__global__ void stack_permute_kernel(const T* __restrict__ y, T* __restrict__ x, int64_t S, int64_t N, int64_t H)
{
    const int64_t total = S * 2 * N * H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t u = i % H, r = i / H;        // r = (t*2 + d)*N + n over y
        const int64_t n = r % N, td = r / N, d = td % 2, t = td / 2;
        x[(t * N + n) * 2 * H + d * H + u] = y[i];
    }
}

// Tensor-core kernel: hx[b][d][r][u] (fp16, 128 rows) = initial_h for b = 0
// and r < N, else 0; step counters 0.
__global__ void tc_state_init_kernel(const RecParams p)
{
    __half* hx = reinterpret_cast<__half*>(p.hbuf);
    const int64_t total = (int64_t)2 * p.D * 128 * p.H;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t u = i % p.H, r = (i / p.H) % 128, d = (i / ((int64_t)p.H * 128)) % p.D;
        const int64_t b = i / ((int64_t)p.H * 128 * p.D);
        float v = 0.0f;
        if (b == 0 && r < p.N && p.h0) {
            const int64_t si = p.layout == 0 ? (d * p.N + r) * p.H + u : (r * p.D + d) * p.H + u;
            v = io_load(p.h0, si, p.io);
        }
        hx[i] = __float2half_rn(v);
        if (p.rhbuf) reinterpret_cast<__half*>(p.rhbuf)[i] = __float2half_rn(0.0f);   // GRU lbr = 0: r (.) h
    }
    if (blockIdx.x == 0 && threadIdx.x < p.D) {
        p.bar[threadIdx.x] = 0u;
        if (p.flags) p.flags[threadIdx.x] = 0u;
    }
}

}  // namespace

cudaError_t launch_pack_r_split(const float* R, void* Rp, int D, int64_t H, cudaStream_t stream)
{
    const int64_t rows = (int64_t)D * 3 * H;
    if (rows <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>(rows, 152 * 8);
    pack_r_split_kernel<<<blocks, 128, 0, stream>>>(R, (__half*)Rp, H, rows);
    return cudaGetLastError();
}

cudaError_t launch_stack_permute(const void* y, void* x, int64_t S, int64_t N, int64_t H, int elem,
                                 cudaStream_t stream)
{
    const int64_t total = S * 2 * N * H;
    if (total <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)std::min<int64_t>((total + 255) / 256, 152 * 16);
    if (elem == 2)
        stack_permute_kernel<<<blocks, 256, 0, stream>>>((const unsigned short*)y, (unsigned short*)x, S, N, H);
    else
        stack_permute_kernel<<<blocks, 256, 0, stream>>>((const float*)y, (float*)x, S, N, H);
    return cudaGetLastError();
}

cudaError_t launch_rank_rows(const int32_t* lens, int32_t* perm, int N, cudaStream_t stream)
{
    if (N <= 0) return cudaSuccess;
    rank_rows_kernel<<<(N + 127) / 128, 128, 0, stream>>>(lens, perm, N);
    return cudaGetLastError();
}

cudaError_t launch_tc_state_init(const RecParams& p, cudaStream_t stream)
{
    const int64_t total = (int64_t)2 * p.D * 128 * p.H;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + 255) / 256, 4096));
    tc_state_init_kernel<<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_wave_state_init(const WaveParams& p, cudaStream_t stream)
{
    const int64_t total = (int64_t)p.L * kWaveRing * p.H * p.npad;
    const int threads = 256;
    const int blocks = (int)std::max<int64_t>(1, std::min<int64_t>((total + threads - 1) / threads, 4096));
    wave_state_init_kernel<<<blocks, threads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_state_init(const RecParams& p, cudaStream_t stream)
{
    const int64_t total = (int64_t)p.D * p.row_groups * p.npad * (p.kernel == 2 ? p.hpad : p.H);
    int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    if (blocks < 1) blocks = 1;
    state_init_kernel<<<blocks, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_mask_tail(float* Y, int layout, int64_t S, int64_t D, int64_t N, int64_t H, int64_t t0, int io,
                             cudaStream_t stream)
{
    if (!Y || t0 >= S) return cudaSuccess;
    const int64_t total = (S - t0) * D * N * H;
    int blocks = (int)std::min<int64_t>((total + 255) / 256, 8192);
    if (blocks < 1) blocks = 1;
    mask_tail_kernel<<<blocks, 256, 0, stream>>>(Y, layout, S, D, N, H, t0, io);
    return cudaGetLastError();
}

}  // namespace rnngb
