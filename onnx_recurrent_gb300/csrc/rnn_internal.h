// Internal interfaces between the C-ABI host code and the CUDA kernels.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace rnngb {

struct ActSpec {
    int fn;        // RNN_ACT_* id, -1 when the slot is unused
    float alpha;
    float beta;
};

// Arguments of the persistent recurrent kernel (one launch covers all
// directions; CTAs [d*ctas_per_dir, (d+1)*ctas_per_dir) serve direction d).
struct RecParams {
    int op, G, D, N, H, S, layout;
    int lbr, input_forget;
    int has_B, has_P, has_h0, has_c0, has_lens, has_clip;
    float clip;
    ActSpec act[2][3];           // per direction: f, g, h
    int max_len;                 // steps to run: max over rows of the length
    int dir_reverse[2];          // per direction: 1 if it walks time backwards

    // geometry
    int ctas_per_dir;            // C
    int umax;                    // ceil(H / C): unit slots per CTA
    int rows_per_thread;         // TN (template parameter mirrored here)
    int r_resident;              // 1: R slice lives in shared memory
    int npad;                    // N rounded up to a multiple of 4

    // tensors
    const float* XW;             // [S*N rows][D*G*H], columns u*G + g per direction
    const float* Rt;             // [D][H (k)][G*H], columns u*G + g
    const float* B;              // [D][2*G*H] (may be null)
    const float* P;              // [D][3*H]   (may be null)
    const float* h0;             // layout-dependent [D,N,H] / [N,D,H] (may be null)
    const float* c0;
    const int32_t* lens;         // [N] device (may be null)
    float* Y;                    // may be null
    float* Yh;
    float* Yc;
    float* hbuf;                 // [D][2][H][npad]: h exchanged between steps
    float* rhbuf;                // [D][H][npad]: r (.) h for GRU lbr = 0
    unsigned* bar;               // [D] barrier arrival counters (zeroed per run)
    int* status;                 // device status word (0 ok, 6 timeout)
    long long spin_limit_ns;
    int debug_skip_cta;
};

// Shared-memory layout of the recurrent kernel, computed on the host.
constexpr int kRecKC = 32;       // k rows per staged chunk
constexpr int kRecStages = 4;    // chunks in the cp.async ring

__host__ __device__ inline int rec_ugp(int umax, int G) { return ((umax * G) + 3) / 4 * 4; }

inline size_t rec_smem_bytes(int H, int umax, int G, int npad, int r_resident)
{
    size_t ugp = (size_t)rec_ugp(umax, G);
    size_t rbytes = r_resident ? (size_t)H * ugp * 4 : (size_t)kRecStages * kRecKC * ugp * 4;
    size_t hbytes = (size_t)kRecStages * kRecKC * (size_t)npad * 4;
    return rbytes + hbytes;
}

// Launchers (one per op; `exact` selects FMUL+FADD vs FFMA products).
cudaError_t launch_recurrent(const RecParams& p, bool exact, int threads, size_t smem,
                             cudaStream_t stream);
cudaError_t recurrent_occupancy(int op, int rows_per_thread, bool exact, int threads,
                                size_t smem, int* blocks_per_sm);

// Input projection XW[M][ldc] = X[M][K] . Bt[K][ncols] (Bt row stride ldb).
cudaError_t launch_projection(const float* X, const float* Bt, float* XW, int64_t M,
                              int64_t K, int64_t ncols, bool exact, cudaStream_t stream);

// Pack: Wt[k][d*GH + u*G + g] = W[d][g*H + u][k]  (ld = D*GH),
//       Rt[d][k][u*G + g]    = R[d][g*H + u][k].
cudaError_t launch_pack(const float* W, const float* R, float* Wt, float* Rt, int D, int G,
                        int64_t H, int64_t I, cudaStream_t stream);

// hbuf[d][0][u][n] = initial_h (or 0), padding columns 0; bar[d] = 0.
cudaError_t launch_state_init(const RecParams& p, cudaStream_t stream);

// Y = +0 at t >= t0 for every row (rows that ended earlier are written by
// the recurrent kernel).
cudaError_t launch_mask_tail(float* Y, int layout, int64_t S, int64_t D, int64_t N, int64_t H,
                             int64_t t0, cudaStream_t stream);

// Device address and size of the fixed scratch array used by
// rnn_run_static_scratch (looked up once per device; see rnn_static.cu).
cudaError_t static_scratch(void** ptr, size_t* bytes);

}  // namespace rnngb
