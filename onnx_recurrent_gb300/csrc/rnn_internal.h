// Internal interfaces between the C-ABI host code and the CUDA kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
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
    // dataflow kernel: TMA descriptors of the h and r (.) h exchange buffers
    // ([blocks][hpad/32 chunks][rows][36], box 36 x rows x cpb x 1) and of R
    // as given ([D][G][H units][H], box 36 x units x G x 1), no swizzle
    CUtensorMap hmap, rhmap, rmap;
    // GRU lbr = 0, R's candidate rows: tensor-core kernel, box npad2 rows;
    // dataflow kernel, box 36 x units x 1 x 1 (rmap then has a box of the
    // z and r gates)
    CUtensorMap rmap2;
    int op, G, D, N, H, S, layout;
    int lbr, input_forget;
    int has_B, has_P, has_h0, has_c0, has_lens, has_clip;
    float clip;
    int io;                      // element type of X, initial states and outputs: 0 fp32, 1 fp16, 2 bf16
    ActSpec act[2][3];           // per direction: f, g, h
    int max_len;                 // steps to run: max over rows of the length
    int dir_reverse[2];          // per direction: 1 if it walks time backwards

    // geometry
    int kernel;                  // 1: staged kernel, 2: dataflow kernel, 3: tensor-core kernel
    int ctas_per_dir;            // CTAs per direction (unit_groups * row_groups)
    int unit_groups;             // CU
    int row_groups;              // CR (1 for the staged kernel)
    int unit_quant;              // unit groups hold multiples of this many units
    int slots;                   // dataflow kernel: ring slots (one piece each)
    int chunks_per_piece;        // dataflow kernel: 32-k chunks per tensor copy
    int umax;                    // most units in one group
    int rows_per_thread;         // TN (template parameter mirrored here)
    int r_resident;              // 1: R slice lives in shared memory
    int res_chunks;              // staged kernel: the first res_chunks 32-k chunks of the R slice stay in
                                 // shared memory, the rest stream through the ring (all: r_resident)
    int npad;                    // rows per row group, padded (staged kernel: N padded to 8);
                                 // tensor-core kernel: gate columns per CTA (GRU lbr = 0: z and r only)
    int npad2;                   // tensor-core kernel, GRU lbr = 0: candidate columns per CTA
    int hpad;                    // dataflow kernel: H rounded up to 32 (chunks x 32)
    int unit_stride;             // dataflow kernel: floats per unit of the resident R slice
    int unit_fastest;            // dataflow kernel: compute thread t takes unit t % umax and row tile t / umax
    int gate_split;              // dataflow kernel: lanes per (unit, row tile), each with G / gate_split gates
    int cluster;                 // dataflow kernel: each row group is one cluster exchanging h in shared memory
                                 // (else row tile t % tiles, unit t / tiles)

    // tensors
    const float* XW;             // [S*N rows][D*G*H], columns u*G + g per direction
    const float* Rt;             // staged kernel: [D][H (k)][G*H], columns u*G + g
    const float* Rorig;          // dataflow kernel: R as given, [D][G*H][H]
    const float* B;              // [D][2*G*H] (may be null)
    const float* P;              // [D][3*H]   (may be null)
    const float* h0;             // layout-dependent [D,N,H] / [N,D,H] (may be null)
    const float* c0;
    const int32_t* lens;         // [N] device (may be null)
    const int32_t* perm;         // staged and dataflow kernels with lens: internal row r is the caller's
                                 // row perm[r] (rows by length, longest first; null = identity)
    float* Y;                    // may be null
    float* Yh;
    float* Yc;
    float* hbuf;                 // staged: [D][2][H][npad]; dataflow: [D][2][row_groups][hpad/32][npad][36]
    float* rhbuf;                // r (.) h for GRU lbr = 0, same layout as hbuf
    unsigned* bar;               // [D] barrier arrival counters (zeroed per run)
    unsigned* flags;             // dataflow kernel: [D][row_groups] publication counters (zeroed per run)
    int* status;                 // device status word (0 ok, 6 timeout)
    long long spin_limit_ns;
    int debug_skip_cta;
};

// Stacked unidirectional layers in one launch (the wavefront kernel,
// k_wave.cuh).  Every layer has the same operator, hidden size, direction and
// layout; layer l's CTAs are [cta0, cta0 + C).
constexpr int kWaveMaxLayers = 8;
constexpr int kWaveRing = 4;     // h buffers per layer (the next layer may lag by up to 3 steps)

struct WaveLayer {
    int cta0, C;                 // this layer's CTAs
    int umax, ugp;               // most units per CTA; floats per k-row of a resident slice (rec_ugp)
    int I;                       // K of the in-kernel input product (layers >= 1: hidden size), 0 for layer 0
    int lbr, input_forget;
    int has_B, has_P, has_h0, has_c0, has_clip;
    float clip;
    ActSpec act[3];              // f, g, h
    const float* XW;             // layer 0: [S*N][G*H] projection (columns u*G + g)
    const float* Wt;             // layers >= 1: W k-major [I][G*H] (columns u*G + g)
    const float* Rt;             // R k-major [H][G*H]
    const float* B;              // [2*G*H] (may be null)
    const float* P;              // [3*H]   (may be null)
    const float* h0;             // [N][H]  (may be null)
    const float* c0;
    float* Y;                    // the last layer's output sequence (null for the others)
    float* Yh;
    float* Yc;
    float* hbuf;                 // [kWaveRing][H][npad], k-major, internal rows
    float* rhbuf;                // GRU lbr = 0: r (.) h [H][npad]
};

struct WaveParams {
    int L, N, H, S, layout, reverse, npad, max_len;
    int has_lens;
    const int32_t* lens;         // [N] device (may be null)
    const int32_t* perm;         // internal row r is the caller's row perm[r] (null = identity)
    unsigned* bar;               // [L] arrival counters (zeroed per run)
    int* status;
    long long spin_limit_ns;
    int debug_skip_cta;
    WaveLayer layer[kWaveMaxLayers];
};

// Shared-memory layout of the recurrent kernels, computed on the host.
constexpr int kRecKC = 32;       // k rows per chunk
constexpr int kRecStages = 3;    // chunks in the cp.async ring (staged kernel; measured: 2-4 within 2%)
constexpr int kMaxSlots = 32;    // ring slots of the dataflow kernel

__host__ __device__ inline int rec_ugp(int umax, int G) { return ((umax * G) + 3) / 4 * 4; }

// Staged kernel: res_chunks resident 32-k chunks of the R slice, a ring of
// streamed R chunks when some are not resident, the ring of h chunks.
inline size_t rec_smem_bytes(int H, int umax, int G, int npad, int res_chunks)
{
    const int nchunks = (H + kRecKC - 1) / kRecKC;
    const size_t ugp = (size_t)rec_ugp(umax, G);
    const size_t chunk = (size_t)kRecKC * ugp * 4;
    const size_t rres = res_chunks >= nchunks ? (size_t)H * ugp * 4 : (size_t)res_chunks * chunk;
    const size_t rring = res_chunks >= nchunks ? 0 : (size_t)kRecStages * chunk;
    const size_t hbytes = (size_t)kRecStages * kRecKC * (size_t)npad * 4;
    return rres + rring + hbytes;
}

// Dataflow kernel: floats between the gate rows of a unit in the resident R
// slice (rows of kr k, 12 floats apart modulo the 32 banks, so the lanes of
// a gate-split group, one gate each, read different banks), and per unit
// (G rows, padded so that consecutive units start 16 bytes apart modulo the
// 128-byte bank window: conflict-free 16-byte loads across units).
constexpr int kDfGatePad = 12;
__host__ __device__ inline int df_gate_stride(int kr) { return kr + kDfGatePad; }
inline int df_unit_stride(int kr, int G)
{
    const int gh = G * df_gate_stride(kr);
    return gh + (((4 - gh) % 32) + 32) % 32;
}

// Dataflow kernel: a 32-k chunk of one operand row is stored with a pitch of
// 36 floats (144 bytes), so that the rows read by the 8 (or 4) threads of a
// quarter warp fall in distinct bank groups.  The exchange buffers are kept
// in that form; tensor copies of R take 36 k (the 4 extra are never used).
constexpr int kDfPitch = 36;

// Bytes of one chunk of streamed R: G x umax rows of 144 bytes, 128-aligned.
__host__ __device__ inline size_t df_rsub_bytes(int umax, int G) { return (((size_t)G * umax * kDfPitch * 4 + 127) / 128) * 128; }

// Dataflow kernel: bytes between h ring slots.  A slot holds one piece (cpb
// chunks of npad rows of 36 floats) and is a tensor-copy destination, so its
// start must be 128-byte aligned: the pitch is rounded up to 128 bytes (npad
// need not be a multiple of 8).
__host__ __device__ inline size_t df_hslot_bytes(int npad, int cpb)
{
    return (((size_t)npad * cpb * kDfPitch * 4 + 127) / 128) * 128;
}

// Dataflow kernel: dynamic shared memory (128-byte alignment slack + R
// resident, in full or its leading res_chunks 32-k chunks + a ring of
// streamed R pieces unless all of R is resident + a ring of h pieces; a slot
// holds one piece of cpb chunks).
// Dataflow kernel with the in-cluster exchange: slack + resident R + two h
// buffers (three with r (.) h), each one row group's exchange block.
inline size_t df_cluster_smem_bytes(int H, int umax, int G, int npad, bool two)
{
    const size_t rres = (((size_t)umax * df_unit_stride(H, G) * 4 + 127) / 128) * 128;
    const size_t blk = (((size_t)npad * ((H + kRecKC - 1) / kRecKC) * kDfPitch * 4 + 127) / 128) * 128;
    return 128 + rres + (two ? 3 : 2) * blk;
}

inline size_t df_smem_bytes(int H, int umax, int G, int npad, int r_resident, int cpb, int slots,
                            int res_chunks = 0)
{
    const int kr = r_resident ? H : res_chunks * kRecKC;
    const size_t rres = kr > 0 ? (((size_t)umax * df_unit_stride(kr, G) * 4 + 127) / 128) * 128 : 0;
    const size_t rslot = (size_t)cpb * df_rsub_bytes(umax, G);
    const size_t rring = r_resident ? 0 : (size_t)slots * rslot;
    return 128 + rres + rring + (size_t)slots * df_hslot_bytes(npad, cpb);
}

// The control block: barrier counters, status word, publication flags.
constexpr size_t kCtrlBytes = 4096;
constexpr size_t kCtrlStatusOffset = 64;
constexpr size_t kCtrlFlagsOffset = 256;
constexpr int kMaxFlags = (int)((kCtrlBytes - kCtrlFlagsOffset) / 4);

// Launchers (one per op; `exact` selects FMUL+FADD vs FFMA products;
// p.kernel selects the staged or the dataflow kernel).
cudaError_t launch_recurrent(const RecParams& p, bool exact, int threads, size_t smem,
                             cudaStream_t stream);
cudaError_t recurrent_occupancy(int op, int lbr, int kernel, int rows_per_thread, bool exact, int threads,
                                size_t smem, int* blocks_per_sm, int gate_split = 1);
// In-cluster dataflow launches: clusters of `cluster` CTAs that fit at once.
cudaError_t cluster_occupancy(int op, int lbr, int rows_per_thread, bool exact, int ctas, int cluster, int threads,
                              size_t smem, int* clusters);

// Input projection XW[M][ncols] = X[M][K] . Bt[K][ncols].  A wait of the
// tensor-copy loader that gives up writes RNN_ERR_TIMEOUT to *status.
cudaError_t launch_projection(const float* X, const float* Bt, float* XW, int64_t M,
                              int64_t K, int64_t ncols, bool exact, int* status, long long limit_ns,
                              cudaStream_t stream);

// Encodes a tiled tensor map (no swizzle, or 128-byte swizzle; out-of-range
// reads as zero) of fp32 (dtype 0), bf16 (1) or fp16 (2) elements; false when
// the driver entry point is missing or rejects the shape.
bool encode_tensor_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, bool swizzle128 = false,
                       int dtype = 0);

// Input projection on the tensor cores (TF32 products of fp32 operands, or
// bf16 operands; FP32 sums): XW[M][ncols] = X[M][K] . Wk[ncols][K]^T with Wk
// K-major (see launch_pack_kmajor).  X and Wk are fp32, or bf16 when `bf16`.
bool projection_tc_supported(const void* X, const void* Wk, float* XW, int64_t M, int64_t K, int64_t ncols,
                             bool bf16);
cudaError_t launch_projection_tc(const void* X, const void* Wk, float* XW, int64_t M, int64_t K, int64_t ncols,
                                 bool bf16, int* status, long long limit_ns, cudaStream_t stream);

// Wk[d*G*H + u*G + g][k] = W[d][g*H + u][k]: W's rows in the projection's
// column order, K contiguous; written as fp32 (dtype 0), or rounded to bf16
// (1) or fp16 (2) (Wk then holds 2-byte elements).  Also packs R (I = H) for
// the tensor-core recurrent kernel.
cudaError_t launch_pack_kmajor(const float* W, void* Wk, int D, int G, int64_t H, int64_t I, int dtype,
                               cudaStream_t stream);

// dst[i] = src[i] rounded to bf16 (nearest even), n elements.
cudaError_t launch_to_bf16(const float* src, void* dst, int64_t n, cudaStream_t stream);
// dst = src between element types 0 fp32, 1 fp16, 2 bf16 (n elements).
cudaError_t launch_convert(const void* src, int src_type, void* dst, int dst_type, int64_t n, cudaStream_t stream);

// Pack: Wt[k][d*GH + u*G + g] = W[d][g*H + u][k]  (ld = D*GH),
//       Rt[d][k][u*G + g]    = R[d][g*H + u][k].
cudaError_t launch_pack(const float* W, const float* R, float* Wt, float* Rt, int D, int G,
                        int64_t H, int64_t I, cudaStream_t stream);

// Tensor-core recurrent kernel (kernel 3): shared memory for hidden size H
// and npad padded gate columns, threads per CTA, the most gate columns a CTA
// may own, occupancy, launch.  Its exchange buffer p.hbuf holds fp16
// [2][D][128][H]; launch_tc_state_init fills buffer 0 from initial_h (rows
// past the batch 0), buffer 1 with 0, and zeroes the step counters.
size_t tc_recurrent_smem(int H, int npad, int umax, int stages);
int tc_recurrent_max_stages();
int tc_recurrent_threads();
int tc_recurrent_max_columns();
int tc_recurrent_max_units(int op);
cudaError_t tc_recurrent_occupancy(int op, bool two, size_t smem, int* blocks_per_sm);   // two: GRU lbr = 0
cudaError_t launch_tc_recurrent(const RecParams& p, size_t smem, cudaStream_t stream);
cudaError_t launch_tc_state_init(const RecParams& p, cudaStream_t stream);

// perm[rank] = n, rank = the number of rows longer than n or as long and
// before it: the rows sorted by length, longest first (stable).
cudaError_t launch_rank_rows(const int32_t* lens, int32_t* perm, int N, cudaStream_t stream);
// GRU R [D][3H][H] to fp16 K-major rows in the tensor-core kernel's split
// order for linear_before_reset = 0: per direction the z and r rows of every
// unit interleaved (row 2u + g), then the candidate rows (row 2H + u).
// Stacked layers, layout 0: a bidirectional layer's Y [S][2][N][H] as the
// next layer's X [S][N][2H] (elem: 4 or 2 bytes).
cudaError_t launch_stack_permute(const void* y, void* x, int64_t S, int64_t N, int64_t H, int elem,
                                 cudaStream_t stream);
cudaError_t launch_pack_r_split(const float* R, void* Rp, int D, int64_t H, cudaStream_t stream);
// Single RNN cell: Ho = f(clip((X.W^T + Hp.R^T) + B)); fn 0 Relu, 1 Tanh, 2
// Sigmoid; X [N, I], Hp and Ho [N, H], W [H, I], R [H, H], B [H].
cudaError_t launch_cell(const float* X, const float* Hp, const float* W, const float* R, const float* B, float* Ho,
                        int64_t N, int64_t I, int64_t H, int fn, int has_clip, float clip, bool exact,
                        cudaStream_t stream);

// Exchange buffer 0 = initial_h (or 0), everything else 0; bar, flags = 0.
cudaError_t launch_state_init(const RecParams& p, cudaStream_t stream);

// Y = +0 at t >= t0 for every row (rows that ended earlier are written by
// the recurrent kernel).
cudaError_t launch_mask_tail(float* Y, int layout, int64_t S, int64_t D, int64_t N, int64_t H, int64_t t0, int io,
                             cudaStream_t stream);

// Wavefront kernel launch (op 0 RNN, 1 GRU, 2 LSTM; tn rows per thread 1, 2
// or 4), its occupancy, and its set-up: every layer's ring buffer 0 from its
// initial_h (rows through perm), the other buffers, r (.) h and the counters 0.
cudaError_t launch_wavefront(int op, const WaveParams& p, bool exact, int tn, int ctas, int threads, size_t smem,
                             cudaStream_t stream);
cudaError_t wavefront_occupancy(int op, int tn, bool exact, int threads, size_t smem, int* blocks_per_sm);
cudaError_t launch_wave_state_init(const WaveParams& p, cudaStream_t stream);

// Device address and size of the fixed scratch array used by
// rnn_run_static_scratch (looked up once per device; see rnn_static.cu).
cudaError_t static_scratch(void** ptr, size_t* bytes);

}  // namespace rnngb
