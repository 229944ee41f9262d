/*
 * onnx_recurrent.h -- C ABI of the GB300 (sm_103a) ONNX RNN / GRU / LSTM
 * sequence operator.
 *
 * The operator is the one defined by the page "Recurrent operators: RNN, GRU,
 * LSTM" (sections Support, Computation, Activations, Choices the specification
 * leaves open, Exact mode, Fast mode, Limits), with the input and output
 * tables of the page "ai.onnx.RNN" (webgpu-kernels README, Inputs / Outputs /
 * Attributes).  Every step of a run executes in this library's own CUDA
 * kernels; nothing falls back to the CPU.
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers owned by the caller, dense, fp32
 *     (sequence_lens int32), in the shapes below for the plan's layout.
 *     S = seq_length, N = batch_size, I = input_size, H = hidden_size,
 *     D = 2 for bidirectional else 1, G = 1 (RNN), 3 (GRU), 4 (LSTM).
 *       X          layout 0: [S, N, I]        layout 1: [N, S, I]
 *       W          [D, G*H, I]     gate blocks LSTM i,o,f,c; GRU z,r,h
 *       R          [D, G*H, H]
 *       B          [D, 2*G*H]      all W biases (gate order) then all R biases
 *       P          [D, 3*H]        peepholes i, o, f (LSTM only)
 *       initial_h, initial_c, Y_h, Y_c
 *                  layout 0: [D, N, H]        layout 1: [N, D, H]
 *       Y          layout 0: [S, D, N, H]     layout 1: [N, S, D, H]
 *       sequence_lens  [N] int32
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Runs are
 *     stream-ordered and asynchronous.
 *   - A plan is not re-entrant: one run at a time per plan (it owns scratch).
 *   - The recurrent kernel of a run keeps all its CTAs resident and they wait
 *     on one another every step, so two of them must not share the SMs.  The
 *     library orders recurrent launches on a device: each waits (through an
 *     event, on its own stream) for the previous one from any plan or
 *     stream; the rest of a run overlaps freely.  Launches queued under stream
 *     capture get no such ordering: graphs that hold recurrent kernels must
 *     not be replayed concurrently with each other or with uncaptured runs.
 *   - No C++ exception crosses this boundary.  A failing call returns a
 *     status and leaves a message for rnn_last_error() on the calling thread.
 */
#ifndef ONNX_RECURRENT_H
#define ONNX_RECURRENT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rnn_plan* rnn_plan_t;
typedef struct rnn_stack* rnn_stack_t;

typedef enum {
    RNN_OK = 0,
    RNN_ERR_INVALID_ARGUMENT = 1, /* bad attribute, enum, shape or pointer      */
    RNN_ERR_INVALID_INPUT = 2,    /* a sequence length outside [0, seq_length]  */
    RNN_ERR_UNSUPPORTED = 3,      /* scratch limit, or a shape with no launch   */
    RNN_ERR_CUDA = 4,             /* a CUDA runtime call failed                 */
    RNN_ERR_OOM = 5,              /* device scratch allocation failed           */
    RNN_ERR_TIMEOUT = 6           /* the device-wide step barrier gave up       */
} rnn_status;

enum { RNN_OP_RNN = 0, RNN_OP_GRU = 1, RNN_OP_LSTM = 2 };
enum { RNN_DIR_FORWARD = 0, RNN_DIR_REVERSE = 1, RNN_DIR_BIDIRECTIONAL = 2 };

/* Arithmetic modes (page "Recurrent operators", Exact mode / Fast mode).
 *   EXACT: fp32, canonical order (one accumulator per output, k increasing
 *          from +0, every multiply and add rounded separately), the library's
 *          own IEEE-only transcendentals; bit-identical to the CPU oracle.
 *   FAST:  same order; the two matrix products use fused multiply-add and the
 *          elementwise functions use CUDA's expf/tanhf/logf.  The gate
 *          arithmetic stays unfused. */
enum { RNN_MODE_EXACT = 0, RNN_MODE_FAST = 1, RNN_MODE_FAST_TF32 = 2, RNN_MODE_FAST_BF16 = 3 };

/* Element types of the activation tensors (rnn_plan_set_io_type). */
enum { RNN_IO_F32 = 0, RNN_IO_F16 = 1, RNN_IO_BF16 = 2 };

/* Activation function ids (page "Recurrent operators", Activations). */
enum {
    RNN_ACT_RELU = 0, RNN_ACT_TANH = 1, RNN_ACT_SIGMOID = 2, RNN_ACT_AFFINE = 3,
    RNN_ACT_LEAKYRELU = 4, RNN_ACT_THRESHOLDEDRELU = 5, RNN_ACT_SCALEDTANH = 6,
    RNN_ACT_HARDSIGMOID = 7, RNN_ACT_ELU = 8, RNN_ACT_SOFTSIGN = 9, RNN_ACT_SOFTPLUS = 10
};

/* Create a plan (no device work; callable without a GPU).
 * Page "Recurrent operators": Support, Activations, Choices the specification
 * leaves open (hidden_size), Computation (clip).
 *   op            RNN_OP_*.
 *   direction     RNN_DIR_*.
 *   hidden_size   H > 0 (0 or negative: RNN_ERR_INVALID_ARGUMENT).
 *   input_size    I >= 0 (0 gives an all-zero input projection).
 *   activations   NULL/0 for the defaults (LSTM Sigmoid,Tanh,Tanh; GRU
 *                 Sigmoid,Tanh; RNN Tanh), else k or 2k names (k = 3, 2, 1),
 *                 matched case-insensitively; one set serves both directions
 *                 of a bidirectional layer, two sets are forward then reverse
 *                 (a unidirectional op uses the first set).
 *   alpha, beta   activation_alpha / activation_beta (may be NULL/0); read
 *                 with separate cursors in activation order; missing values
 *                 take each activation's default.  The arrays are copied.
 *   clip          applied to every gate input when > 0; NaN or <= 0: no clip.
 *   layout        0 or 1.
 *   linear_before_reset, input_forget   0 or 1 (ignored by the ops they do
 *                 not apply to).
 * On success *out receives a plan to be released with rnn_plan_destroy. */
rnn_status rnn_plan_create(rnn_plan_t* out, int op, int direction,
                           int64_t hidden_size, int64_t input_size,
                           const char* const* activations, int n_activations,
                           const float* alpha, int n_alpha,
                           const float* beta, int n_beta,
                           float clip, int layout, int linear_before_reset,
                           int input_forget);

/* Run the operator on device tensors (shapes above).
 * Page "Recurrent operators": Computation (projection, recurrent product,
 * GRU second product, gate order of operations), Choices the specification
 * leaves open (sequence_lens, zero-size, omitted inputs), Exact mode (NaN
 * written as 0x7FC00000), Limits.
 *   seq_length, batch_size  S >= 0, N >= 0 (the C ABI needs them explicitly).
 *   X, W, R       required (W and R may be NULL after rnn_plan_set_weights).
 *   B, sequence_lens, initial_h, initial_c, P   optional (NULL = absent:
 *                 bias adds and peepholes are skipped, states start at +0,
 *                 every row runs all S steps).
 *   Y, Y_h, Y_c   optional outputs (NULL = not written); Y_c is LSTM only.
 * Zero-size (S == 0 or N == 0): nothing runs; Y_h/Y_c receive the initial
 * states or zeros.  If sequence_lens is given it is copied to the host and
 * checked first (the call waits for that copy on `stream`): a length outside
 * [0, S] returns RNN_ERR_INVALID_INPUT and nothing is written.  A run whose
 * per-direction scratch (S*N*G*H + 4*N*H + G*H*(I+H) floats, the last term
 * dropped for constant weights) reaches 2^30 floats returns
 * RNN_ERR_UNSUPPORTED.  Otherwise the kernels are queued on `stream` and the
 * call returns RNN_OK; device-side failures (a barrier timeout) are reported
 * by rnn_plan_sync(). */
rnn_status rnn_run(rnn_plan_t plan, int64_t seq_length, int64_t batch_size,
                   const float* X, const float* W, const float* R, const float* B,
                   const int32_t* sequence_lens, const float* initial_h,
                   const float* initial_c, const float* P,
                   float* Y, float* Y_h, float* Y_c, void* stream);

/* Release a plan and its device scratch (waits for its last run).  NULL is
 * ignored. */
void rnn_plan_destroy(rnn_plan_t plan);

/* ---------------------------------------------------------------- extras */

/* Select RNN_MODE_EXACT (default), RNN_MODE_FAST, RNN_MODE_FAST_TF32 or
 * RNN_MODE_FAST_BF16 (page "Recurrent operators", Exact mode / Fast mode).
 *   EXACT      bit-identical to the library's reference arithmetic: one
 *              accumulator per output, k ascending, every product and sum
 *              rounded separately, own IEEE-only transcendentals.
 *   FAST       fused multiply-adds and CUDA's accurate transcendentals; within
 *              1e-5 (absolute) of EXACT for the transcendental activations.
 *   FAST_TF32  FAST, with the input projection on the tensor cores: products
 *              of the operands' TF32 parts (10-bit mantissas), sums in FP32;
 *              within 5e-3 of EXACT.  Shapes the tensor-core path cannot take
 *              (input_size or G*H*D not a multiple of 4, unaligned pointers)
 *              run the FAST projection instead.
 *   FAST_BF16  FAST, with X and W rounded to bf16 (nearest even) and the
 *              input projection on the tensor cores, sums in FP32; within
 *              5e-3 of EXACT; input_size must be a multiple of 8 (else the
 *              FAST projection).  Scratch grows by 2 bytes per element of X.
 * An unknown mode returns RNN_ERR_INVALID_ARGUMENT. */
rnn_status rnn_plan_set_mode(rnn_plan_t plan, int mode);

/* Element type of the activation tensors of the plan's runs: RNN_IO_F32
 * (default), RNN_IO_F16 or RNN_IO_BF16 (the fp16/bf16 variants of the
 * operator's type T, Apple BNNS page; the WebGPU page's kernels take fp32
 * only).  It applies to X, initial_h, initial_c (read) and Y, Y_h, Y_c
 * (written); their pointers in rnn_run / rnn_run_static_scratch then point
 * to 2-byte elements (cast to float*), in the same shapes and layouts.  W, R,
 * B and P stay fp32.  The arithmetic is the mode's, in fp32: an input is
 * widened exactly, every output is the fp32 result rounded to nearest even
 * once, and a NaN output is the type's canonical quiet NaN (0x7E00 fp16,
 * 0x7FC0 bf16).  So EXACT mode gives the oracle's fp32 outputs rounded.
 * The recurrent kernels write the 2-byte outputs directly; X is widened to
 * fp32 in scratch for the FP32 and TF32 projections (4 bytes per element of
 * X), while in RNN_MODE_FAST_BF16 a bf16 X feeds the tensor-core projection
 * as it stands.  An unknown type is RNN_ERR_INVALID_ARGUMENT; a cell plan
 * (rnn_cell_plan_create) takes RNN_IO_F32 only (RNN_ERR_UNSUPPORTED). */
rnn_status rnn_plan_set_io_type(rnn_plan_t plan, int io);

/* Declare W and R constant (page "Recurrent operators", Computation: weights
 * are transposed once per plan when they are constants).  Packs them now on
 * `stream` into plan-owned device memory; later runs ignore their W and R
 * arguments.  W [D, G*H, I] and R [D, G*H, H] are device pointers; the
 * input_size used is the plan's. */
rnn_status rnn_plan_set_weights(rnn_plan_t plan, const float* W, const float* R,
                                void* stream);

/* Wait for the plan's last run and report its device status: RNN_OK, or
 * RNN_ERR_TIMEOUT if the step barrier gave up (the outputs are then
 * incomplete).  Clears the status.  After rnn_run_static_scratch it waits for
 * the whole device and reads the status word of the fixed scratch array,
 * which every static-scratch run on that device shares (the latest such run's
 * status). */
rnn_status rnn_plan_sync(rnn_plan_t plan);

/* The resolved activation of slot `slot` (0 = f, 1 = g, 2 = h) of direction
 * `dir`: its RNN_ACT_* id and alpha, beta (page "Recurrent operators",
 * Activations).  Slots the op does not use report fn = -1. */
rnn_status rnn_plan_get_activation(rnn_plan_t plan, int dir, int slot, int* fn,
                                   float* alpha, float* beta);

/* Launch geometry of the recurrent product, for tuning and testing.
 * rnn_plan_set_launch overrides the planner (0, or -1 for r_resident, means
 * "choose"): kernel 1 is the staged kernel (CTAs hold all batch rows; h moves
 * through a shared-memory ring; one device-wide barrier per step), kernel 2
 * the dataflow kernel (CTAs tile unit groups x row groups; a loader warp
 * fetches h with TMA tensor copies once every CTA of its row group has
 * published the step on the row group's counter), kernel 5 the dataflow
 * kernel with the exchange inside a thread-block cluster (each row group of
 * a direction is one cluster of at most 16 CTAs that hold all of R and write
 * h into each other's shared memory; 1 or 2 rows per thread; R must fit).
 * unit_groups: CTAs per direction along
 * hidden units; row_groups: along batch rows (dataflow kernels only);
 * rows_per_thread: 1, 2, 4 or 8; r_resident: R slice
 * kept in shared memory (1) or streamed through it (0); 2 asks the dataflow
 * kernel to keep the slice's leading pieces resident and stream the rest
 * (the staged kernel does that by itself whenever the slice does not fit,
 * and takes 2 as -1).  Every geometry gives
 * the same results.  rnn_plan_get_launch reports the geometry of the last
 * run (kernel 5: the in-cluster exchange, which the planner also picks by
 * itself where it models it faster; kernel 4 on a stack's first plan: the
 * run was the stack's wavefront launch, unit_groups its first layer's
 * CTAs); a shape the override cannot serve makes the run return
 * RNN_ERR_UNSUPPORTED. */
rnn_status rnn_plan_set_launch(rnn_plan_t plan, int unit_groups, int rows_per_thread,
                               int r_resident, int row_groups, int kernel);
rnn_status rnn_plan_get_launch(rnn_plan_t plan, int* unit_groups, int* rows_per_thread,
                               int* r_resident, int* row_groups, int* kernel,
                               int* threads_per_cta, int* smem_bytes);

/* Per-kernel device time, in milliseconds, measured with CUDA events that the
 * run records on its own stream around each kernel while timing is enabled:
 * out[0] weight pack, out[1] input projection, out[2] state set-up,
 * out[3] recurrence, out[4] mask epilogue (0 when a kernel did not run).
 * rnn_plan_set_timing(plan, 1) enables timing and clears the totals.
 * rnn_plan_last_timing reports the last run (waits for it).
 * rnn_plan_timing_totals reports the sums over every run since timing was
 * enabled or the totals were last read, stores their number in *runs, waits
 * for them and clears the totals.  Back-to-back timed runs never wait on the
 * device: each run's events are read at most once, after the run. */
rnn_status rnn_plan_set_timing(rnn_plan_t plan, int enable);
rnn_status rnn_plan_last_timing(rnn_plan_t plan, float* out, int n);
rnn_status rnn_plan_timing_totals(rnn_plan_t plan, float* out, int n, int* runs);

/* Test hook for the barrier's failure path: limit each device-wide barrier
 * wait to `spin_limit_ns` nanoseconds (0 restores the default of 2 s) and,
 * if skip_cta >= 0, make that CTA of the recurrent grid withhold its first
 * arrival, so that the wait runs out and the run reports RNN_ERR_TIMEOUT
 * through rnn_plan_sync() with the device still usable. */
rnn_status rnn_plan_debug_barrier(rnn_plan_t plan, int64_t spin_limit_ns, int skip_cta);

/* Number of kernel launches queued by the last rnn_run on this plan. */
int rnn_plan_last_launch_count(rnn_plan_t plan);

/* rnn_run for callers that cannot allocate device memory while they run:
 * for example a serving runtime that hands all of a GPU's memory to its own
 * pool at start-up, or a latency-critical caller for which cudaMalloc and
 * cudaFree (which synchronises the device) are not acceptable mid-run.  The
 * pages describe no such entry point: it has no counterpart there.
 * Same arguments, results and checks as rnn_run, but the call allocates
 * nothing: its scratch comes from one fixed 32 MiB device array that every
 * GPU loading this library holds until the process exits, and
 * sequence_lens (at most 4096 rows) is checked through a stack buffer.
 * A run whose scratch (4 KiB of control words, the packed weights unless
 * they are constant, seq*batch*D*G*H floats of projection and the h exchange
 * buffers) does not fit returns RNN_ERR_UNSUPPORTED before any device work.
 * The first call on a device looks up the array's device address (once per
 * device, cached for the life of the process: a device reset with
 * cudaDeviceReset makes the cached address stale, so do not call this entry
 * point on a device after resetting it); make that first call before any
 * stream capture.  Every call shares the one array and leaves its contents
 * behind; what must start at zero (barrier counters, the status word) is
 * cleared by each call, so calls that overlap on the GPU (another stream,
 * another thread or another plan) race and must be serialised by the
 * caller.  Outside a stream capture the recurrent launch is ordered behind
 * the device's other recurrent launches, as in rnn_run.  Barrier waits are
 * bounded as in rnn_run (rnn_plan_debug_barrier applies): rnn_plan_sync
 * reports a timed-out run as RNN_ERR_TIMEOUT (its outputs are then
 * incomplete).  Timing (rnn_plan_set_timing) does not apply. */
rnn_status rnn_run_static_scratch(rnn_plan_t plan, int64_t seq_length, int64_t batch_size,
                                  const float* X, const float* W, const float* R,
                                  const float* B, const int32_t* sequence_lens,
                                  const float* initial_h, const float* initial_c,
                                  const float* P, float* Y, float* Y_h, float* Y_c,
                                  void* stream);

/* Stacked layers.  The pages define single layers; a stack chains them by
 * the output sequence (this library's reading): layer l+1's X is layer l's
 * Y with the directions side by side per step, forward units first,
 *     layout 0:  X[t, n, d*H + u] = Y[t, d, n, u]
 *     layout 1:  X[n, t, d*H + u] = Y[n, t, d, u]   (Y's memory as it stands)
 * so layer l+1's input_size must be dirs(l) * hidden(l); sequence_lens is
 * shared by every layer.
 *
 * rnn_stack_create: `layers` is a host array of n_layers >= 1 plans, which
 * stay the caller's (borrowed: they must outlive the stack, and their modes,
 * weights and timing apply per layer); all share one layout and one io type
 * (rnn_plan_set_io_type); cell plans are refused.  Any mismatch is
 * RNN_ERR_INVALID_ARGUMENT.
 *
 * rnn_stack_run: W, R (required) and B, initial_h, initial_c, P, Y_h, Y_c
 * (each optional: NULL, or entries that may be NULL) are HOST arrays of
 * n_layers device pointers, each with rnn_run's meaning for its layer; X
 * feeds layer 0 and Y (may be NULL) receives the last layer's output
 * sequence.  sequence_lens is checked once (RNN_ERR_INVALID_INPUT before any
 * write).  Errors are rnn_run's, for the first failing layer.
 *
 * Two ways to run a stack, both giving rnn_run's results layer by layer
 * (bit for bit in RNN_MODE_EXACT):
 *   - the wavefront: when every layer is unidirectional, with one operator,
 *     one hidden size, one direction and one mode (RNN_MODE_EXACT or
 *     RNN_MODE_FAST), fp32 I/O, 2 to 8 layers, and the layers' slices of R
 *     and W fit in shared memory (and rnn_stack_set_wavefront allows it),
 *     the stack runs as one persistent launch
 *     (after layer 0's input projection) in which the SMs are split between
 *     the layers and layer l+1 takes step t while layer l takes step t+1;
 *     layer l+1 forms its input product from layer l's h in that launch, so
 *     no intermediate sequence is stored.  Its scratch (layer 0's
 *     projection, the packed weights, h ring buffers) is stack-owned and
 *     grown with cudaMalloc when a run needs more (which synchronises the
 *     device); the device status (a bounded wait that gave up) is reported
 *     by rnn_plan_sync on the first layer's plan, and the first layer's plan
 *     also carries the run's timing (rnn_plan_set_timing) and its
 *     rnn_plan_debug_barrier settings.
 *   - otherwise the layers run one after another on `stream`; the
 *     intermediate sequences live in two stack-owned device buffers (grown
 *     with cudaMalloc when a run needs more), and a layout-0 bidirectional
 *     layer's Y is rearranged into the next X by one kernel (any other
 *     layer's Y is the next X as it stands). */
rnn_status rnn_stack_create(rnn_stack_t* out, const rnn_plan_t* layers, int n_layers);
rnn_status rnn_stack_run(rnn_stack_t stack, int64_t seq_length, int64_t batch_size,
                         const float* X, const float* const* W, const float* const* R,
                         const float* const* B, const int32_t* sequence_lens,
                         const float* const* initial_h, const float* const* initial_c,
                         const float* const* P, float* Y, float* const* Y_h, float* const* Y_c,
                         void* stream);
void rnn_stack_destroy(rnn_stack_t stack);
/* Kernels the last rnn_stack_run queued (all layers). */
int rnn_stack_last_launch_count(rnn_stack_t stack);
/* rnn_stack_set_wavefront: 0 runs the layers one after another; 1 (the
 * default) runs a qualifying stack as one wavefront launch when its layers
 * are small enough for that to be faster (batch * G * hidden * (hidden +
 * input) products per step at most 8e6 in every layer after the first: the
 * step is then mostly exchange latency, which the layers overlap; larger
 * layers run faster one after another, their input products in the
 * projection GEMM); 2 runs every qualifying stack as a wavefront launch.
 * Other values: RNN_ERR_INVALID_ARGUMENT.  The first layer's plan's
 * unit_groups override (rnn_plan_set_launch) caps the CTAs per layer of a
 * wavefront launch.  rnn_stack_last_wavefront: 1 if the last rnn_stack_run
 * used the wavefront launch, else 0. */
rnn_status rnn_stack_set_wavefront(rnn_stack_t stack, int enable);
int rnn_stack_last_wavefront(rnn_stack_t stack);

/* Single RNN cell (page "RNNCell", RNNCell-3: Detailed description,
 * Attributes, Inputs, Outputs):  Ho = f(clip(X.W^T + H.R^T + B)), where B is
 * the sum of the input and recurrence biases, given once.
 *
 * rnn_cell_plan_create: `activation` is "Relu", "Sigmoid" or "Tanh" (any
 * case; NULL = Tanh, the page's default; any other name is
 * RNN_ERR_INVALID_ARGUMENT, as are hidden_size <= 0 and input_size < 0).
 * `clip` clamps f's input to [-clip, clip]; it must be positive, and
 * +INFINITY (the page's default) clamps nothing; NaN, 0 or a negative value
 * is RNN_ERR_INVALID_ARGUMENT.  The result is an RNN plan (forward, layout 0,
 * one activation) marked as a cell: rnn_plan_set_mode, rnn_plan_set_weights,
 * rnn_plan_sync, the timing calls and rnn_plan_destroy apply to it, and
 * rnn_run works on it as on any forward RNN plan.
 *
 * rnn_cell_run: device pointers, row-major fp32:
 *     X  [batch_size, input_size]       H  [batch_size, hidden_size]
 *     W  [hidden_size, input_size]      R  [hidden_size, hidden_size]
 *     B  [hidden_size]                  Ho [batch_size, hidden_size] (out)
 * X, H, W, R and B are read only and stay the caller's; Ho must not overlap
 * them.  H, B and Ho are required (W and R may be NULL once constant
 * weights are set with rnn_plan_set_weights, shapes [1, hidden, input] and
 * [1, hidden, hidden]; X may be NULL when input_size is 0).  One kernel
 * computes every cell: xw and rec each with one accumulator from +0, k
 * increasing, then pre = (xw + rec) + B, clip, f, canonical NaN.  Exact
 * mode rounds every product and sum separately and uses the library's own
 * tanh and sigmoid, bit-identical to the sequence operator run for one
 * step with bias [B | -0]; every other mode (FAST, FAST_TF32, FAST_BF16)
 * runs the FAST arithmetic (fused multiply-add, CUDA's tanhf / expf), within
 * FAST's 1e-5.  batch_size 0 returns RNN_OK with nothing queued and no
 * pointer read.  Stream-ordered and asynchronous; with timing on, the
 * kernel is reported as the recurrence.  One call at a time per plan. */
rnn_status rnn_cell_plan_create(rnn_plan_t* out, int64_t hidden_size, int64_t input_size,
                                const char* activation, float clip);
rnn_status rnn_cell_run(rnn_plan_t plan, int64_t batch_size, const float* X, const float* H,
                        const float* W, const float* R, const float* B, float* Ho, void* stream);

/* Message of the last failing call on this thread ("" if none). */
const char* rnn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ONNX_RECURRENT_H */
