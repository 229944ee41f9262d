// C ABI of the operator: plan creation (attribute validation and activation
// resolution), run-time checks, scratch management, launch planning and the
// kernel sequence.  See include/onnx_recurrent.h for the contract.
#include "../../include/onnx_recurrent.h"

#include <algorithm>
#include <cctype>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "rnn_internal.h"

namespace rnngb {
cudaError_t launch_recurrent_rnn(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t launch_recurrent_gru(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t launch_recurrent_lstm(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t recurrent_occupancy_rnn(int, int, int, int, bool, int, size_t, int*);
cudaError_t recurrent_occupancy_gru(int, int, int, int, bool, int, size_t, int*);
cudaError_t recurrent_occupancy_lstm(int, int, int, int, bool, int, size_t, int*);

cudaError_t launch_cluster_rnn(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t launch_cluster_gru(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t launch_cluster_lstm(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t cluster_occupancy_rnn(int, bool, bool, int, int, int, size_t, int*);
cudaError_t cluster_occupancy_gru(int, bool, bool, int, int, int, size_t, int*);
cudaError_t cluster_occupancy_lstm(int, bool, bool, int, int, int, size_t, int*);

cudaError_t cluster_occupancy(int op, int lbr, int tn, bool exact, int ctas, int cluster, int threads, size_t smem,
                              int* clusters)
{
    const bool two = op == 1 && lbr == 0;
    switch (op) {
    case 0: return cluster_occupancy_rnn(tn, exact, two, ctas, cluster, threads, smem, clusters);
    case 1: return cluster_occupancy_gru(tn, exact, two, ctas, cluster, threads, smem, clusters);
    default: return cluster_occupancy_lstm(tn, exact, two, ctas, cluster, threads, smem, clusters);
    }
}

cudaError_t launch_recurrent(const RecParams& p, bool exact, int threads, size_t smem, cudaStream_t s)
{
    if (p.kernel == 2 && p.cluster) {
        switch (p.op) {
        case 0: return launch_cluster_rnn(p, exact, threads, smem, s);
        case 1: return launch_cluster_gru(p, exact, threads, smem, s);
        default: return launch_cluster_lstm(p, exact, threads, smem, s);
        }
    }
    switch (p.op) {
    case 0: return launch_recurrent_rnn(p, exact, threads, smem, s);
    case 1: return launch_recurrent_gru(p, exact, threads, smem, s);
    default: return launch_recurrent_lstm(p, exact, threads, smem, s);
    }
}

cudaError_t launch_wavefront_rnn(const WaveParams&, bool, int, int, int, size_t, cudaStream_t);
cudaError_t launch_wavefront_gru(const WaveParams&, bool, int, int, int, size_t, cudaStream_t);
cudaError_t launch_wavefront_lstm(const WaveParams&, bool, int, int, int, size_t, cudaStream_t);
cudaError_t wavefront_occupancy_rnn(int, bool, int, size_t, int*);
cudaError_t wavefront_occupancy_gru(int, bool, int, size_t, int*);
cudaError_t wavefront_occupancy_lstm(int, bool, int, size_t, int*);

cudaError_t launch_wavefront(int op, const WaveParams& p, bool exact, int tn, int ctas, int threads, size_t smem,
                             cudaStream_t s)
{
    switch (op) {
    case 0: return launch_wavefront_rnn(p, exact, tn, ctas, threads, smem, s);
    case 1: return launch_wavefront_gru(p, exact, tn, ctas, threads, smem, s);
    default: return launch_wavefront_lstm(p, exact, tn, ctas, threads, smem, s);
    }
}

cudaError_t wavefront_occupancy(int op, int tn, bool exact, int threads, size_t smem, int* blocks)
{
    switch (op) {
    case 0: return wavefront_occupancy_rnn(tn, exact, threads, smem, blocks);
    case 1: return wavefront_occupancy_gru(tn, exact, threads, smem, blocks);
    default: return wavefront_occupancy_lstm(tn, exact, threads, smem, blocks);
    }
}

cudaError_t recurrent_occupancy(int op, int lbr, int kernel, int tn, bool exact, int threads, size_t smem, int* blocks,
                                int gs)
{
    switch (op) {
    case 0: return recurrent_occupancy_rnn(kernel, lbr, tn, gs, exact, threads, smem, blocks);
    case 1: return recurrent_occupancy_gru(kernel, lbr, tn, gs, exact, threads, smem, blocks);
    default: return recurrent_occupancy_lstm(kernel, lbr, tn, gs, exact, threads, smem, blocks);
    }
}
}  // namespace rnngb

using namespace rnngb;

namespace {

thread_local std::string g_error;

rnn_status fail(rnn_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_error = buf;
    return st;
}

rnn_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(e == cudaErrorMemoryAllocation ? RNN_ERR_OOM : RNN_ERR_CUDA, "%s: %s", what,
                cudaGetErrorString(e));
}

constexpr int kMaxThreads = 512;          // staged kernel
// The staged kernel's threads per CTA for rows_per_thread tn (eight rows
// per thread take up to 255 registers: at most 256 threads).
int staged_thread_limit(int tn) { return tn == 8 ? 256 : kMaxThreads; }
// Threads of a one-CTA staged launch over H units and N rows with the
// widest row tile that fits, or 0 if none does.
bool staged_single_cta_fits(int64_t H, int64_t N)
{
    return H * ((N + 3) / 4) <= kMaxThreads || H * ((N + 7) / 8) <= staged_thread_limit(8);
}
constexpr int kMaxComputeThreads = 480;   // dataflow kernel (plus one loader warp)
constexpr long long kDefaultSpinNs = 2000000000LL;   // 2 s per barrier wait

int gates_of(int op) { return op == RNN_OP_RNN ? 1 : (op == RNN_OP_GRU ? 3 : 4); }
int acts_per_dir(int op) { return op == RNN_OP_RNN ? 1 : (op == RNN_OP_GRU ? 2 : 3); }

struct ActInfo {
    const char* name;
    bool takes_alpha, takes_beta;
    float alpha0, beta0;
};

// Page "Recurrent operators", Activations: the supported functions, which
// parameters each takes and their defaults.
const ActInfo kActs[] = {
    {"relu", false, false, 0.0f, 0.0f},        {"tanh", false, false, 0.0f, 0.0f},
    {"sigmoid", false, false, 0.0f, 0.0f},     {"affine", true, true, 1.0f, 0.0f},
    {"leakyrelu", true, false, 0.01f, 0.0f},   {"thresholdedrelu", true, false, 1.0f, 0.0f},
    {"scaledtanh", true, true, 1.0f, 0.0f},    {"hardsigmoid", true, true, 0.2f, 0.5f},
    {"elu", true, false, 1.0f, 0.0f},          {"softsign", false, false, 0.0f, 0.0f},
    {"softplus", false, false, 0.0f, 0.0f},
};
constexpr int kNumActs = (int)(sizeof kActs / sizeof kActs[0]);

int act_id(const char* s)
{
    if (!s) return -1;
    std::string low;
    for (const char* q = s; *q; ++q) low.push_back((char)std::tolower((unsigned char)*q));
    for (int i = 0; i < kNumActs; ++i)
        if (low == kActs[i].name) return i;
    return -1;
}

int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int smem_optin = 0;
    bool coop = false;
};

}  // namespace

struct rnn_plan {
    int op = 0, direction = 0, D = 1, G = 1, layout = 0, lbr = 0, input_forget = 0;
    int64_t H = 0, I = 0;
    float clip = 0.0f;
    int has_clip = 0;
    ActSpec act[2][3];
    int mode = RNN_MODE_EXACT;

    // constant weights (rnn_plan_set_weights)
    bool const_weights = false;
    float* wt_const = nullptr;   // [I][D*G*H]
    float* wk_const = nullptr;   // [D*G*H][I] (the tensor-core projection's operand)
    void* wkb_const = nullptr;   // the same rounded to bf16
    void* rp16_const = nullptr;  // R [D*G*H][H] fp16 (tensor-core recurrence): the projection's column order, GRU lbr = 0 the split order
    float* rt_const = nullptr;   // [D][H][G*H]
    float* r_orig_const = nullptr;   // R as given, [D][G*H][H] (the dataflow kernel reads this layout)

    // scratch
    char* scratch = nullptr;
    size_t scratch_bytes = 0;
    char* ctrl = nullptr;        // bar[2] + status
    int32_t* lens_host = nullptr;
    int64_t lens_cap = 0;
    int device = -1;

    // launch overrides and record
    int ov_units = 0, ov_tn = 0, ov_rres = -1, ov_rows = 0, ov_kernel = 0;
    int g_units = 0, g_tn = 0, g_rres = 0, g_rows = 0, g_kernel = 0, g_threads = 0, g_smem = 0;
    int last_launches = 0;

    // timing: a ring of event sets, one per run, harvested lazily so that
    // timing many back-to-back runs never waits on the device mid-stream
    static constexpr int kRing = 256;
    bool timing = false;
    bool events_ready = false;
    cudaEvent_t ev[kRing][6]{};
    bool ev_used[kRing][6]{};
    bool slot_pending[kRing]{};
    int slot = 0;                // slot of the current / last run
    double totals_ms[5]{};
    int totals_runs = 0;
    cudaEvent_t done{};
    bool done_ready = false;
    bool ran = false;

    long long spin_limit_ns = kDefaultSpinNs;
    int skip_cta = -1;

    bool cell = false;   // made by rnn_cell_plan_create
    int io = 0;          // element type of X, initial states, Y, Y_h, Y_c (RNN_IO_*)

    // the last run came from rnn_run_static_scratch: its status word lives in
    // the fixed array (shared by every static run on that device)
    bool last_static = false;
    int* static_status = nullptr;
};

namespace {

rnn_status device_info(DeviceInfo* out)
{
    static thread_local DeviceInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(RNN_ERR_CUDA, "device ordinal %d out of range", dev);
    DeviceInfo& c = cache[dev];
    if (c.device != dev) {
        cudaDeviceProp prop;
        e = cudaGetDeviceProperties(&prop, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
        c.device = dev;
        c.sms = prop.multiProcessorCount;
        c.smem_optin = (int)prop.sharedMemPerBlockOptin;
        c.coop = prop.cooperativeLaunch != 0;
    }
    *out = c;
    return RNN_OK;
}

struct Geometry {
    int kernel;       // 1 staged, 2 dataflow
    int ctas;         // CTAs per direction
    int units;        // unit groups
    int rows;         // row groups
    int quant;        // unit quantum
    int slots;        // dataflow ring slots
    int umax, tn, threads, rres;
    int res_chunks;   // staged: resident 32-k chunks of the R slice (all of them when rres)
    size_t smem;
    int npad;         // rows per row group (padded); tensor-core kernel: gate columns per CTA
    int npad2;        // tensor-core kernel, GRU lbr = 0: candidate columns per CTA
    int hpad;         // dataflow: exchange-buffer row length
    int cpb;          // dataflow: chunks per tensor copy
    int ustride;      // dataflow: floats per unit of the resident R slice
    int ufast;        // dataflow: compute threads take units fastest (wide row tiles)
    int gs;           // dataflow: gate split (lanes per unit and row)
    int cluster;      // dataflow: in-cluster exchange of h (each row group one cluster)
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Staged kernel: C CTAs per direction, all rows, device-wide barrier per step.
rnn_status plan_staged(rnn_plan* pl, int64_t N, const DeviceInfo& di, Geometry* g)
{
    const int64_t H = pl->H;
    const int G = pl->G, D = pl->D;
    g->kernel = 1;
    g->rows = 1;
    g->quant = 1;
    g->slots = 0;
    g->npad = (int)round_up(N, 8);
    int C;
    if (pl->ov_units > 0) {
        C = (int)std::min<int64_t>(pl->ov_units, H);
    } else {
        const long long macs = (long long)N * G * H * H;
        if (macs <= 262144 && staged_single_cta_fits(H, N))
            C = 1;   // tiny step: one CTA per direction, no device-wide barrier
        else
            C = (int)std::max<int64_t>(1, std::min<int64_t>(di.sms / D, H));
        const int64_t umax0 = (H + C - 1) / C;
        C = (int)((H + umax0 - 1) / umax0);
    }
    g->ctas = C;
    g->units = C;
    g->umax = (int)((H + C - 1) / C);
    const int tns[4] = {1, 2, 4, 8};
    g->tn = 0;
    if (pl->ov_tn > 0) {
        g->tn = pl->ov_tn;
    } else {
        for (int tn : tns)
            if ((int64_t)g->umax * ((N + tn - 1) / tn) <= staged_thread_limit(tn)) { g->tn = tn; break; }
    }
    if (g->tn == 0)
        return fail(RNN_ERR_UNSUPPORTED,
                    "no recurrent launch for batch %lld with %d hidden units per CTA (threads > %d)",
                    (long long)N, g->umax, kMaxThreads);
    const int64_t thr = (int64_t)g->umax * ((N + g->tn - 1) / g->tn);
    if (thr > staged_thread_limit(g->tn))
        return fail(RNN_ERR_UNSUPPORTED, "recurrent launch needs %lld threads per CTA (max %d)",
                    (long long)thr, staged_thread_limit(g->tn));
    g->threads = (int)round_up(thr, 32);
    // R slice: all resident when it fits; else as many leading 32-k chunks as
    // fit beside the two rings, the rest streamed (override 0: all streamed)
    const int nch = (int)ceil_div(H, kRecKC);
    const size_t cap = (size_t)di.smem_optin - 1024;
    const size_t sres = rec_smem_bytes((int)H, g->umax, G, g->npad, nch);
    if (pl->ov_rres == 1) g->rres = 1;
    else if (pl->ov_rres == 0) g->rres = 0;
    else g->rres = sres <= cap ? 1 : 0;
    g->res_chunks = g->rres ? nch : 0;
    if (!g->rres && pl->ov_rres != 0)
        while (g->res_chunks + 1 < nch && rec_smem_bytes((int)H, g->umax, G, g->npad, g->res_chunks + 1) <= cap)
            ++g->res_chunks;
    g->smem = rec_smem_bytes((int)H, g->umax, G, g->npad, g->res_chunks);
    if (g->smem > (size_t)di.smem_optin)
        return fail(RNN_ERR_UNSUPPORTED, "recurrent kernel needs %zu bytes of shared memory (max %d)",
                    g->smem, di.smem_optin);
    int blocks = 0;
    cudaError_t e = recurrent_occupancy(pl->op, pl->lbr, 1, g->tn, pl->mode == RNN_MODE_EXACT, g->threads, g->smem, &blocks);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (blocks < 1 || (int64_t)D * C > (int64_t)blocks * di.sms)
        return fail(RNN_ERR_UNSUPPORTED,
                    "recurrent grid of %d CTAs cannot be co-resident (%d per SM, %d SMs)", D * C, blocks,
                    di.sms);
    return RNN_OK;
}

// Dataflow kernel: CU unit groups x CR row groups per direction, TMA ring,
// per-CTA flags.  Picks the cheapest feasible shape under a simple cost
// model (cycles per step: k-loop issue + h/R bytes into the SM + epilogue +
// a fixed latency for the flags and the first copy).
// Cycles of one thread's k-loop over H (k ascending, groups of 4 k) with
// `warps` warps of tn rows x nc gate columns a thread: per group the largest
// of the busiest scheduler's issue, the shared-memory wavefronts of all
// warps (about 2.75 per 16-byte warp load with these broadcast patterns,
// measured) and one warp's dependent issue (about 1.7 cycles an instruction,
// measured on one warp).
double kloop_cycles(int64_t H, int warps, int tn, int nc, bool exact)
{
    const double instr = (exact ? 2.0 : 1.0) * 4.0 * tn * nc + tn + nc;
    const double group = std::max({instr * (double)ceil_div(warps, 4), warps * (tn + nc) * 2.75, 1.7 * instr});
    return (double)H / 4.0 * group;
}

// In-cluster exchange against the device-wide one, cycles a step beyond the
// k-loop (fitted to per-step times of both on LSTM, GRU and RNN with hidden
// 128-512 and batch 1-128): about 5000 in a cluster (fenced remote stores,
// arrivals, the wait, the epilogue), about 8000 device-wide (publication,
// counter, tensor copy of h); the cluster's longer per-CTA k-loops ran about
// 1.3 times the model.
constexpr double kClusterExchangeCost = 5000.0;
constexpr double kDeviceExchangeCost = 8000.0;
constexpr double kClusterKloopScale = 1.3;

// Dataflow planner: cycles charged per piece of a product (a ring slot's
// wait, release and tensor copies).  Measured on GRU, hidden 2048, batch 4
// with R streamed: each halving of the piece adds about half a microsecond a
// step, more than the resident chunks it makes room for save.
constexpr double kDfPieceCost = 1000.0;

rnn_status plan_dataflow(rnn_plan* pl, int64_t N, const DeviceInfo& di, Geometry* out)
{
    const int64_t H = pl->H;
    const int G = pl->G, D = pl->D;
    const bool exact = pl->mode == RNN_MODE_EXACT;
    const int nchunks = (int)ceil_div(H, kRecKC);
    const int phases = (pl->op == RNN_OP_GRU && pl->lbr == 0) ? 2 : 1;
    const size_t smem_cap = (size_t)di.smem_optin - 1024;   // static shared: mbarriers, flags
    if (H % 4 != 0 || H > (1 << 20))
        return fail(RNN_ERR_UNSUPPORTED, "the dataflow kernel needs hidden_size a multiple of 4");
    double best_cost = 1e300;
    bool found = false;
    const int cr_auto[6] = {1, 2, 4, 8, 16, 32};
    const int ncr = pl->ov_rows > 0 ? 1 : 6;
    for (int cri = 0; cri < ncr; ++cri) {
        const int CRc = pl->ov_rows > 0 ? pl->ov_rows : cr_auto[cri];
        // rows per group padded to 8; a single group of at most 4 rows to 4
        // (padding rows skip their products but still take lanes: a batch of
        // 4 in an 8-row group left half of every warp idle).  Measured: 4-row
        // groups elsewhere (LSTM batch 32 as 8 groups) were slower than 8.
        const int64_t NRP = round_up(ceil_div(N, CRc), (CRc == 1 && N <= 4) ? 4 : 8);
        const int CR = (int)ceil_div(N, NRP);
        if (CR != CRc) continue;                                   // would leave an empty row group
        if (NRP > 256) continue;                                   // a tensor-copy box spans at most 256 rows
        const int64_t cu_cap = pl->ov_units > 0 ? pl->ov_units : di.sms / ((int64_t)D * CR);
        if (cu_cap < 1) continue;
        for (int rr = 1; rr >= 0; --rr) {
            if (pl->ov_rres >= 0 && rr != (pl->ov_rres == 2 ? 0 : pl->ov_rres)) continue;
            const int quant = 1;
            const int64_t Q = H;
            int64_t CU = std::min<int64_t>(cu_cap, Q);
            const int64_t qmax = ceil_div(Q, CU);
            if (pl->ov_units <= 0) CU = ceil_div(Q, qmax);
            const int umax = (int)(qmax * quant);
            if ((int64_t)D * CR > kMaxFlags) continue;
            int tn = 0;
            const int tlist[4] = {1, 2, 4, 8};
            for (int t : tlist) {
                if (pl->ov_tn > 0 && t != pl->ov_tn) continue;
                if (NRP % t) continue;
                const int cap = (t == 1 || t == 8) ? 224 : 352;   // the kernel's launch bound, less the loader
                if ((int64_t)umax * (NRP / t) <= cap) { tn = t; break; }
            }
            if (!tn) continue;
            if (rr == 0 && (H < kDfPitch || umax > 256)) continue;   // R boxes: 36 k wide, <= 256 units
            // gate split (GRU, one row per thread, one product per step): three
            // lanes share a (unit, row) and take a gate column each, when that
            // fits the launch bound (a warp holds ten such groups).  Measured:
            // 5-9% faster on GRU with batch 4, hidden 256-2048; LSTM with four
            // lanes per (unit, row) (batch 8, hidden 1024) was 47% slower, its
            // h loads quadrupled.
            int gs = 1;
            if (pl->op == RNN_OP_GRU && tn == 1 && phases == 1 && ceil_div((int64_t)umax * NRP, 32 / G) * 32 <= 224)
                gs = G;
            const int compute = gs == 1 ? (int)round_up((int64_t)umax * (NRP / tn), 32)
                                        : (int)ceil_div((int64_t)umax * NRP, 32 / G) * 32;
            // pieces: the whole block in one tensor copy per product (measured:
            // every extra piece boundary costs more than the earlier start
            // it buys), halved until the ring holds two pieces
            int cpb0 = 0, slots0 = 0;
            for (int c = nchunks; c >= 1; c /= 2) {
                const size_t fixed = df_smem_bytes((int)H, umax, G, (int)NRP, rr, c, 0);
                const size_t per_slot = df_smem_bytes((int)H, umax, G, (int)NRP, rr, c, 1) - fixed;
                if (fixed + 2 * per_slot > smem_cap) continue;
                const int np = (int)ceil_div(nchunks, c);
                cpb0 = c;
                slots0 = (int)std::min<size_t>(std::min<size_t>((size_t)kMaxSlots, (size_t)2 * np * phases),
                                               (smem_cap - fixed) / per_slot);
                break;
            }
            if (cpb0 == 0 || slots0 < 2) continue;
            // streamed R: besides the ring alone, smaller pieces in a ring of
            // 2-4 slots with as many leading pieces of R resident as the rest
            // of shared memory holds
            struct Ring { int cpb, slots, res; };
            Ring cands[48];
            int ncand = 0;
            if (pl->ov_rres != 2) cands[ncand++] = {cpb0, slots0, 0};   // 2: only partly resident
            if (!rr && pl->ov_rres != 0)
                for (int c = cpb0; c >= 1 && ncand + 3 <= 48; c /= 2) {
                    const int np = (int)ceil_div(nchunks, c);
                    for (int sl = 2; sl <= 4; ++sl) {
                        int r = 0;
                        while (r + 1 < np &&
                               df_smem_bytes((int)H, umax, G, (int)NRP, 0, c, sl, (r + 1) * c) <= smem_cap)
                            ++r;
                        if (r > 0) cands[ncand++] = {c, sl, r * c};
                    }
                }
            for (int ci = 0; ci < ncand; ++ci) {
                const int cpb = cands[ci].cpb, slots = cands[ci].slots, res = cands[ci].res;
                const int np = (int)ceil_div(nchunks, cpb);
                const size_t smem = df_smem_bytes((int)H, umax, G, (int)NRP, rr, cpb, slots, res);
                if (smem > smem_cap) continue;
                const double wps = (double)ceil_div(compute / 32, 4);
                const double per_k = ((exact ? 2.0 : 1.0) * 4.0 * tn * G + tn + G) / 4.0;
                const double kloop = (double)H * per_k * wps;
                // GRU with linear_before_reset = 0 streams each gate's rows once a
                // step (z and r in the first product, the candidate's in the second)
                const double bytes =
                    (double)NRP * H * 4 * phases + (rr ? 0.0 : (double)(H - res * kRecKC) * umax * G * 4);
                const double fetch = bytes / 64.0 * (slots >= np * phases ? 0.5 : 1.0);
                const double cost = kloop + fetch + kDfPieceCost * np * phases + 600.0 * tn * phases + 2500.0 * phases;
                if (cost >= best_cost) continue;
                int blocks = 0;
                cudaError_t e = recurrent_occupancy(pl->op, pl->lbr, 2, tn, exact, compute + 32, smem, &blocks, gs);
                if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
                if (blocks < 1 || (int64_t)D * CR * CU > (int64_t)blocks * di.sms) continue;
                best_cost = cost;
                found = true;
                out->kernel = 2;
                out->units = (int)CU;
                out->rows = CR;
                out->ctas = (int)CU * CR;
                out->quant = quant;
                out->slots = slots;
                out->umax = umax;
                out->tn = tn;
                out->threads = compute + 32;
                out->rres = rr;
                out->smem = smem;
                out->npad = (int)NRP;
                out->hpad = (int)round_up(H, kRecKC);
                out->cpb = cpb;
                out->res_chunks = res;
                out->ustride = df_unit_stride(rr ? (int)H : res * kRecKC, G);
                out->ufast = tn >= 4 ? 1 : 0;
                out->gs = gs;
            }
        }
    }
    if (!found)
        return fail(RNN_ERR_UNSUPPORTED, "no dataflow launch fits batch %lld, hidden %lld", (long long)N,
                    (long long)H);
    return RNN_OK;
}

// Dataflow kernel with the in-cluster exchange: each row group of a direction
// is one cluster of CU <= 16 CTAs that hold all of R between them (resident)
// and pass h through each other's shared memory; no device-wide counters.
// Cost (cycles a step): the k-loop as in plan_dataflow, the remote stores
// of h (every value to every CTA of the cluster) and a fixed exchange.
rnn_status plan_cluster(rnn_plan* pl, int64_t N, const DeviceInfo& di, Geometry* out, double* cost_out)
{
    const int64_t H = pl->H;
    const int G = pl->G, D = pl->D;
    const bool exact = pl->mode == RNN_MODE_EXACT;
    const bool two = pl->op == RNN_OP_GRU && pl->lbr == 0;
    const int phases = two ? 2 : 1;
    const size_t smem_cap = (size_t)di.smem_optin - 1024;
    if (H % 4 != 0 || H > (1 << 20))
        return fail(RNN_ERR_UNSUPPORTED, "the in-cluster dataflow kernel needs hidden_size a multiple of 4");
    if (pl->ov_rres == 0 || pl->ov_rres == 2)
        return fail(RNN_ERR_UNSUPPORTED, "the in-cluster dataflow kernel keeps all of R resident");
    double best = 1e300;
    bool found = false;
    const int cr_auto[6] = {1, 2, 4, 8, 16, 32};
    const int ncr = pl->ov_rows > 0 ? 1 : 6;
    for (int cri = 0; cri < ncr; ++cri) {
        const int CRc = pl->ov_rows > 0 ? pl->ov_rows : cr_auto[cri];
        const int64_t NRP = round_up(ceil_div(N, CRc), (CRc == 1 && N <= 4) ? 4 : 8);
        const int CR = (int)ceil_div(N, NRP);
        if (CR != CRc || NRP > 256) continue;
        for (int CU = 16; CU >= 1; --CU) {
            if (pl->ov_units > 0 && CU != pl->ov_units) continue;
            if (CU > H) continue;
            const int umax = (int)ceil_div(H, CU);
            if (ceil_div(H, umax) != CU) continue;                      // a CTA without units
            const size_t smem = df_cluster_smem_bytes((int)H, umax, G, (int)NRP, two);
            if (smem > smem_cap) continue;
            // two rows per thread only when asked for (kernel 5): measured
            // slower (GRU hidden 256 batch 16: 5.5 vs 3.9 us a step)
            for (int tn = 1; tn <= (pl->ov_kernel == 5 ? 2 : 1); ++tn) {
                if (pl->ov_tn > 0 && tn != pl->ov_tn) continue;
                if (NRP % tn) continue;
                const int64_t thr = (int64_t)umax * (NRP / tn);
                if (thr > (tn == 1 ? 224 : 352)) continue;
                const int compute = (int)round_up(thr, 32);
                const double kloop = kloop_cycles(H, compute / 32, tn, G, exact) * kClusterKloopScale;
                const double stores = (double)tn * CU * phases * 8.0;
                const double cost = kloop + stores + kClusterExchangeCost * phases;
                if (cost >= best) continue;
                int clusters = 0;
                cudaError_t e = cluster_occupancy(pl->op, pl->lbr, tn, exact, D * CR * CU, CU, compute + 32, smem,
                                                  &clusters);
                if (e != cudaSuccess) {
                    cudaGetLastError();
                    continue;
                }
                if (clusters < 1) continue;
                // clusters beyond those that fit at once run in later waves;
                // more CTAs than SMs share them
                const double waves = std::max(std::ceil((double)D * CR / clusters),
                                              (double)D * CR * CU / di.sms);
                if (cost * waves >= best) continue;
                best = cost * waves;
                found = true;
                *out = Geometry{};
                out->kernel = 2;
                out->cluster = 1;
                out->units = CU;
                out->rows = CR;
                out->ctas = CU * CR;
                out->quant = 1;
                out->slots = 1;
                out->umax = umax;
                out->tn = tn;
                out->threads = compute + 32;
                out->rres = 1;
                out->smem = smem;
                out->npad = (int)NRP;
                out->hpad = (int)round_up(H, kRecKC);
                out->cpb = (int)ceil_div(H, kRecKC);
                out->res_chunks = 0;
                out->ustride = df_unit_stride((int)H, G);
                out->ufast = 0;
                out->gs = 1;
            }
        }
    }
    if (!found)
        return fail(RNN_ERR_UNSUPPORTED, "no in-cluster dataflow launch fits batch %lld, hidden %lld", (long long)N,
                    (long long)H);
    if (cost_out) *cost_out = best;
    return RNN_OK;
}

// The tensor-core recurrent kernel keeps h in fp16: it is used only when
// every h the operator produces is bounded, i.e. the activation that makes h
// is one of Tanh, Sigmoid, ScaledTanh, HardSigmoid, Softsign (and, for GRU,
// the update gate z is in [0, 1]: Sigmoid or HardSigmoid).
bool tc_bounded_h(const rnn_plan* pl)
{
    auto bounded = [](int fn) { return fn == 1 || fn == 2 || fn == 6 || fn == 7 || fn == 9; };
    for (int d = 0; d < pl->D; ++d) {
        const int f = pl->act[d][0].fn, g = pl->act[d][1].fn, h = pl->act[d][2].fn;
        if (pl->op == RNN_OP_RNN && !bounded(f)) return false;
        if (pl->op == RNN_OP_GRU && !((f == 2 || f == 7) && bounded(g))) return false;
        if (pl->op == RNN_OP_LSTM && !(bounded(f) && bounded(h))) return false;
    }
    return true;
}

rnn_status plan_tc(rnn_plan* pl, int64_t N, const DeviceInfo& di, Geometry* out)
{
    const int64_t H = pl->H;
    const int G = pl->G, D = pl->D;
    if (N > 128) return fail(RNN_ERR_UNSUPPORTED, "the tensor-core kernel takes at most 128 batch rows");
    if (H % 8 != 0) return fail(RNN_ERR_UNSUPPORTED, "the tensor-core kernel needs hidden_size a multiple of 8");
    const bool two = pl->op == RNN_OP_GRU && pl->lbr == 0;   // z, r product, then the candidate's
    if (!tc_bounded_h(pl)) return fail(RNN_ERR_UNSUPPORTED, "the tensor-core kernel needs bounded h activations");
    int64_t C = std::min<int64_t>(di.sms / D, H);
    if (pl->ov_units > 0) C = std::min<int64_t>(pl->ov_units, H);
    if (C < 1) return fail(RNN_ERR_UNSUPPORTED, "no SM for the tensor-core kernel");
    const int64_t U = ceil_div(H, C);
    C = ceil_div(H, U);
    const int NP = (int)round_up(U * (two ? 2 : G), 16);
    const int NP2 = two ? (int)round_up(U, 16) : 0;
    if (NP > tc_recurrent_max_columns() || U > tc_recurrent_max_units(pl->op))
        return fail(RNN_ERR_UNSUPPORTED, "hidden_size %lld is too large for the tensor-core kernel", (long long)H);
    // h ring: as many 16 KB stages as fit (at least 2)
    const size_t cap = (size_t)di.smem_optin - 2048;
    const size_t fixed = tc_recurrent_smem((int)H, NP + NP2, (int)U, 0);
    const size_t per_stage = tc_recurrent_smem((int)H, NP + NP2, (int)U, 1) - fixed;
    if (fixed + 2 * per_stage > cap) return fail(RNN_ERR_UNSUPPORTED, "tensor-core kernel: shared memory");
    const int stages = (int)std::min<size_t>((size_t)tc_recurrent_max_stages(), (cap - fixed) / per_stage);
    const size_t smem = tc_recurrent_smem((int)H, NP + NP2, (int)U, stages);
    int blocks = 0;
    cudaError_t e = tc_recurrent_occupancy(pl->op, two, smem, &blocks);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (blocks < 1 || (int64_t)D * C > (int64_t)blocks * di.sms)
        return fail(RNN_ERR_UNSUPPORTED, "tensor-core kernel: the grid does not fit");
    *out = Geometry{};
    out->kernel = 3;
    out->units = (int)C;
    out->rows = 1;
    out->ctas = (int)C;
    out->quant = 1;
    out->umax = (int)U;
    out->tn = 1;
    out->threads = tc_recurrent_threads();
    out->rres = 1;
    out->smem = smem;
    out->npad = NP;
    out->npad2 = NP2;
    out->slots = stages;
    return RNN_OK;
}

// Launch geometry of the recurrent kernel for batch N.
rnn_status plan_geometry(rnn_plan* pl, int64_t N, const DeviceInfo& di, const float* R, Geometry* g)
{
    if (pl->ov_kernel == 1) return plan_staged(pl, N, di, g);
    if (pl->ov_kernel == 3) return plan_tc(pl, N, di, g);
    if (pl->ov_kernel == 5 && (uintptr_t)(pl->const_weights ? pl->r_orig_const : R) % 16 != 0)
        return fail(RNN_ERR_UNSUPPORTED, "the dataflow kernel needs R 16-byte aligned");
    // tensor-core modes: the tensor-core kernel for batches of 32..128 rows
    if ((pl->mode == RNN_MODE_FAST_TF32 || pl->mode == RNN_MODE_FAST_BF16) && pl->ov_kernel == 0 && N >= 32) {
        const std::string saved = g_error;
        if (plan_tc(pl, N, di, g) == RNN_OK) return RNN_OK;
        g_error = saved;
    }
    // the dataflow kernel reads R (as given) with TMA: 16-byte aligned base
    const float* rsrc = pl->const_weights ? pl->r_orig_const : R;
    if ((uintptr_t)rsrc % 16 != 0) {
        if (pl->ov_kernel == 2) return fail(RNN_ERR_UNSUPPORTED, "the dataflow kernel needs R 16-byte aligned");
        return plan_staged(pl, N, di, g);
    }
    if (pl->ov_kernel == 2) return plan_dataflow(pl, N, di, g);
    if (pl->ov_kernel == 5) return plan_cluster(pl, N, di, g, nullptr);
    const int64_t H = pl->H;
    const long long macs = (long long)N * pl->G * H * H;
    if (macs <= 262144 && staged_single_cta_fits(H, N) && pl->ov_units <= 0 && pl->ov_rows <= 0)
        return plan_staged(pl, N, di, g);                          // one CTA per direction
    const std::string saved = g_error;
    // In-cluster exchange where all of R fits in the shared memory of at most
    // 16 CTAs per row group, with one row per thread and one product a step,
    // when the model above puts it below the device-wide exchange.  Measured
    // (exact, per step): LSTM hidden 128 batch 8 3.0 vs 4.1 us, LSTM 256
    // batch 4 4.1 vs 5.3, batch 32 4.4 vs 5.2, GRU 256 batch 16 3.8 vs 4.4,
    // RNN 512 batch 4 4.6 vs 5.4; slower with long per-CTA k-loops (LSTM 384
    // batch 16: 7.1 vs 6.6) or more clusters than fit at once (LSTM 256 batch
    // 128); GRU with linear_before_reset = 0 (two exchanges a step) gained
    // nothing.
    Geometry cg{};
    double ccost = 0.0;
    bool have_cl = false;
    if (!(pl->op == RNN_OP_GRU && pl->lbr == 0)) {
        have_cl = plan_cluster(pl, N, di, &cg, &ccost) == RNN_OK;
        g_error = saved;
    }
    if (plan_dataflow(pl, N, di, g) == RNN_OK) {
        if (have_cl) {
            const int nc = g->gs > 1 ? 1 : pl->G;
            const double dcost = kloop_cycles(H, (g->threads - 32) / 32, g->tn, nc, pl->mode == RNN_MODE_EXACT) +
                                 kDeviceExchangeCost;
            if (ccost < dcost) {
                *g = cg;
                return RNN_OK;
            }
        }
        // Measured on GB300: the dataflow kernel wins while a CTA's share of a
        // step is small (its per-step latency dominates: 512 to 2048 hidden,
        // a few rows); with more than about a million products per CTA and
        // step the staged kernel, with more threads per CTA, keeps its
        // arithmetic pipes busier.
        const double work = (double)g->umax * pl->G * g->npad * (double)H;
        if (work <= (double)(1 << 20)) return RNN_OK;
        Geometry st{};
        if (plan_staged(pl, N, di, &st) == RNN_OK) {
            *g = st;
            return RNN_OK;
        }
        g_error = saved;
        return plan_dataflow(pl, N, di, g);
    }
    g_error = saved;
    return plan_staged(pl, N, di, g);
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

rnn_status ensure_scratch(rnn_plan* pl, size_t bytes)
{
    if (!pl->ctrl) {
        cudaError_t e = cudaMalloc((void**)&pl->ctrl, kCtrlBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(control)");
        e = cudaMemset(pl->ctrl, 0, kCtrlBytes);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(control)");
    }
    if (bytes <= pl->scratch_bytes) return RNN_OK;
    if (pl->scratch) {
        cudaFree(pl->scratch);   // synchronises with outstanding work
        pl->scratch = nullptr;
        pl->scratch_bytes = 0;
    }
    cudaError_t e = cudaMalloc((void**)&pl->scratch, bytes);
    if (e != cudaSuccess) {
        pl->scratch = nullptr;
        return cuda_fail(e, "cudaMalloc(scratch)");
    }
    pl->scratch_bytes = bytes;
    return RNN_OK;
}

void record(rnn_plan* pl, int i, cudaStream_t s)
{
    if (pl->timing && pl->events_ready) {
        cudaEventRecord(pl->ev[pl->slot][i], s);
        pl->ev_used[pl->slot][i] = true;
    }
}

// Durations of one run's kernels (waits for that run).
cudaError_t slot_times(rnn_plan* pl, int slot, float* out)
{
    for (int i = 0; i < 5; ++i) {
        out[i] = 0.0f;
        if (!pl->ev_used[slot][i] || !pl->ev_used[slot][i + 1]) continue;
        cudaError_t e = cudaEventSynchronize(pl->ev[slot][i + 1]);
        if (e != cudaSuccess) return e;
        e = cudaEventElapsedTime(&out[i], pl->ev[slot][i], pl->ev[slot][i + 1]);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t harvest(rnn_plan* pl, int slot)
{
    if (!pl->slot_pending[slot]) return cudaSuccess;
    float t[5];
    cudaError_t e = slot_times(pl, slot, t);
    if (e != cudaSuccess) return e;
    for (int i = 0; i < 5; ++i) pl->totals_ms[i] += t[i];
    pl->totals_runs += 1;
    pl->slot_pending[slot] = false;
    return cudaSuccess;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on the driver library): a tiled fp32 map, no swizzle,
// out-of-range elements read as zero.
typedef CUresult (*TmapEncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

TmapEncodeFn tmap_encoder()
{
    static TmapEncodeFn fn = []() -> TmapEncodeFn {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<TmapEncodeFn>(f);
    }();
    return fn;
}

CUresult tmap_encode_raw(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                         const cuuint64_t* strides, const cuuint32_t* box, bool swizzle128 = false,
                         int dtype = 0)
{
    const TmapEncodeFn fn = tmap_encoder();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType dt = dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dtype == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), dims, strides, box,
              es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

rnn_status tmap_encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box)
{
    if (!tmap_encoder()) return fail(RNN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
    const CUresult r = tmap_encode_raw(map, base, rank, dims, strides, box);
    if (r != CUDA_SUCCESS) return fail(RNN_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return RNN_OK;
}

struct RunArgs {
    int64_t S, N;
    const float *X, *W, *R, *B;
    const int32_t* lens;
    const float *h0, *c0, *P;
    float *Y, *Yh, *Yc;
    cudaStream_t st;
};

// Checks that need no device work: sizes, required pointers, the scratch
// limit.  Sets *done when the zero-size rule applies (after queueing the
// copies of the initial states).
rnn_status check_run(rnn_plan* pl, RunArgs& a, bool* done)
{
    *done = false;
    if (a.S < 0 || a.N < 0) return fail(RNN_ERR_INVALID_ARGUMENT, "seq_length and batch_size must be >= 0");
    if (a.S > (1 << 30) || a.N > (1 << 24)) return fail(RNN_ERR_UNSUPPORTED, "seq_length or batch_size too large");
    const int64_t H = pl->H, I = pl->I, GH = (int64_t)pl->G * H, D = pl->D;
    if (pl->op != RNN_OP_LSTM) { a.c0 = nullptr; a.P = nullptr; a.Yc = nullptr; }
    // Limits: per-direction scratch below 2^30 floats.
    const double per_dir = (double)a.S * a.N * GH + 4.0 * a.N * H + (pl->const_weights ? 0.0 : (double)GH * (I + H));
    if (per_dir >= 1073741824.0)
        return fail(RNN_ERR_UNSUPPORTED, "per-direction scratch of %.0f floats reaches the 2^30 limit", per_dir);
    // Zero-size: nothing runs; final states are the initial states or zeros.
    if (a.S == 0 || a.N == 0) {
        const size_t sb = (pl->io == 0 ? sizeof(float) : 2) * (size_t)D * a.N * H;
        cudaError_t e = cudaSuccess;
        if (a.Yh && sb)
            e = a.h0 ? cudaMemcpyAsync(a.Yh, a.h0, sb, cudaMemcpyDeviceToDevice, a.st) : cudaMemsetAsync(a.Yh, 0, sb, a.st);
        if (e == cudaSuccess && a.Yc && sb)
            e = a.c0 ? cudaMemcpyAsync(a.Yc, a.c0, sb, cudaMemcpyDeviceToDevice, a.st) : cudaMemsetAsync(a.Yc, 0, sb, a.st);
        if (e != cudaSuccess) return cuda_fail(e, "zero-size copy");
        *done = true;
        return RNN_OK;
    }
    if (!a.X && I > 0) return fail(RNN_ERR_INVALID_ARGUMENT, "X is NULL");
    if (!pl->const_weights && (!a.R || (!a.W && I > 0))) return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are required");
    return RNN_OK;
}

// sequence_lens already copied to `host`: check every length, find the longest.
rnn_status check_lengths(const int32_t* host, int64_t N, int64_t S, int64_t* max_len)
{
    *max_len = 0;
    for (int64_t n = 0; n < N; ++n) {
        const int32_t L = host[n];
        if (L < 0 || (int64_t)L > S)
            return fail(RNN_ERR_INVALID_INPUT, "sequence_lens[%lld] = %d is outside [0, %lld]", (long long)n, L,
                        (long long)S);
        *max_len = std::max<int64_t>(*max_len, L);
    }
    return RNN_OK;
}

struct Layout {
    size_t wt, rt, rp, xw, xb, xf, hb, rh, perm, total;
    bool need_rh;
};

// Scratch layout after `base` bytes (control words live elsewhere).
Layout scratch_layout(const rnn_plan* pl, const Geometry& geo, int64_t S, int64_t N, size_t base)
{
    const int64_t H = pl->H, I = pl->I, GH = (int64_t)pl->G * H, D = pl->D;
    Layout L;
    size_t off = base;
    L.wt = off; off += pl->const_weights ? 0 : align256(sizeof(float) * (size_t)I * D * GH);
    L.rt = off; off += (pl->const_weights || geo.kernel != 1) ? 0 : align256(sizeof(float) * (size_t)D * H * GH);
    L.rp = off; off += (pl->const_weights || geo.kernel != 3) ? 0 : align256((size_t)2 * D * GH * H);   // R fp16
    L.xw = off; off += align256(sizeof(float) * (size_t)S * N * D * GH);
    L.xb = off; off += pl->mode == RNN_MODE_FAST_BF16 ? align256((size_t)2 * S * N * I) : 0;   // X as bf16
    L.xf = off; off += pl->io != 0 ? align256(sizeof(float) * (size_t)S * N * I) : 0;          // fp16/bf16 X widened
    const size_t row = geo.kernel == 2 ? (size_t)geo.hpad / kRecKC * kDfPitch : (size_t)H;
    const size_t hbuf = geo.kernel == 3 ? (size_t)2 * 2 * D * 128 * H   // fp16 [2][D][128][H]
                                        : sizeof(float) * (size_t)D * 2 * geo.rows * geo.npad * row;
    L.hb = off; off += align256(hbuf);
    L.need_rh = pl->op == RNN_OP_GRU && pl->lbr == 0;
    L.rh = off; off += L.need_rh ? align256(hbuf) : 0;
    L.perm = off; off += (geo.kernel == 1 || geo.kernel == 2) ? align256(sizeof(int32_t) * (size_t)N) : 0;   // rows by length
    L.total = off;
    return L;
}

// The recurrent kernels need every CTA of their grid resident at once (they
// wait on one another every step).  Two of them launched on different streams
// may each get only part of the SMs and then wait for CTAs that cannot be
// placed until a wait limit runs out.  So recurrent launches on one device
// are put in one order: each waits, through an event, for the previous one,
// whichever stream or plan it came from.  Work captured into a graph is left
// alone (an event from outside a capture cannot be waited on inside it).
struct RecurrentGate {
    std::mutex m;
    cudaEvent_t last = nullptr;
};

template <class F>
cudaError_t launch_ordered(cudaStream_t st, F launch)
{
    static RecurrentGate gates[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(st, &cs);
    if (e != cudaSuccess) return e;
    if (cs != cudaStreamCaptureStatusNone || dev < 0 || dev >= 64) return launch();
    RecurrentGate& g = gates[dev];
    std::lock_guard<std::mutex> lock(g.m);
    if (!g.last) {
        e = cudaEventCreateWithFlags(&g.last, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            g.last = nullptr;
            return e;
        }
    } else {
        e = cudaStreamWaitEvent(st, g.last, 0);
        if (e != cudaSuccess) return e;
    }
    e = launch();
    if (e != cudaSuccess) return e;
    return cudaEventRecord(g.last, st);
}

cudaError_t launch_recurrent_ordered(const RecParams& p, const Geometry& geo, bool exact, cudaStream_t st)
{
    return launch_ordered(st, [&]() {
        return geo.kernel == 3 ? launch_tc_recurrent(p, geo.smem, st)
                               : launch_recurrent(p, exact, geo.threads, geo.smem, st);
    });
}

// Queue the kernels of one run.  `scratch` holds the layout, `ctrl` the
// control block (the set-up kernel zeroes its counters and flags).
rnn_status enqueue(rnn_plan* pl, const RunArgs& a, const Geometry& geo, int64_t max_len, char* scratch,
                   const Layout& L, char* ctrl, bool timed, long long spin_ns, int skip_cta, int* launches_out)
{
    const int64_t H = pl->H, I = pl->I, G = pl->G, D = pl->D, GH = G * H;
    const int64_t M = a.S * a.N;
    float* wt = pl->const_weights ? pl->wt_const : (float*)(scratch + L.wt);
    // tensor-core projection: W as K-major rows in the projection's column
    // order (the same scratch bytes as the k-major pack), and in BF16 mode X
    // and W rounded to bf16
    const bool bf16 = pl->mode == RNN_MODE_FAST_BF16;
    void* wk = pl->const_weights ? (bf16 ? pl->wkb_const : (void*)pl->wk_const) : (void*)(scratch + L.wt);
    // an fp16/bf16 X is widened to fp32 for the FP32 and TF32 projections; in
    // BF16 mode a bf16 X is the tensor-core operand as it stands
    const float* x32 = pl->io != 0 ? (const float*)(scratch + L.xf) : a.X;
    const bool x_is_bf16 = bf16 && pl->io == 2;
    const void* xin = bf16 ? (x_is_bf16 ? (const void*)a.X : (const void*)(scratch + L.xb)) : (const void*)x32;
    const bool use_tc = (pl->mode == RNN_MODE_FAST_TF32 || bf16) &&
                        projection_tc_supported(xin, wk ? wk : (const void*)scratch, (float*)(scratch + L.xw), M, I,
                                                D * GH, bf16);
    float* rt = pl->const_weights ? pl->rt_const : (float*)(scratch + L.rt);
    float* xw = (float*)(scratch + L.xw);
    const bool exact = pl->mode == RNN_MODE_EXACT;
    int launches = 0;
    cudaError_t e;
    if (timed) record(pl, 0, a.st);
    if (!pl->const_weights) {
        const bool pack_r = geo.kernel == 1;   // the dataflow kernel reads R as given, the tensor-core one fp16
        e = launch_pack(use_tc ? nullptr : a.W, pack_r ? a.R : nullptr, wt, pack_r ? rt : nullptr, (int)D, (int)G, H,
                        I, a.st);
        if (e != cudaSuccess) return cuda_fail(e, "pack launch");
        launches += (int)D * ((I > 0 && !use_tc ? 1 : 0) + (pack_r ? 1 : 0));
        if (use_tc) {
            e = launch_pack_kmajor(a.W, wk, (int)D, (int)G, H, I, bf16, a.st);
            if (e != cudaSuccess) return cuda_fail(e, "pack launch");
            launches += 1;
        }
    }
    if (geo.kernel == 3 && !pl->const_weights) {
        e = (pl->op == RNN_OP_GRU && pl->lbr == 0) ? launch_pack_r_split(a.R, scratch + L.rp, (int)D, H, a.st)
                                                    : launch_pack_kmajor(a.R, scratch + L.rp, (int)D, (int)G, H, H, 2, a.st);
        if (e != cudaSuccess) return cuda_fail(e, "pack launch");
        launches += 1;
    }
    if (use_tc && bf16) {
        if (!x_is_bf16) {
            e = pl->io == 0 ? launch_to_bf16(a.X, scratch + L.xb, M * I, a.st)
                            : launch_convert(a.X, pl->io, scratch + L.xb, 2, M * I, a.st);
            if (e != cudaSuccess) return cuda_fail(e, "bf16 conversion launch");
            launches += 1;
        }
    } else if (pl->io != 0 && M * I > 0) {
        e = launch_convert(a.X, pl->io, scratch + L.xf, 0, M * I, a.st);
        if (e != cudaSuccess) return cuda_fail(e, "X conversion launch");
        launches += 1;
    }
    if (timed) record(pl, 1, a.st);
    if (use_tc)
        e = launch_projection_tc(xin, wk, xw, M, I, D * GH, bf16, (int*)(ctrl + kCtrlStatusOffset), spin_ns, a.st);
    else
        e = launch_projection(x32, wt, xw, M, I, D * GH, exact, (int*)(ctrl + kCtrlStatusOffset), spin_ns, a.st);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    launches += 1;
    if (timed) record(pl, 2, a.st);

    RecParams p;
    std::memset(&p, 0, sizeof p);
    p.op = pl->op; p.G = (int)G; p.D = (int)D; p.N = (int)a.N; p.H = (int)H; p.S = (int)a.S;
    p.layout = pl->layout; p.lbr = pl->lbr; p.input_forget = pl->input_forget;
    p.has_B = a.B != nullptr; p.has_P = a.P != nullptr; p.has_h0 = a.h0 != nullptr; p.has_c0 = a.c0 != nullptr;
    p.has_lens = a.lens != nullptr; p.has_clip = pl->has_clip; p.clip = pl->clip;
    p.io = pl->io;
    for (int d = 0; d < 2; ++d)
        for (int s = 0; s < 3; ++s) p.act[d][s] = pl->act[d][s];
    p.max_len = (int)max_len;
    p.dir_reverse[0] = pl->direction == RNN_DIR_REVERSE ? 1 : 0;
    p.dir_reverse[1] = 1;
    p.kernel = geo.kernel;
    p.ctas_per_dir = geo.ctas; p.unit_groups = geo.units; p.row_groups = geo.rows; p.unit_quant = geo.quant;
    p.slots = geo.slots; p.umax = geo.umax; p.rows_per_thread = geo.tn; p.r_resident = geo.rres;
    p.res_chunks = geo.res_chunks;
    p.npad = geo.npad;
    p.npad2 = geo.npad2;
    p.hpad = geo.hpad;
    p.chunks_per_piece = geo.cpb;
    p.unit_stride = geo.ustride;
    p.unit_fastest = geo.ufast;
    p.gate_split = geo.kernel == 2 && geo.gs > 1 ? geo.gs : 1;
    p.cluster = geo.kernel == 2 && geo.cluster ? 1 : 0;
    p.XW = xw; p.Rt = rt; p.Rorig = pl->const_weights ? pl->r_orig_const : a.R; p.B = a.B; p.P = a.P; p.h0 = a.h0; p.c0 = a.c0; p.lens = a.lens;
    p.Y = a.Y; p.Yh = a.Yh; p.Yc = a.Yc;
    p.hbuf = (float*)(scratch + L.hb);
    p.rhbuf = L.need_rh ? (float*)(scratch + L.rh) : nullptr;
    p.bar = (unsigned*)ctrl;
    p.status = (int*)(ctrl + kCtrlStatusOffset);
    p.flags = (unsigned*)(ctrl + kCtrlFlagsOffset);
    p.spin_limit_ns = spin_ns;
    p.debug_skip_cta = skip_cta;
    if (geo.kernel == 3) {
        // h exchange buffer fp16 [2 buffers][D][128 rows][H]: box 64 k x 128 rows x 1;
        // R fp16 [D*G*H columns][H]: box 64 k x npad columns; both 128-byte swizzled
        const void* rp = pl->const_weights ? pl->rp16_const : (const void*)(scratch + L.rp);
        const cuuint64_t hdims[3] = {(cuuint64_t)H, 128, (cuuint64_t)(2 * D)};
        const cuuint64_t hstrides[2] = {(cuuint64_t)H * 2, (cuuint64_t)H * 2 * 128};
        // only the batch's rows (rounded up to an 8-row swizzle group) are
        // copied; the kernel keeps the other rows of its ring at zero
        const cuuint32_t hbox[3] = {64, (cuuint32_t)round_up(a.N, 8), 1};
        const cuuint64_t rdims[2] = {(cuuint64_t)H, (cuuint64_t)(D * GH)};
        const cuuint64_t rstrides[1] = {(cuuint64_t)H * 2};
        const cuuint32_t rbox[2] = {64, (cuuint32_t)geo.npad};
        if (!encode_tensor_map(&p.hmap, p.hbuf, 3, hdims, hstrides, hbox, true, 2) ||
            !encode_tensor_map(&p.rmap, rp, 2, rdims, rstrides, rbox, true, 2))
            return fail(RNN_ERR_CUDA, "tensor map for the tensor-core kernel");
        p.rhmap = p.hmap;   // GRU lbr = 0 only
        p.rmap2 = p.rmap;
        if (geo.npad2 > 0) {
            // GRU lbr = 0: the r (.) h exchange buffer (as h) and R's candidate rows (box npad2 rows)
            const cuuint32_t rbox2[2] = {64, (cuuint32_t)geo.npad2};
            if (!p.rhbuf || !encode_tensor_map(&p.rhmap, p.rhbuf, 3, hdims, hstrides, hbox, true, 2) ||
                !encode_tensor_map(&p.rmap2, rp, 2, rdims, rstrides, rbox2, true, 2))
                return fail(RNN_ERR_CUDA, "tensor map for the tensor-core kernel");
        }
    }
    if (geo.kernel == 2) {
        // h / r (.) h exchange buffers [D*2*CR blocks][hpad/32 chunks][npad rows][36],
        // box 36 x npad x cpb x 1 (one piece of one row group, contiguous)
        const cuuint64_t nck = (cuuint64_t)(geo.hpad / kRecKC);
        const cuuint64_t hdims[4] = {(cuuint64_t)kDfPitch, (cuuint64_t)geo.npad, nck, (cuuint64_t)(D * 2 * geo.rows)};
        const cuuint64_t hstrides[3] = {(cuuint64_t)kDfPitch * 4, (cuuint64_t)geo.npad * kDfPitch * 4,
                                        nck * geo.npad * kDfPitch * 4};
        const cuuint32_t hbox[4] = {(cuuint32_t)kDfPitch, (cuuint32_t)geo.npad, (cuuint32_t)geo.cpb, 1};
        rnn_status rs = tmap_encode(&p.hmap, p.hbuf, 4, hdims, hstrides, hbox);
        if (rs != RNN_OK) return rs;
        rs = tmap_encode(&p.rhmap, p.rhbuf ? p.rhbuf : p.hbuf, 4, hdims, hstrides, hbox);
        if (rs != RNN_OK) return rs;
        if (!geo.rres) {
            // R as given [D][G][H units][H k], box 36 x umax x gates x 1 (one
            // chunk; k past H reads 0): all G gates, or for GRU with
            // linear_before_reset = 0 the z and r rows (first product of a
            // step) and the candidate's rows (second product)
            const cuuint64_t rdims[4] = {(cuuint64_t)H, (cuuint64_t)H, (cuuint64_t)G, (cuuint64_t)D};
            const cuuint64_t rstrides[3] = {(cuuint64_t)H * 4, (cuuint64_t)H * H * 4, (cuuint64_t)G * H * H * 4};
            const bool two = pl->op == RNN_OP_GRU && pl->lbr == 0;
            const cuuint32_t rbox[4] = {(cuuint32_t)kDfPitch, (cuuint32_t)geo.umax, (cuuint32_t)(two ? 2 : G), 1};
            rs = tmap_encode(&p.rmap, p.Rorig, 4, rdims, rstrides, rbox);
            if (rs != RNN_OK) return rs;
            p.rmap2 = p.rmap;
            if (two) {
                const cuuint32_t rbox2[4] = {(cuuint32_t)kDfPitch, (cuuint32_t)geo.umax, 1, 1};
                rs = tmap_encode(&p.rmap2, p.Rorig, 4, rdims, rstrides, rbox2);
                if (rs != RNN_OK) return rs;
            }
        } else {
            p.rmap = p.hmap;   // unused
            p.rmap2 = p.hmap;
        }
    }

    if ((geo.kernel == 1 || geo.kernel == 2) && a.lens) {
        // the FP32 kernels take the rows longest first, so that finished row
        // tiles (and, with several per warp, whole warps) drop out of the
        // products
        p.perm = (const int32_t*)(scratch + L.perm);
        e = launch_rank_rows(a.lens, (int32_t*)(scratch + L.perm), (int)a.N, a.st);
        if (e != cudaSuccess) return cuda_fail(e, "row ranking launch");
        launches += 1;
    }
    e = geo.kernel == 3 ? launch_tc_state_init(p, a.st) : launch_state_init(p, a.st);
    if (e != cudaSuccess) return cuda_fail(e, "state set-up launch");
    launches += 1;
    if (timed) record(pl, 3, a.st);
    e = launch_recurrent_ordered(p, geo, exact, a.st);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent launch");
    launches += 1;
    if (timed) record(pl, 4, a.st);
    if (a.Y && max_len < a.S) {
        e = launch_mask_tail(a.Y, pl->layout, a.S, D, a.N, H, max_len, pl->io, a.st);
        if (e != cudaSuccess) return cuda_fail(e, "mask launch");
        launches += 1;
    }
    if (timed) record(pl, 5, a.st);
    pl->g_units = geo.units; pl->g_tn = geo.tn; pl->g_rres = geo.rres; pl->g_rows = geo.rows;
    pl->g_kernel = geo.kernel == 2 && geo.cluster ? 5 : geo.kernel; pl->g_threads = geo.threads; pl->g_smem = (int)geo.smem;
    *launches_out = launches;
    return RNN_OK;
}

}  // namespace

struct rnn_stack {
    std::vector<rnn_plan*> layers;   // the caller's plans, borrowed
    void* buf[2] = {nullptr, nullptr};
    size_t cap[2] = {0, 0};
    int last_launches = 0;
    int wave_mode = 1;               // 0: layer by layer; 1: the wavefront where it is measured faster;
                                     // 2: the wavefront whenever the stack qualifies
    bool last_wave = false;          // the last run used the wavefront kernel
    void* wbuf = nullptr;            // the wavefront run's scratch
    size_t wcap = 0;
};

namespace {

// Layers chain by the output sequence: layer l+1's input_size is layer l's
// dirs * hidden; one layout and one activation element type throughout.
rnn_status stack_check(const rnn_stack* st)
{
    for (size_t l = 0; l < st->layers.size(); ++l) {
        const rnn_plan* pl = st->layers[l];
        if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "layer %zu: plan is NULL", l);
        if (pl->cell) return fail(RNN_ERR_INVALID_ARGUMENT, "layer %zu: a cell plan cannot be stacked", l);
        if (l == 0) continue;
        const rnn_plan* prev = st->layers[l - 1];
        if (pl->layout != prev->layout) return fail(RNN_ERR_INVALID_ARGUMENT, "layer %zu: layout differs", l);
        if (pl->io != prev->io) return fail(RNN_ERR_INVALID_ARGUMENT, "layer %zu: io type differs", l);
        if (pl->I != (int64_t)prev->D * prev->H)
            return fail(RNN_ERR_INVALID_ARGUMENT, "layer %zu: input_size %lld, the layer below gives %lld", l,
                        (long long)pl->I, (long long)prev->D * prev->H);
    }
    return RNN_OK;
}

}  // namespace

extern "C" {

const char* rnn_last_error(void) { return g_error.c_str(); }

rnn_status rnn_plan_create(rnn_plan_t* out, int op, int direction, int64_t hidden_size, int64_t input_size,
                           const char* const* activations, int n_activations, const float* alpha,
                           int n_alpha, const float* beta, int n_beta, float clip, int layout,
                           int linear_before_reset, int input_forget)
{
    g_error.clear();
    if (!out) return fail(RNN_ERR_INVALID_ARGUMENT, "out is NULL");
    *out = nullptr;
    if (op < 0 || op > 2) return fail(RNN_ERR_INVALID_ARGUMENT, "unknown op %d", op);
    if (direction < 0 || direction > 2) return fail(RNN_ERR_INVALID_ARGUMENT, "unknown direction %d", direction);
    if (hidden_size <= 0) return fail(RNN_ERR_INVALID_ARGUMENT, "hidden_size must be positive");
    if (hidden_size > (1 << 20)) return fail(RNN_ERR_UNSUPPORTED, "hidden_size too large");
    if (input_size < 0) return fail(RNN_ERR_INVALID_ARGUMENT, "input_size must be >= 0");
    if (layout != 0 && layout != 1) return fail(RNN_ERR_INVALID_ARGUMENT, "layout must be 0 or 1");
    if (linear_before_reset != 0 && linear_before_reset != 1)
        return fail(RNN_ERR_INVALID_ARGUMENT, "linear_before_reset must be 0 or 1");
    if (input_forget != 0 && input_forget != 1)
        return fail(RNN_ERR_INVALID_ARGUMENT, "input_forget must be 0 or 1");
    if (n_activations < 0 || n_alpha < 0 || n_beta < 0)
        return fail(RNN_ERR_INVALID_ARGUMENT, "negative list length");

    const int k = acts_per_dir(op);
    const int D = direction == RNN_DIR_BIDIRECTIONAL ? 2 : 1;
    ActSpec list[6];
    int nlist = 0;
    if (n_activations == 0) {
        const int defaults[3][3] = {{1, -1, -1}, {2, 1, -1}, {2, 1, 1}};   // Tanh | Sigmoid,Tanh | S,T,T
        for (int i = 0; i < k; ++i) {
            const int id = defaults[op][i];
            list[i] = {id, kActs[id].alpha0, kActs[id].beta0};
        }
        nlist = k;
    } else {
        if (n_activations != k && n_activations != 2 * k)
            return fail(RNN_ERR_INVALID_ARGUMENT, "expected %d or %d activations, got %d", k, 2 * k,
                        n_activations);
        if (!activations) return fail(RNN_ERR_INVALID_ARGUMENT, "activations is NULL");
        int ca = 0, cb = 0;   // separate cursors over alpha and beta
        for (int i = 0; i < n_activations; ++i) {
            const int id = act_id(activations[i]);
            if (id < 0)
                return fail(RNN_ERR_INVALID_ARGUMENT, "unknown activation '%s'",
                            activations[i] ? activations[i] : "(null)");
            ActSpec a{id, kActs[id].alpha0, kActs[id].beta0};
            if (kActs[id].takes_alpha) {
                if (alpha && ca < n_alpha) a.alpha = alpha[ca];
                ++ca;
            }
            if (kActs[id].takes_beta) {
                if (beta && cb < n_beta) a.beta = beta[cb];
                ++cb;
            }
            list[i] = a;
        }
        nlist = n_activations;
    }

    rnn_plan* pl = new (std::nothrow) rnn_plan();
    if (!pl) return fail(RNN_ERR_OOM, "out of host memory");
    pl->op = op;
    pl->direction = direction;
    pl->D = D;
    pl->G = gates_of(op);
    pl->layout = layout;
    pl->lbr = op == RNN_OP_GRU ? linear_before_reset : 0;
    pl->input_forget = op == RNN_OP_LSTM ? input_forget : 0;
    pl->H = hidden_size;
    pl->I = input_size;
    pl->has_clip = clip > 0.0f ? 1 : 0;   // NaN and <= 0: no clip
    pl->clip = pl->has_clip ? clip : 0.0f;
    for (int d = 0; d < 2; ++d)
        for (int s = 0; s < 3; ++s) {
            const int base = (nlist == 2 * k && d == 1) ? k : 0;
            pl->act[d][s] = s < k ? list[base + s] : ActSpec{-1, 0.0f, 0.0f};
        }
    *out = pl;
    return RNN_OK;
}

void rnn_plan_destroy(rnn_plan_t pl)
{
    if (!pl) return;
    if (pl->ran) cudaDeviceSynchronize();
    if (pl->scratch) cudaFree(pl->scratch);
    if (pl->ctrl) cudaFree(pl->ctrl);
    if (pl->wt_const) cudaFree(pl->wt_const);
    if (pl->wk_const) cudaFree(pl->wk_const);
    if (pl->wkb_const) cudaFree(pl->wkb_const);
    if (pl->rp16_const) cudaFree(pl->rp16_const);
    if (pl->rt_const) cudaFree(pl->rt_const);
    if (pl->r_orig_const) cudaFree(pl->r_orig_const);
    if (pl->lens_host) cudaFreeHost(pl->lens_host);
    if (pl->events_ready)
        for (auto& set : pl->ev)
            for (auto& e : set) cudaEventDestroy(e);
    if (pl->done_ready) cudaEventDestroy(pl->done);
    delete pl;
}

rnn_status rnn_plan_set_mode(rnn_plan_t pl, int mode)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (mode != RNN_MODE_EXACT && mode != RNN_MODE_FAST && mode != RNN_MODE_FAST_TF32 && mode != RNN_MODE_FAST_BF16)
        return fail(RNN_ERR_INVALID_ARGUMENT, "unknown mode %d", mode);
    pl->mode = mode;
    return RNN_OK;
}

rnn_status rnn_plan_get_activation(rnn_plan_t pl, int dir, int slot, int* fn, float* alpha, float* beta)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (dir < 0 || dir >= pl->D || slot < 0 || slot > 2)
        return fail(RNN_ERR_INVALID_ARGUMENT, "direction or slot out of range");
    if (fn) *fn = pl->act[dir][slot].fn;
    if (alpha) *alpha = pl->act[dir][slot].alpha;
    if (beta) *beta = pl->act[dir][slot].beta;
    return RNN_OK;
}

rnn_status rnn_plan_set_launch(rnn_plan_t pl, int unit_groups, int rows_per_thread, int r_resident,
                               int row_groups, int kernel)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (unit_groups < 0 || rows_per_thread < 0 || r_resident < -1 || r_resident > 2 || row_groups < 0 ||
        kernel < 0 || kernel > 5 || kernel == 4)
        return fail(RNN_ERR_INVALID_ARGUMENT, "bad launch override");
    if (kernel == 3 && (row_groups > 1 || rows_per_thread > 1))
        return fail(RNN_ERR_INVALID_ARGUMENT, "the tensor-core kernel has one row group and one row per thread");
    if (rows_per_thread != 0 && rows_per_thread != 1 && rows_per_thread != 2 && rows_per_thread != 4 &&
        rows_per_thread != 8)
        return fail(RNN_ERR_INVALID_ARGUMENT, "rows_per_thread must be 0, 1, 2, 4 or 8");
    if (kernel == 1 && row_groups > 1) return fail(RNN_ERR_INVALID_ARGUMENT, "the staged kernel has one row group");
    if (kernel == 5 && (rows_per_thread > 2 || unit_groups > 16))
        return fail(RNN_ERR_INVALID_ARGUMENT, "the in-cluster kernel takes 1 or 2 rows per thread and <= 16 unit groups");
    pl->ov_units = unit_groups;
    pl->ov_tn = rows_per_thread;
    pl->ov_rres = r_resident;
    pl->ov_rows = row_groups;
    pl->ov_kernel = kernel;
    return RNN_OK;
}

rnn_status rnn_plan_get_launch(rnn_plan_t pl, int* unit_groups, int* rows_per_thread, int* r_resident,
                               int* row_groups, int* kernel, int* threads, int* smem_bytes)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (unit_groups) *unit_groups = pl->g_units;
    if (rows_per_thread) *rows_per_thread = pl->g_tn;
    if (r_resident) *r_resident = pl->g_rres;
    if (row_groups) *row_groups = pl->g_rows;
    if (kernel) *kernel = pl->g_kernel;
    if (threads) *threads = pl->g_threads;
    if (smem_bytes) *smem_bytes = pl->g_smem;
    return RNN_OK;
}

rnn_status rnn_plan_set_timing(rnn_plan_t pl, int enable)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (enable && !pl->events_ready) {
        for (auto& set : pl->ev)
            for (auto& e : set) {
                cudaError_t er = cudaEventCreate(&e);
                if (er != cudaSuccess) return cuda_fail(er, "cudaEventCreate");
            }
        pl->events_ready = true;
    }
    pl->timing = enable != 0;
    for (auto& b : pl->slot_pending) b = false;
    for (double& t : pl->totals_ms) t = 0.0;
    pl->totals_runs = 0;
    return RNN_OK;
}

rnn_status rnn_plan_last_timing(rnn_plan_t pl, float* out, int n)
{
    if (!pl || !out) return fail(RNN_ERR_INVALID_ARGUMENT, "plan or out is NULL");
    for (int i = 0; i < n; ++i) out[i] = 0.0f;
    if (!pl->events_ready || !pl->ran) return RNN_OK;
    // events: 0 start, 1 after pack, 2 after projection, 3 after set-up,
    // 4 after recurrence, 5 after mask
    float t[5];
    cudaError_t e = slot_times(pl, pl->slot, t);
    if (e != cudaSuccess) return cuda_fail(e, "reading timing events");
    for (int i = 0; i < 5 && i < n; ++i) out[i] = t[i];
    return RNN_OK;
}

rnn_status rnn_plan_timing_totals(rnn_plan_t pl, float* out, int n, int* runs)
{
    if (!pl || !out) return fail(RNN_ERR_INVALID_ARGUMENT, "plan or out is NULL");
    for (int s = 0; s < rnn_plan::kRing; ++s) {
        cudaError_t e = harvest(pl, s);
        if (e != cudaSuccess) return cuda_fail(e, "reading timing events");
    }
    for (int i = 0; i < n; ++i) out[i] = i < 5 ? (float)pl->totals_ms[i] : 0.0f;
    if (runs) *runs = pl->totals_runs;
    for (double& t : pl->totals_ms) t = 0.0;
    pl->totals_runs = 0;
    return RNN_OK;
}

rnn_status rnn_plan_debug_barrier(rnn_plan_t pl, int64_t spin_limit_ns, int skip_cta)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (spin_limit_ns < 0) return fail(RNN_ERR_INVALID_ARGUMENT, "negative limit");
    pl->spin_limit_ns = spin_limit_ns == 0 ? kDefaultSpinNs : spin_limit_ns;
    pl->skip_cta = skip_cta;
    return RNN_OK;
}

int rnn_plan_last_launch_count(rnn_plan_t pl) { return pl ? pl->last_launches : 0; }

rnn_status rnn_plan_sync(rnn_plan_t pl)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (!pl->ran) return RNN_OK;
    if (pl->last_static) {
        // a static-scratch run records no event of its own: wait for the
        // device, then read (and clear) the status word of the fixed array
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return cuda_fail(e, "waiting for the run");
        int st = 0;
        e = cudaMemcpy(&st, pl->static_status, sizeof st, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
        if (st != 0) {
            const int zero = 0;
            cudaMemcpy(pl->static_status, &zero, sizeof zero, cudaMemcpyHostToDevice);
            if (st == RNN_ERR_TIMEOUT)
                return fail(RNN_ERR_TIMEOUT, "a device-side wait (step barrier or copy) timed out; outputs are incomplete");
            return fail((rnn_status)st, "device reported status %d", st);
        }
        return RNN_OK;
    }
    cudaError_t e = pl->done_ready ? cudaEventSynchronize(pl->done) : cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "waiting for the run");
    if (!pl->ctrl) return RNN_OK;      // only cell runs so far: no device-side waits, no status word
    int st = 0;
    e = cudaMemcpy(&st, pl->ctrl + kCtrlStatusOffset, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    if (st != 0) {
        const int zero = 0;
        cudaMemcpy(pl->ctrl + kCtrlStatusOffset, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (st == RNN_ERR_TIMEOUT)
            return fail(RNN_ERR_TIMEOUT, "a device-side wait (step barrier or copy) timed out; outputs are incomplete");
        return fail((rnn_status)st, "device reported status %d", st);
    }
    return RNN_OK;
}

rnn_status rnn_plan_set_weights(rnn_plan_t pl, const float* W, const float* R, void* stream)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (!R || (!W && pl->I > 0)) return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are required");
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t GH = (int64_t)pl->G * pl->H;
    if (!pl->rt_const) {
        cudaError_t e = cudaMalloc((void**)&pl->rt_const, sizeof(float) * (size_t)pl->D * pl->H * GH);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(R pack)");
        if (pl->I > 0) {
            e = cudaMalloc((void**)&pl->wt_const, sizeof(float) * (size_t)pl->I * pl->D * GH);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(W pack)");
            e = cudaMalloc((void**)&pl->wk_const, sizeof(float) * (size_t)pl->I * pl->D * GH);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(W K-major pack)");
            e = cudaMalloc(&pl->wkb_const, 2 * (size_t)pl->I * pl->D * GH);
            if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(W bf16 pack)");
        }
    }
    if (!pl->r_orig_const) {
        cudaError_t e = cudaMalloc((void**)&pl->r_orig_const, sizeof(float) * (size_t)pl->D * GH * pl->H);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(R copy)");
        e = cudaMalloc(&pl->rp16_const, 2 * (size_t)pl->D * GH * pl->H);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(R fp16 pack)");
    }
    cudaError_t e = cudaMemcpyAsync(pl->r_orig_const, R, sizeof(float) * (size_t)pl->D * GH * pl->H,
                                    cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "copying R");
    e = launch_pack(W, R, pl->wt_const, pl->rt_const, pl->D, pl->G, pl->H, pl->I, s);
    if (e == cudaSuccess && pl->wk_const) e = launch_pack_kmajor(W, pl->wk_const, pl->D, pl->G, pl->H, pl->I, false, s);
    if (e == cudaSuccess && pl->wkb_const) e = launch_pack_kmajor(W, pl->wkb_const, pl->D, pl->G, pl->H, pl->I, true, s);
    if (e == cudaSuccess && pl->rp16_const)
        e = (pl->op == RNN_OP_GRU && pl->lbr == 0) ? launch_pack_r_split(R, pl->rp16_const, pl->D, pl->H, s)
                                                    : launch_pack_kmajor(R, pl->rp16_const, pl->D, pl->G, pl->H, pl->H, 2, s);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    pl->const_weights = true;
    return RNN_OK;
}

// sequence_lens (device) to the plan's pinned host buffer, every length
// checked against [0, S], the longest in *max_len.
static rnn_status read_lengths(rnn_plan_t pl, const int32_t* lens, int64_t N, int64_t S, cudaStream_t st,
                               int64_t* max_len)
{
    if (N > pl->lens_cap) {
        if (pl->lens_host) cudaFreeHost(pl->lens_host);
        pl->lens_host = nullptr;
        cudaError_t e = cudaMallocHost((void**)&pl->lens_host, sizeof(int32_t) * (size_t)N);
        if (e != cudaSuccess) { pl->lens_cap = 0; return cuda_fail(e, "cudaMallocHost(lens)"); }
        pl->lens_cap = N;
    }
    cudaError_t e = cudaMemcpyAsync(pl->lens_host, lens, sizeof(int32_t) * (size_t)N, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "copying sequence_lens");
    return check_lengths(pl->lens_host, N, S, max_len);
}

// One run of a plan.  known_max_len >= 0: sequence_lens was already checked
// (by a stack's first layer) and its maximum is known.
static rnn_status run_plan(rnn_plan_t pl, int64_t S, int64_t N, const float* X, const float* W, const float* R,
                    const float* B, const int32_t* lens, const float* h0, const float* c0, const float* P,
                    float* Y, float* Yh, float* Yc, void* stream, int64_t known_max_len, int64_t* max_len_out)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    pl->last_launches = 0;
    RunArgs a{S, N, X, W, R, B, lens, h0, c0, P, Y, Yh, Yc, (cudaStream_t)stream};
    bool done = false;
    rnn_status rs = check_run(pl, a, &done);
    if (max_len_out) *max_len_out = 0;
    if (rs != RNN_OK || done) return rs;

    DeviceInfo di;
    rs = device_info(&di);
    if (rs != RNN_OK) return rs;
    if (!di.coop) return fail(RNN_ERR_UNSUPPORTED, "device lacks cooperative launch");

    // sequence_lens: check on the host before anything is written.
    int64_t max_len = known_max_len >= 0 ? known_max_len : S;
    if (lens && known_max_len < 0) {
        rs = read_lengths(pl, lens, N, S, a.st, &max_len);
        if (rs != RNN_OK) return rs;
    }

    Geometry geo{};
    rs = plan_geometry(pl, N, di, R, &geo);
    if (rs != RNN_OK) return rs;
    const Layout L = scratch_layout(pl, geo, S, N, 0);
    rs = ensure_scratch(pl, std::max<size_t>(L.total, 256));
    if (rs != RNN_OK) return rs;
    if (pl->device < 0) cudaGetDevice(&pl->device);
    if (pl->timing && !pl->events_ready) {
        rs = rnn_plan_set_timing(pl, 1);
        if (rs != RNN_OK) return rs;
    }
    if (!pl->done_ready) {
        cudaError_t e = cudaEventCreateWithFlags(&pl->done, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
        pl->done_ready = true;
    }
    if (pl->timing) {
        pl->slot = (pl->slot + 1) % rnn_plan::kRing;
        cudaError_t eh = harvest(pl, pl->slot);   // a run kRing runs ago: long finished
        if (eh != cudaSuccess) return cuda_fail(eh, "reading timing events");
        for (bool& u : pl->ev_used[pl->slot]) u = false;
    }
    int launches = 0;
    pl->last_static = false;
    rs = enqueue(pl, a, geo, max_len, pl->scratch, L, pl->ctrl, pl->timing, pl->spin_limit_ns, pl->skip_cta,
                 &launches);
    if (rs != RNN_OK) return rs;
    if (pl->timing) pl->slot_pending[pl->slot] = true;
    cudaEventRecord(pl->done, a.st);
    pl->ran = true;
    pl->last_launches = launches;
    if (max_len_out) *max_len_out = max_len;
    return RNN_OK;
}

rnn_status rnn_run(rnn_plan_t pl, int64_t S, int64_t N, const float* X, const float* W, const float* R,
                   const float* B, const int32_t* lens, const float* h0, const float* c0, const float* P,
                   float* Y, float* Yh, float* Yc, void* stream)
{
    g_error.clear();
    return run_plan(pl, S, N, X, W, R, B, lens, h0, c0, P, Y, Yh, Yc, stream, -1, nullptr);
}

// ------------------------------------------------------------ stacked layers

rnn_status rnn_stack_create(rnn_stack_t* out, const rnn_plan_t* layers, int n_layers)
{
    g_error.clear();
    if (!out) return fail(RNN_ERR_INVALID_ARGUMENT, "out is NULL");
    *out = nullptr;
    if (n_layers < 1 || !layers) return fail(RNN_ERR_INVALID_ARGUMENT, "a stack needs at least one layer");
    rnn_stack* st = new (std::nothrow) rnn_stack();
    if (!st) return fail(RNN_ERR_OOM, "out of host memory");
    st->layers.assign(layers, layers + n_layers);
    rnn_status rs = stack_check(st);
    if (rs != RNN_OK) {
        delete st;
        return rs;
    }
    *out = st;
    return RNN_OK;
}

namespace {

// Launch geometry of the wavefront kernel: CTAs per layer in proportion to
// the layer's products per step (layer 0: the recurrent one; the others: the
// recurrent and the input one), all slices of R and W resident.
struct WaveGeometry {
    int tn = 0, threads = 0, ctas = 0, npad = 0;
    size_t smem = 0;
    int C[kWaveMaxLayers] = {}, umax[kWaveMaxLayers] = {}, ugp[kWaveMaxLayers] = {}, cta0[kWaveMaxLayers] = {};
};

// Products per step of a layer (batch x gate columns x k of both products)
// up to which the wavefront launch was measured faster than running the
// layers one after another: such layers leave most of a step to exchange
// latency, which the wavefront overlaps across the layers.  Larger layers
// keep the SMs busy on their own, and layer by layer their input products
// run in the projection GEMM, which is faster than the recurrent k-loop.
constexpr double kWaveMaxProducts = 8.0e6;

// Whether a stack can run as one wavefront launch; the reason if not.
bool wave_eligible(const rnn_stack* st, int64_t S, int64_t N, std::string* why)
{
    const int L = (int)st->layers.size();
    const rnn_plan* p0 = st->layers[0];
    auto no = [&](const char* r) { *why = r; return false; };
    if (st->wave_mode == 0) return no("disabled");
    if (L < 2 || L > kWaveMaxLayers) return no("layer count");
    if (S <= 0 || N <= 0) return no("zero size");
    if (p0->io != RNN_IO_F32) return no("fp16/bf16 I/O rounds each layer's output");
    if (p0->mode != RNN_MODE_EXACT && p0->mode != RNN_MODE_FAST) return no("tensor-core modes");
    for (const rnn_plan* pl : st->layers) {
        if (pl->D != 1) return no("bidirectional layer");
        if (pl->direction != p0->direction || pl->op != p0->op || pl->H != p0->H || pl->mode != p0->mode)
            return no("layers differ in direction, operator, hidden size or mode");
    }
    if (st->wave_mode == 1) {
        for (int l = 1; l < L; ++l) {
            const rnn_plan* pl = st->layers[l];
            if ((double)N * pl->G * pl->H * (double)(pl->H + pl->I) > kWaveMaxProducts)
                return no("layers large enough to run faster one after another");
        }
    }
    return true;
}

rnn_status plan_wave(const rnn_stack* st, int64_t N, const DeviceInfo& di, WaveGeometry* g)
{
    const int L = (int)st->layers.size();
    const rnn_plan* p0 = st->layers[0];
    const int64_t H = p0->H;
    const int G = p0->G;
    const bool exact = p0->mode == RNN_MODE_EXACT;
    g->npad = (int)round_up(N, 8);
    double total = 0.0;
    for (int l = 0; l < L; ++l) total += (double)H + (l > 0 ? (double)st->layers[l]->I : 0.0);
    // at most this many CTAs per layer (the first plan's unit_groups
    // override, else the SMs' share); enough that the layer's resident
    // slices of R and W fit in shared memory
    const int64_t cap = p0->ov_units > 0 ? p0->ov_units : (int64_t)di.sms;
    const size_t ring = (size_t)kRecStages * kRecKC * g->npad * 4;
    int ctas = 0, umax_all = 0;
    for (int l = 0; l < L; ++l) {
        const double w = (double)H + (l > 0 ? (double)st->layers[l]->I : 0.0);
        const size_t krows = (size_t)H + (l > 0 ? (size_t)st->layers[l]->I : 0);
        int64_t C = std::max<int64_t>(1, (int64_t)std::floor(di.sms * w / total));
        C = std::min<int64_t>(std::min<int64_t>(C, cap), H);
        int64_t um = ceil_div(H, C);
        while (um > 1 && krows * rec_ugp((int)um, G) * 4 + ring > (size_t)di.smem_optin) --um;
        C = ceil_div(H, um);
        g->C[l] = (int)C;
        g->umax[l] = (int)um;
        g->ugp[l] = rec_ugp((int)um, G);
        g->cta0[l] = ctas;
        ctas += (int)C;
        umax_all = std::max(umax_all, (int)um);
    }
    g->ctas = ctas;
    g->tn = 0;
    const int tns[3] = {1, 2, 4};
    for (int t : tns)
        if ((int64_t)umax_all * ceil_div(N, t) <= kMaxThreads) { g->tn = t; break; }
    if (!g->tn) return fail(RNN_ERR_UNSUPPORTED, "wavefront: batch %lld needs more threads per CTA", (long long)N);
    g->threads = (int)round_up((int64_t)umax_all * ceil_div(N, g->tn), 32);
    size_t smem = 0;
    for (int l = 0; l < L; ++l) {
        const size_t k = (size_t)H + (l > 0 ? (size_t)st->layers[l]->I : 0);
        smem = std::max(smem, k * g->ugp[l] * 4);
    }
    smem += (size_t)kRecStages * kRecKC * g->npad * 4;
    if (smem > (size_t)di.smem_optin) return fail(RNN_ERR_UNSUPPORTED, "wavefront: weight slices do not fit");
    g->smem = smem;
    int blocks = 0;
    cudaError_t e = wavefront_occupancy(p0->op, g->tn, exact, g->threads, smem, &blocks);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (blocks < 1 || ctas > blocks * di.sms) return fail(RNN_ERR_UNSUPPORTED, "wavefront: the grid does not fit");
    return RNN_OK;
}

// One stack run as a single wavefront launch (after the layer-0 projection).
// Returns RNN_ERR_UNSUPPORTED, having queued nothing, when the geometry does
// not fit (the caller then runs the layers one by one).
rnn_status stack_run_wave(rnn_stack* st, int64_t S, int64_t N, const float* X, const float* const* W,
                          const float* const* R, const float* const* B, const int32_t* lens,
                          const float* const* h0, const float* const* c0, const float* const* P, float* Y,
                          float* const* Yh, float* const* Yc, cudaStream_t stream, int* launches_out)
{
    const int L = (int)st->layers.size();
    rnn_plan* p0 = st->layers[0];
    const int64_t H = p0->H, G = p0->G, GH = G * H, I0 = p0->I;
    const bool exact = p0->mode == RNN_MODE_EXACT;
    // the checks rnn_run makes for each layer (pointers, sizes, the scratch limit)
    if (S > (1 << 30) || N > (1 << 24)) return fail(RNN_ERR_UNSUPPORTED, "seq_length or batch_size too large");
    if (!X && I0 > 0) return fail(RNN_ERR_INVALID_ARGUMENT, "X is NULL");
    for (int l = 0; l < L; ++l) {
        const rnn_plan* pl = st->layers[l];
        if (!pl->const_weights && (!R[l] || (!W[l] && pl->I > 0)))
            return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are required (layer %d)", l);
        const double per_dir = (double)S * N * GH + 4.0 * N * H + (pl->const_weights ? 0.0 : (double)GH * (pl->I + H));
        if (per_dir >= 1073741824.0)
            return fail(RNN_ERR_UNSUPPORTED, "per-direction scratch of %.0f floats reaches the 2^30 limit", per_dir);
    }
    DeviceInfo di;
    rnn_status rs = device_info(&di);
    if (rs != RNN_OK) return rs;
    if (!di.coop) return fail(RNN_ERR_UNSUPPORTED, "device lacks cooperative launch");
    WaveGeometry wg;
    rs = plan_wave(st, N, di, &wg);
    if (rs != RNN_OK) return rs;
    int64_t max_len = S;
    if (lens) {
        rs = read_lengths(p0, lens, N, S, stream, &max_len);
        if (rs != RNN_OK) return rs;
    }

    // scratch: XW of layer 0, packed weights, ring buffers, row ranking
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t o = off; off += align256(bytes); return o; };
    const size_t o_xw = take(sizeof(float) * (size_t)S * N * GH);
    const size_t o_wt0 = take(p0->const_weights ? 0 : sizeof(float) * (size_t)I0 * GH);
    size_t o_rt[kWaveMaxLayers], o_wt[kWaveMaxLayers], o_hb[kWaveMaxLayers], o_rh[kWaveMaxLayers];
    for (int l = 0; l < L; ++l) {
        const rnn_plan* pl = st->layers[l];
        const bool two = pl->op == RNN_OP_GRU && pl->lbr == 0;
        o_rt[l] = take(pl->const_weights ? 0 : sizeof(float) * (size_t)H * GH);
        o_wt[l] = take((l == 0 || pl->const_weights) ? 0 : sizeof(float) * (size_t)pl->I * GH);
        o_hb[l] = take(sizeof(float) * (size_t)kWaveRing * H * wg.npad);
        o_rh[l] = take(two ? sizeof(float) * (size_t)H * wg.npad : 0);
    }
    const size_t o_perm = take(sizeof(int32_t) * (size_t)N);
    if (off > st->wcap) {
        if (st->wbuf) cudaFree(st->wbuf);   // synchronises with outstanding work
        st->wbuf = nullptr;
        st->wcap = 0;
        cudaError_t e = cudaMalloc(&st->wbuf, off);
        if (e != cudaSuccess) {
            st->wbuf = nullptr;
            return cuda_fail(e, "cudaMalloc(wavefront scratch)");
        }
        st->wcap = off;
    }
    rs = ensure_scratch(p0, 0);        // the first layer's control block: counters and status
    if (rs != RNN_OK) return rs;
    char* sb = (char*)st->wbuf;
    if (p0->device < 0) cudaGetDevice(&p0->device);
    if (p0->timing && !p0->events_ready) {
        rs = rnn_plan_set_timing(p0, 1);
        if (rs != RNN_OK) return rs;
    }
    if (!p0->done_ready) {
        cudaError_t e = cudaEventCreateWithFlags(&p0->done, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
        p0->done_ready = true;
    }
    if (p0->timing) {
        p0->slot = (p0->slot + 1) % rnn_plan::kRing;
        cudaError_t eh = harvest(p0, p0->slot);
        if (eh != cudaSuccess) return cuda_fail(eh, "reading timing events");
        for (bool& u : p0->ev_used[p0->slot]) u = false;
    }
    const bool timed = p0->timing;
    int launches = 0;
    cudaError_t e;
    int* status = (int*)(p0->ctrl + kCtrlStatusOffset);

    // pack every layer's weights k-major (layer 0's W for the projection)
    if (timed) record(p0, 0, stream);
    WaveParams wp;
    std::memset(&wp, 0, sizeof wp);
    float* wt0 = p0->const_weights ? p0->wt_const : (float*)(sb + o_wt0);
    for (int l = 0; l < L; ++l) {
        rnn_plan* pl = st->layers[l];
        WaveLayer& ly = wp.layer[l];
        float* rt = pl->const_weights ? pl->rt_const : (float*)(sb + o_rt[l]);
        float* wt = l == 0 ? wt0 : (pl->const_weights ? pl->wt_const : (float*)(sb + o_wt[l]));
        if (!pl->const_weights) {
            e = launch_pack(pl->I > 0 ? W[l] : nullptr, R[l], wt, rt, 1, (int)G, H, pl->I, stream);
            if (e != cudaSuccess) return cuda_fail(e, "pack launch");
            launches += (pl->I > 0 ? 1 : 0) + 1;
        }
        ly.cta0 = wg.cta0[l]; ly.C = wg.C[l]; ly.umax = wg.umax[l]; ly.ugp = wg.ugp[l];
        ly.I = l == 0 ? 0 : (int)pl->I;
        ly.lbr = pl->lbr; ly.input_forget = pl->input_forget;
        ly.has_B = B && B[l]; ly.has_P = P && P[l] && pl->op == RNN_OP_LSTM;
        ly.has_h0 = h0 && h0[l]; ly.has_c0 = c0 && c0[l] && pl->op == RNN_OP_LSTM;
        ly.has_clip = pl->has_clip; ly.clip = pl->clip;
        for (int k = 0; k < 3; ++k) ly.act[k] = pl->act[0][k];
        ly.XW = l == 0 ? (const float*)(sb + o_xw) : nullptr;
        ly.Wt = l == 0 ? nullptr : wt;
        ly.Rt = rt;
        ly.B = ly.has_B ? B[l] : nullptr;
        ly.P = ly.has_P ? P[l] : nullptr;
        ly.h0 = ly.has_h0 ? h0[l] : nullptr;
        ly.c0 = ly.has_c0 ? c0[l] : nullptr;
        ly.Y = l + 1 == L ? Y : nullptr;
        ly.Yh = Yh ? Yh[l] : nullptr;
        ly.Yc = (Yc && pl->op == RNN_OP_LSTM) ? Yc[l] : nullptr;
        ly.hbuf = (float*)(sb + o_hb[l]);
        ly.rhbuf = (pl->op == RNN_OP_GRU && pl->lbr == 0) ? (float*)(sb + o_rh[l]) : nullptr;
    }
    if (timed) record(p0, 1, stream);
    e = launch_projection(X, wt0, (float*)(sb + o_xw), S * N, I0, GH, exact, status, p0->spin_limit_ns, stream);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    launches += 1;
    if (timed) record(p0, 2, stream);

    wp.L = L; wp.N = (int)N; wp.H = (int)H; wp.S = (int)S; wp.layout = p0->layout;
    wp.reverse = p0->direction == RNN_DIR_REVERSE ? 1 : 0;
    wp.npad = wg.npad; wp.max_len = (int)max_len;
    wp.has_lens = lens != nullptr; wp.lens = lens;
    wp.bar = (unsigned*)p0->ctrl;
    wp.status = status;
    wp.spin_limit_ns = p0->spin_limit_ns;
    wp.debug_skip_cta = p0->skip_cta;
    if (lens) {
        wp.perm = (const int32_t*)(sb + o_perm);
        e = launch_rank_rows(lens, (int32_t*)(sb + o_perm), (int)N, stream);
        if (e != cudaSuccess) return cuda_fail(e, "row ranking launch");
        launches += 1;
    }
    e = launch_wave_state_init(wp, stream);
    if (e != cudaSuccess) return cuda_fail(e, "state set-up launch");
    launches += 1;
    if (timed) record(p0, 3, stream);
    e = launch_ordered(stream, [&]() {
        return launch_wavefront(p0->op, wp, exact, wg.tn, wg.ctas, wg.threads, wg.smem, stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "wavefront launch");
    launches += 1;
    if (timed) record(p0, 4, stream);
    if (Y && max_len < S) {
        e = launch_mask_tail(Y, p0->layout, S, 1, N, H, max_len, 0, stream);
        if (e != cudaSuccess) return cuda_fail(e, "mask launch");
        launches += 1;
    }
    if (timed) {
        record(p0, 5, stream);
        p0->slot_pending[p0->slot] = true;
    }
    cudaEventRecord(p0->done, stream);
    p0->ran = true;
    p0->last_static = false;
    p0->last_launches = launches;
    p0->g_units = wg.C[0]; p0->g_tn = wg.tn; p0->g_rres = 1; p0->g_rows = 1;
    p0->g_kernel = 4; p0->g_threads = wg.threads; p0->g_smem = (int)wg.smem;
    *launches_out = launches;
    return RNN_OK;
}

}  // namespace

rnn_status rnn_stack_set_wavefront(rnn_stack_t st, int enable)
{
    g_error.clear();
    if (!st) return fail(RNN_ERR_INVALID_ARGUMENT, "stack is NULL");
    if (enable < 0 || enable > 2) return fail(RNN_ERR_INVALID_ARGUMENT, "the wavefront mode must be 0, 1 or 2");
    st->wave_mode = enable;
    return RNN_OK;
}

int rnn_stack_last_wavefront(rnn_stack_t st) { return st && st->last_wave ? 1 : 0; }

rnn_status rnn_stack_run(rnn_stack_t st, int64_t S, int64_t N, const float* X, const float* const* W,
                         const float* const* R, const float* const* B, const int32_t* lens,
                         const float* const* h0, const float* const* c0, const float* const* P, float* Y,
                         float* const* Yh, float* const* Yc, void* stream)
{
    g_error.clear();
    if (!st) return fail(RNN_ERR_INVALID_ARGUMENT, "stack is NULL");
    rnn_status rs = stack_check(st);
    if (rs != RNN_OK) return rs;
    const int L = (int)st->layers.size();
    if (!W || !R) return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are per-layer arrays");
    st->last_wave = false;
    std::string why;
    if (wave_eligible(st, S, N, &why)) {
        const std::string saved = g_error;
        int launches = 0;
        rs = stack_run_wave(st, S, N, X, W, R, B, lens, h0, c0, P, Y, Yh, Yc, (cudaStream_t)stream, &launches);
        if (rs == RNN_OK) {
            st->last_wave = true;
            st->last_launches = launches;
            return RNN_OK;
        }
        if (rs != RNN_ERR_UNSUPPORTED) return rs;
        g_error = saved;   // no launch fits: run the layers one by one
    }
    const size_t elem = st->layers[0]->io == 0 ? 4 : 2;
    size_t need = 0;
    for (int l = 0; l + 1 < L; ++l)
        need = std::max(need, elem * (size_t)S * N * st->layers[l]->D * st->layers[l]->H);
    for (int b = 0; b < 2; ++b) {
        if (need > st->cap[b]) {
            if (st->buf[b]) cudaFree(st->buf[b]);   // synchronises with outstanding work
            st->buf[b] = nullptr;
            st->cap[b] = 0;
            cudaError_t e = cudaMalloc(&st->buf[b], need);
            if (e != cudaSuccess) {
                st->buf[b] = nullptr;
                return cuda_fail(e, "cudaMalloc(stack buffer)");
            }
            st->cap[b] = need;
        }
    }
    const float* x = X;
    int cur = -1;                 // which stack buffer holds x (-1: the caller's X)
    int64_t max_len = -1;         // sequence_lens is checked by the first layer only
    st->last_launches = 0;
    for (int l = 0; l < L; ++l) {
        rnn_plan* pl = st->layers[l];
        const bool last = l + 1 == L;
        const int yb = cur == 0 ? 1 : 0;
        float* y = last ? Y : (float*)st->buf[yb];
        int64_t ml = 0;
        rs = run_plan(pl, S, N, x, W[l], R[l], B ? B[l] : nullptr, lens, h0 ? h0[l] : nullptr,
                      c0 ? c0[l] : nullptr, P ? P[l] : nullptr, y, Yh ? Yh[l] : nullptr, Yc ? Yc[l] : nullptr,
                      stream, max_len, &ml);
        if (rs != RNN_OK) return rs;
        if (max_len < 0) max_len = ml;
        st->last_launches += pl->last_launches;
        if (last) break;
        if (pl->layout == 0 && pl->D == 2 && S > 0 && N > 0) {
            // [S][2][N][H] -> [S][N][2H]: forward units, then reverse, per (t, n)
            const int pb = 1 - yb;
            cudaError_t e = launch_stack_permute(st->buf[yb], st->buf[pb], S, N, pl->H, (int)elem,
                                                 (cudaStream_t)stream);
            if (e != cudaSuccess) return cuda_fail(e, "stack permute launch");
            st->last_launches += 1;
            x = (const float*)st->buf[pb];
            cur = pb;
        } else {
            x = y;                // [S][1][N][H] is [S][N][H]; layout 1 [N][S][D][H] is [N][S][D*H]
            cur = yb;
        }
    }
    return RNN_OK;
}

void rnn_stack_destroy(rnn_stack_t st)
{
    if (!st) return;
    bool ran = false;
    for (rnn_plan* pl : st->layers) ran = ran || (pl && pl->ran);
    if (ran) cudaDeviceSynchronize();
    for (void* b : st->buf)
        if (b) cudaFree(b);
    if (st->wbuf) cudaFree(st->wbuf);
    delete st;
}

int rnn_stack_last_launch_count(rnn_stack_t st) { return st ? st->last_launches : 0; }

rnn_status rnn_plan_set_io_type(rnn_plan_t pl, int io)
{
    g_error.clear();
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (io < RNN_IO_F32 || io > RNN_IO_BF16) return fail(RNN_ERR_INVALID_ARGUMENT, "unknown io type %d", io);
    if (pl->cell && io != RNN_IO_F32) return fail(RNN_ERR_UNSUPPORTED, "a cell plan takes fp32 tensors only");
    pl->io = io;
    return RNN_OK;
}

rnn_status rnn_cell_plan_create(rnn_plan_t* out, int64_t hidden_size, int64_t input_size, const char* activation,
                                float clip)
{
    g_error.clear();
    if (!out) return fail(RNN_ERR_INVALID_ARGUMENT, "out is NULL");
    *out = nullptr;
    const char* name = activation ? activation : "Tanh";
    const int id = act_id(name);
    if (id != act_id("Relu") && id != act_id("Sigmoid") && id != act_id("Tanh"))
        return fail(RNN_ERR_INVALID_ARGUMENT, "a cell takes Relu, Sigmoid or Tanh, not '%s'", name);
    if (!(clip > 0.0f)) return fail(RNN_ERR_INVALID_ARGUMENT, "clip must be positive (+infinity: no clip)");
    const char* acts[1] = {name};
    const float no_clip = std::nanf("");
    rnn_status rs = rnn_plan_create(out, RNN_OP_RNN, RNN_DIR_FORWARD, hidden_size, input_size, acts, 1, nullptr, 0,
                                    nullptr, 0, std::isinf(clip) ? no_clip : clip, 0, 0, 0);
    if (rs != RNN_OK) return rs;
    (*out)->cell = true;
    return RNN_OK;
}

rnn_status rnn_cell_run(rnn_plan_t pl, int64_t batch_size, const float* X, const float* H, const float* W,
                        const float* R, const float* B, float* Ho, void* stream)
{
    g_error.clear();
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (!pl->cell) return fail(RNN_ERR_INVALID_ARGUMENT, "not a cell plan (rnn_cell_plan_create)");
    if (batch_size < 0) return fail(RNN_ERR_INVALID_ARGUMENT, "batch_size must be >= 0");
    pl->last_launches = 0;
    if (batch_size == 0) return RNN_OK;     // nothing to read or write (the arrays may be empty, NULL)
    if (!H || !B || !Ho) return fail(RNN_ERR_INVALID_ARGUMENT, "H, B and Ho are required");
    if (pl->I > 0 && !X) return fail(RNN_ERR_INVALID_ARGUMENT, "X is required when input_size > 0");
    const float* Wc = pl->const_weights ? pl->wk_const : W;     // K-major pack of a 1-gate W is W itself
    const float* Rc = pl->const_weights ? pl->r_orig_const : R;
    if (!Rc || (pl->I > 0 && !Wc)) return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are required");
    cudaStream_t st = (cudaStream_t)stream;
    if (pl->timing && !pl->events_ready) {
        rnn_status rs = rnn_plan_set_timing(pl, 1);
        if (rs != RNN_OK) return rs;
    }
    if (!pl->done_ready) {
        cudaError_t e = cudaEventCreateWithFlags(&pl->done, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
        pl->done_ready = true;
    }
    if (pl->timing) {
        pl->slot = (pl->slot + 1) % rnn_plan::kRing;
        cudaError_t eh = harvest(pl, pl->slot);
        if (eh != cudaSuccess) return cuda_fail(eh, "reading timing events");
        for (bool& u : pl->ev_used[pl->slot]) u = false;
        record(pl, 3, st);      // the cell kernel is timed as the recurrence (the one event pair)
    }
    cudaError_t e = launch_cell(X, H, Wc, Rc, B, Ho, batch_size, pl->I, pl->H, pl->act[0][0].fn, pl->has_clip,
                                pl->clip, pl->mode == RNN_MODE_EXACT, st);
    if (e != cudaSuccess) return cuda_fail(e, "cell launch");
    if (pl->timing) {
        record(pl, 4, st);
        pl->slot_pending[pl->slot] = true;
    }
    cudaEventRecord(pl->done, st);
    pl->ran = true;
    pl->last_launches = 1;
    return RNN_OK;
}

// rnn_run without any device allocation: all scratch (control words, packed
// weights, projection, h exchange buffers) is carved out of the library's
// fixed device array, and sequence_lens is checked through a stack buffer.
rnn_status rnn_run_static_scratch(rnn_plan_t pl, int64_t S, int64_t N, const float* X, const float* W,
                                  const float* R, const float* B, const int32_t* lens, const float* h0,
                                  const float* c0, const float* P, float* Y, float* Yh, float* Yc,
                                  void* stream)
{
    constexpr int64_t kMaxBatch = 4096;
    g_error.clear();
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    pl->last_launches = 0;
    RunArgs a{S, N, X, W, R, B, lens, h0, c0, P, Y, Yh, Yc, (cudaStream_t)stream};
    bool done = false;
    rnn_status rs = check_run(pl, a, &done);
    if (rs != RNN_OK || done) return rs;      // zero-size runs need no scratch: any batch size
    if (N > kMaxBatch)
        return fail(RNN_ERR_UNSUPPORTED, "static-scratch runs take at most %lld batch rows", (long long)kMaxBatch);

    DeviceInfo di;
    rs = device_info(&di);
    if (rs != RNN_OK) return rs;
    if (!di.coop) return fail(RNN_ERR_UNSUPPORTED, "device lacks cooperative launch");

    int64_t max_len = S;
    if (lens) {
        int32_t host_lens[kMaxBatch];
        cudaError_t e = cudaMemcpyAsync(host_lens, lens, sizeof(int32_t) * (size_t)N, cudaMemcpyDeviceToHost, a.st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(a.st);
        if (e != cudaSuccess) return cuda_fail(e, "copying sequence_lens");
        rs = check_lengths(host_lens, N, S, &max_len);
        if (rs != RNN_OK) return rs;
    }

    Geometry geo{};
    rs = plan_geometry(pl, N, di, R, &geo);
    if (rs != RNN_OK) return rs;

    void* base = nullptr;
    size_t cap = 0;
    cudaError_t e = static_scratch(&base, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "looking up the static scratch");
    const Layout L = scratch_layout(pl, geo, S, N, kCtrlBytes);   // control words first
    if (L.total > cap)
        return fail(RNN_ERR_UNSUPPORTED, "run needs %zu bytes of scratch; the static scratch holds %zu", L.total, cap);
    char* sb = (char*)base;
    e = cudaMemsetAsync(sb + kCtrlStatusOffset, 0, sizeof(int), a.st);   // status starts at 0 on every call
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    int launches = 0;
    rs = enqueue(pl, a, geo, max_len, sb, L, sb, false, pl->spin_limit_ns, pl->skip_cta, &launches);
    if (rs != RNN_OK) return rs;
    pl->last_launches = launches;
    pl->last_static = true;          // rnn_plan_sync reads the fixed array's status word
    pl->static_status = (int*)(sb + kCtrlStatusOffset);
    pl->ran = true;
    return RNN_OK;
}

}  // extern "C"

namespace rnngb {

bool encode_tensor_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                       const cuuint64_t* strides, const cuuint32_t* box, bool swizzle128, int dtype)
{
    return tmap_encode_raw(map, base, rank, dims, strides, box, swizzle128, dtype) == CUDA_SUCCESS;
}

}  // namespace rnngb
