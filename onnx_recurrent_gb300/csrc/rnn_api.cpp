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
#include <new>
#include <string>

#include "rnn_internal.h"

namespace rnngb {
cudaError_t launch_recurrent_rnn(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t launch_recurrent_gru(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t launch_recurrent_lstm(const RecParams&, bool, int, size_t, cudaStream_t);
cudaError_t recurrent_occupancy_rnn(int, bool, int, size_t, int*);
cudaError_t recurrent_occupancy_gru(int, bool, int, size_t, int*);
cudaError_t recurrent_occupancy_lstm(int, bool, int, size_t, int*);

cudaError_t launch_recurrent(const RecParams& p, bool exact, int threads, size_t smem, cudaStream_t s)
{
    switch (p.op) {
    case 0: return launch_recurrent_rnn(p, exact, threads, smem, s);
    case 1: return launch_recurrent_gru(p, exact, threads, smem, s);
    default: return launch_recurrent_lstm(p, exact, threads, smem, s);
    }
}

cudaError_t recurrent_occupancy(int op, int tn, bool exact, int threads, size_t smem, int* blocks)
{
    switch (op) {
    case 0: return recurrent_occupancy_rnn(tn, exact, threads, smem, blocks);
    case 1: return recurrent_occupancy_gru(tn, exact, threads, smem, blocks);
    default: return recurrent_occupancy_lstm(tn, exact, threads, smem, blocks);
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

constexpr int kMaxThreads = 512;
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
    float* rt_const = nullptr;   // [D][H][G*H]

    // scratch
    char* scratch = nullptr;
    size_t scratch_bytes = 0;
    char* ctrl = nullptr;        // bar[2] + status
    int32_t* lens_host = nullptr;
    int64_t lens_cap = 0;
    int device = -1;

    // launch overrides and record
    int ov_ctas = 0, ov_tn = 0, ov_rres = -1;
    int g_ctas = 0, g_tn = 0, g_rres = 0, g_threads = 0, g_smem = 0;
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
    int ctas, umax, tn, threads, rres;
    size_t smem;
    int npad;
};

// Launch geometry of the recurrent kernel for batch N.
rnn_status plan_geometry(rnn_plan* pl, int64_t N, const DeviceInfo& di, Geometry* g)
{
    const int64_t H = pl->H;
    const int G = pl->G, D = pl->D;
    g->npad = (int)round_up(N, 8);
    int C;
    if (pl->ov_ctas > 0) {
        C = (int)std::min<int64_t>(pl->ov_ctas, H);
    } else {
        const long long macs = (long long)N * G * H * H;
        const int64_t single_threads = H * ((N + 7) / 8);
        if (macs <= 262144 && single_threads <= kMaxThreads)
            C = 1;   // tiny step: one CTA per direction, no device-wide barrier
        else
            C = (int)std::max<int64_t>(1, std::min<int64_t>(di.sms / D, H));
        const int64_t umax0 = (H + C - 1) / C;
        C = (int)((H + umax0 - 1) / umax0);
    }
    g->ctas = C;
    g->umax = (int)((H + C - 1) / C);
    const int tns[4] = {1, 2, 4, 8};
    g->tn = 0;
    if (pl->ov_tn > 0) {
        if (pl->ov_tn != 1 && pl->ov_tn != 2 && pl->ov_tn != 4 && pl->ov_tn != 8)
            return fail(RNN_ERR_INVALID_ARGUMENT, "rows_per_thread must be 1, 2, 4 or 8");
        g->tn = pl->ov_tn;
    } else {
        for (int tn : tns)
            if ((int64_t)g->umax * ((N + tn - 1) / tn) <= kMaxThreads) { g->tn = tn; break; }
    }
    if (g->tn == 0)
        return fail(RNN_ERR_UNSUPPORTED,
                    "no recurrent launch for batch %lld with %d hidden units per CTA (threads > %d)",
                    (long long)N, g->umax, kMaxThreads);
    const int64_t thr = (int64_t)g->umax * ((N + g->tn - 1) / g->tn);
    if (thr > kMaxThreads)
        return fail(RNN_ERR_UNSUPPORTED, "recurrent launch needs %lld threads per CTA (max %d)",
                    (long long)thr, kMaxThreads);
    g->threads = (int)round_up(thr, 32);
    const size_t sres = rec_smem_bytes((int)H, g->umax, G, g->npad, 1);
    const size_t sstr = rec_smem_bytes((int)H, g->umax, G, g->npad, 0);
    if (pl->ov_rres == 1) g->rres = 1;
    else if (pl->ov_rres == 0) g->rres = 0;
    else g->rres = sres <= (size_t)di.smem_optin ? 1 : 0;
    g->smem = g->rres ? sres : sstr;
    if (g->smem > (size_t)di.smem_optin)
        return fail(RNN_ERR_UNSUPPORTED, "recurrent kernel needs %zu bytes of shared memory (max %d)",
                    g->smem, di.smem_optin);
    int blocks = 0;
    cudaError_t e = recurrent_occupancy(pl->op, g->tn, pl->mode == RNN_MODE_EXACT, g->threads, g->smem, &blocks);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (blocks < 1 || (int64_t)D * C > (int64_t)blocks * di.sms)
        return fail(RNN_ERR_UNSUPPORTED,
                    "recurrent grid of %d CTAs cannot be co-resident (%d per SM, %d SMs)", D * C, blocks,
                    di.sms);
    return RNN_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

rnn_status ensure_scratch(rnn_plan* pl, size_t bytes)
{
    if (!pl->ctrl) {
        cudaError_t e = cudaMalloc((void**)&pl->ctrl, 256);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(control)");
        e = cudaMemset(pl->ctrl, 0, 256);
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
    if (pl->rt_const) cudaFree(pl->rt_const);
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
    if (mode != RNN_MODE_EXACT && mode != RNN_MODE_FAST)
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

rnn_status rnn_plan_set_launch(rnn_plan_t pl, int ctas_per_dir, int rows_per_thread, int r_resident)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (ctas_per_dir < 0 || rows_per_thread < 0 || r_resident < -1 || r_resident > 1)
        return fail(RNN_ERR_INVALID_ARGUMENT, "bad launch override");
    if (rows_per_thread != 0 && rows_per_thread != 1 && rows_per_thread != 2 && rows_per_thread != 4 &&
        rows_per_thread != 8)
        return fail(RNN_ERR_INVALID_ARGUMENT, "rows_per_thread must be 0, 1, 2, 4 or 8");
    pl->ov_ctas = ctas_per_dir;
    pl->ov_tn = rows_per_thread;
    pl->ov_rres = r_resident;
    return RNN_OK;
}

rnn_status rnn_plan_get_launch(rnn_plan_t pl, int* ctas, int* tn, int* rres, int* threads, int* smem)
{
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    if (ctas) *ctas = pl->g_ctas;
    if (tn) *tn = pl->g_tn;
    if (rres) *rres = pl->g_rres;
    if (threads) *threads = pl->g_threads;
    if (smem) *smem = pl->g_smem;
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
    cudaError_t e = pl->done_ready ? cudaEventSynchronize(pl->done) : cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "waiting for the run");
    int st = 0;
    e = cudaMemcpy(&st, pl->ctrl + 64, sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device status");
    if (st != 0) {
        const int zero = 0;
        cudaMemcpy(pl->ctrl + 64, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (st == RNN_ERR_TIMEOUT)
            return fail(RNN_ERR_TIMEOUT, "the device-wide step barrier timed out; outputs are incomplete");
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
        }
    }
    cudaError_t e = launch_pack(W, R, pl->wt_const, pl->rt_const, pl->D, pl->G, pl->H, pl->I, s);
    if (e != cudaSuccess) return cuda_fail(e, "pack launch");
    pl->const_weights = true;
    return RNN_OK;
}

rnn_status rnn_run(rnn_plan_t pl, int64_t S, int64_t N, const float* X, const float* W, const float* R,
                   const float* B, const int32_t* lens, const float* h0, const float* c0, const float* P,
                   float* Y, float* Yh, float* Yc, void* stream)
{
    g_error.clear();
    if (!pl) return fail(RNN_ERR_INVALID_ARGUMENT, "plan is NULL");
    pl->last_launches = 0;
    cudaStream_t st = (cudaStream_t)stream;
    if (S < 0 || N < 0) return fail(RNN_ERR_INVALID_ARGUMENT, "seq_length and batch_size must be >= 0");
    if (S > (1 << 30) || N > (1 << 24)) return fail(RNN_ERR_UNSUPPORTED, "seq_length or batch_size too large");
    const int64_t H = pl->H, I = pl->I, G = pl->G, D = pl->D, GH = G * H;
    if (pl->op != RNN_OP_LSTM) { c0 = nullptr; P = nullptr; Yc = nullptr; }

    // Limits: per-direction scratch below 2^30 floats.
    const double per_dir = (double)S * N * GH + 4.0 * N * H + (pl->const_weights ? 0.0 : (double)GH * (I + H));
    if (per_dir >= 1073741824.0)
        return fail(RNN_ERR_UNSUPPORTED, "per-direction scratch of %.0f floats reaches the 2^30 limit", per_dir);

    // Zero-size: nothing runs; final states are the initial states or zeros.
    if (S == 0 || N == 0) {
        const size_t sb = sizeof(float) * (size_t)D * N * H;
        cudaError_t e = cudaSuccess;
        if (Yh && sb) e = h0 ? cudaMemcpyAsync(Yh, h0, sb, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(Yh, 0, sb, st);
        if (e == cudaSuccess && Yc && sb)
            e = c0 ? cudaMemcpyAsync(Yc, c0, sb, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(Yc, 0, sb, st);
        if (e != cudaSuccess) return cuda_fail(e, "zero-size copy");
        return RNN_OK;
    }
    if (!X && I > 0) return fail(RNN_ERR_INVALID_ARGUMENT, "X is NULL");
    if (!pl->const_weights && (!R || (!W && I > 0))) return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are required");

    DeviceInfo di;
    rnn_status rs = device_info(&di);
    if (rs != RNN_OK) return rs;
    if (!di.coop) return fail(RNN_ERR_UNSUPPORTED, "device lacks cooperative launch");

    // sequence_lens: check on the host before anything is written.
    int64_t max_len = S;
    if (lens) {
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
        max_len = 0;
        for (int64_t n = 0; n < N; ++n) {
            const int32_t L = pl->lens_host[n];
            if (L < 0 || (int64_t)L > S)
                return fail(RNN_ERR_INVALID_INPUT, "sequence_lens[%lld] = %d is outside [0, %lld]", (long long)n, L,
                            (long long)S);
            max_len = std::max<int64_t>(max_len, L);
        }
    }

    Geometry geo{};
    rs = plan_geometry(pl, N, di, &geo);
    if (rs != RNN_OK) return rs;

    // scratch layout
    const int64_t M = S * N;
    size_t off = 0;
    const size_t o_wt = off; off += pl->const_weights ? 0 : align256(sizeof(float) * (size_t)I * D * GH);
    const size_t o_rt = off; off += pl->const_weights ? 0 : align256(sizeof(float) * (size_t)D * H * GH);
    const size_t o_xw = off; off += align256(sizeof(float) * (size_t)M * D * GH);
    const size_t o_hb = off; off += align256(sizeof(float) * (size_t)D * 2 * H * geo.npad);
    const bool need_rh = pl->op == RNN_OP_GRU && pl->lbr == 0;
    const size_t o_rh = off; off += need_rh ? align256(sizeof(float) * (size_t)D * H * geo.npad) : 0;
    rs = ensure_scratch(pl, std::max<size_t>(off, 256));
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

    float* wt = pl->const_weights ? pl->wt_const : (float*)(pl->scratch + o_wt);
    float* rt = pl->const_weights ? pl->rt_const : (float*)(pl->scratch + o_rt);
    float* xw = (float*)(pl->scratch + o_xw);
    const bool exact = pl->mode == RNN_MODE_EXACT;
    int launches = 0;
    cudaError_t e;

    record(pl, 0, st);
    if (!pl->const_weights) {
        e = launch_pack(W, R, wt, rt, (int)D, (int)G, H, I, st);
        if (e != cudaSuccess) return cuda_fail(e, "pack launch");
        launches += (int)D * (I > 0 ? 2 : 1);
    }
    record(pl, 1, st);
    e = launch_projection(X, wt, xw, M, I, D * GH, exact, st);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    launches += 1;
    record(pl, 2, st);

    RecParams p;
    std::memset(&p, 0, sizeof p);
    p.op = pl->op; p.G = (int)G; p.D = (int)D; p.N = (int)N; p.H = (int)H; p.S = (int)S;
    p.layout = pl->layout; p.lbr = pl->lbr; p.input_forget = pl->input_forget;
    p.has_B = B != nullptr; p.has_P = P != nullptr; p.has_h0 = h0 != nullptr; p.has_c0 = c0 != nullptr;
    p.has_lens = lens != nullptr; p.has_clip = pl->has_clip; p.clip = pl->clip;
    for (int d = 0; d < 2; ++d)
        for (int s = 0; s < 3; ++s) p.act[d][s] = pl->act[d][s];
    p.max_len = (int)max_len;
    p.dir_reverse[0] = pl->direction == RNN_DIR_REVERSE ? 1 : 0;
    p.dir_reverse[1] = 1;
    p.ctas_per_dir = geo.ctas; p.umax = geo.umax; p.rows_per_thread = geo.tn; p.r_resident = geo.rres;
    p.npad = geo.npad;
    p.XW = xw; p.Rt = rt; p.B = B; p.P = P; p.h0 = h0; p.c0 = c0; p.lens = lens;
    p.Y = Y; p.Yh = Yh; p.Yc = Yc;
    p.hbuf = (float*)(pl->scratch + o_hb);
    p.rhbuf = need_rh ? (float*)(pl->scratch + o_rh) : nullptr;
    p.bar = (unsigned*)pl->ctrl;
    p.status = (int*)(pl->ctrl + 64);
    p.spin_limit_ns = pl->spin_limit_ns;
    p.debug_skip_cta = pl->skip_cta;

    e = launch_state_init(p, st);
    if (e != cudaSuccess) return cuda_fail(e, "state set-up launch");
    launches += 1;
    record(pl, 3, st);
    e = launch_recurrent(p, exact, geo.threads, geo.smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent launch");
    launches += 1;
    record(pl, 4, st);
    if (Y && max_len < S) {
        e = launch_mask_tail(Y, pl->layout, S, D, N, H, max_len, st);
        if (e != cudaSuccess) return cuda_fail(e, "mask launch");
        launches += 1;
    }
    record(pl, 5, st);
    if (pl->timing) pl->slot_pending[pl->slot] = true;
    cudaEventRecord(pl->done, st);
    pl->ran = true;
    pl->g_ctas = geo.ctas; pl->g_tn = geo.tn; pl->g_rres = geo.rres; pl->g_threads = geo.threads;
    pl->g_smem = (int)geo.smem;
    pl->last_launches = launches;
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
    cudaStream_t st = (cudaStream_t)stream;
    if (S < 0 || N < 0) return fail(RNN_ERR_INVALID_ARGUMENT, "seq_length and batch_size must be >= 0");
    if (S > (1 << 30) || N > kMaxBatch)
        return fail(RNN_ERR_UNSUPPORTED, "static-scratch runs take at most %lld batch rows", (long long)kMaxBatch);
    const int64_t H = pl->H, I = pl->I, G = pl->G, D = pl->D, GH = G * H;
    if (pl->op != RNN_OP_LSTM) { c0 = nullptr; P = nullptr; Yc = nullptr; }
    const double per_dir = (double)S * N * GH + 4.0 * N * H + (pl->const_weights ? 0.0 : (double)GH * (I + H));
    if (per_dir >= 1073741824.0)
        return fail(RNN_ERR_UNSUPPORTED, "per-direction scratch of %.0f floats reaches the 2^30 limit", per_dir);
    if (S == 0 || N == 0) {
        const size_t sb = sizeof(float) * (size_t)D * N * H;
        cudaError_t e = cudaSuccess;
        if (Yh && sb) e = h0 ? cudaMemcpyAsync(Yh, h0, sb, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(Yh, 0, sb, st);
        if (e == cudaSuccess && Yc && sb)
            e = c0 ? cudaMemcpyAsync(Yc, c0, sb, cudaMemcpyDeviceToDevice, st) : cudaMemsetAsync(Yc, 0, sb, st);
        if (e != cudaSuccess) return cuda_fail(e, "zero-size copy");
        return RNN_OK;
    }
    if (!X && I > 0) return fail(RNN_ERR_INVALID_ARGUMENT, "X is NULL");
    if (!pl->const_weights && (!R || (!W && I > 0))) return fail(RNN_ERR_INVALID_ARGUMENT, "W and R are required");

    DeviceInfo di;
    rnn_status rs = device_info(&di);
    if (rs != RNN_OK) return rs;
    if (!di.coop) return fail(RNN_ERR_UNSUPPORTED, "device lacks cooperative launch");

    int64_t max_len = S;
    if (lens) {
        int32_t host_lens[kMaxBatch];
        cudaError_t e = cudaMemcpyAsync(host_lens, lens, sizeof(int32_t) * (size_t)N, cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e, "copying sequence_lens");
        max_len = 0;
        for (int64_t n = 0; n < N; ++n) {
            const int32_t L = host_lens[n];
            if (L < 0 || (int64_t)L > S)
                return fail(RNN_ERR_INVALID_INPUT, "sequence_lens[%lld] = %d is outside [0, %lld]", (long long)n, L,
                            (long long)S);
            max_len = std::max<int64_t>(max_len, L);
        }
    }

    Geometry geo{};
    rs = plan_geometry(pl, N, di, &geo);
    if (rs != RNN_OK) return rs;

    void* base = nullptr;
    size_t cap = 0;
    cudaError_t e = static_scratch(&base, &cap);
    if (e != cudaSuccess) return cuda_fail(e, "looking up the static scratch");
    const int64_t M = S * N;
    size_t off = 256;   // control words: barrier counters, status
    const size_t o_wt = off; off += pl->const_weights ? 0 : align256(sizeof(float) * (size_t)I * D * GH);
    const size_t o_rt = off; off += pl->const_weights ? 0 : align256(sizeof(float) * (size_t)D * H * GH);
    const size_t o_xw = off; off += align256(sizeof(float) * (size_t)M * D * GH);
    const size_t o_hb = off; off += align256(sizeof(float) * (size_t)D * 2 * H * geo.npad);
    const bool need_rh = pl->op == RNN_OP_GRU && pl->lbr == 0;
    const size_t o_rh = off; off += need_rh ? align256(sizeof(float) * (size_t)D * H * geo.npad) : 0;
    if (off > cap)
        return fail(RNN_ERR_UNSUPPORTED, "run needs %zu bytes of scratch; the static scratch holds %zu", off, cap);
    char* sb = (char*)base;

    e = cudaMemsetAsync(sb + 64, 0, sizeof(int), st);   // status word starts at 0 on every call
    if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
    float* wt = pl->const_weights ? pl->wt_const : (float*)(sb + o_wt);
    float* rt = pl->const_weights ? pl->rt_const : (float*)(sb + o_rt);
    float* xw = (float*)(sb + o_xw);
    const bool exact = pl->mode == RNN_MODE_EXACT;
    int launches = 0;
    if (!pl->const_weights) {
        e = launch_pack(W, R, wt, rt, (int)D, (int)G, H, I, st);
        if (e != cudaSuccess) return cuda_fail(e, "pack launch");
        launches += (int)D * (I > 0 ? 2 : 1);
    }
    e = launch_projection(X, wt, xw, M, I, D * GH, exact, st);
    if (e != cudaSuccess) return cuda_fail(e, "projection launch");
    launches += 1;

    RecParams p;
    std::memset(&p, 0, sizeof p);
    p.op = pl->op; p.G = (int)G; p.D = (int)D; p.N = (int)N; p.H = (int)H; p.S = (int)S;
    p.layout = pl->layout; p.lbr = pl->lbr; p.input_forget = pl->input_forget;
    p.has_B = B != nullptr; p.has_P = P != nullptr; p.has_h0 = h0 != nullptr; p.has_c0 = c0 != nullptr;
    p.has_lens = lens != nullptr; p.has_clip = pl->has_clip; p.clip = pl->clip;
    for (int d = 0; d < 2; ++d)
        for (int s = 0; s < 3; ++s) p.act[d][s] = pl->act[d][s];
    p.max_len = (int)max_len;
    p.dir_reverse[0] = pl->direction == RNN_DIR_REVERSE ? 1 : 0;
    p.dir_reverse[1] = 1;
    p.ctas_per_dir = geo.ctas; p.umax = geo.umax; p.rows_per_thread = geo.tn; p.r_resident = geo.rres;
    p.npad = geo.npad;
    p.XW = xw; p.Rt = rt; p.B = B; p.P = P; p.h0 = h0; p.c0 = c0; p.lens = lens;
    p.Y = Y; p.Yh = Yh; p.Yc = Yc;
    p.hbuf = (float*)(sb + o_hb);
    p.rhbuf = need_rh ? (float*)(sb + o_rh) : nullptr;
    p.bar = (unsigned*)sb;           // zeroed by the state set-up kernel
    p.status = (int*)(sb + 64);
    p.spin_limit_ns = kDefaultSpinNs;
    p.debug_skip_cta = -1;

    e = launch_state_init(p, st);
    if (e != cudaSuccess) return cuda_fail(e, "state set-up launch");
    launches += 1;
    e = launch_recurrent(p, exact, geo.threads, geo.smem, st);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent launch");
    launches += 1;
    if (Y && max_len < S) {
        e = launch_mask_tail(Y, pl->layout, S, D, N, H, max_len, st);
        if (e != cudaSuccess) return cuda_fail(e, "mask launch");
        launches += 1;
    }
    pl->g_ctas = geo.ctas; pl->g_tn = geo.tn; pl->g_rres = geo.rres; pl->g_threads = geo.threads;
    pl->g_smem = (int)geo.smem;
    pl->last_launches = launches;
    return RNN_OK;
}

}  // extern "C"
