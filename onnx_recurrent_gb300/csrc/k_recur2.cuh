// Persistent recurrent kernel, dataflow version: TMA tensor copies, a loader
// warp and per-row-group publication counters instead of a device-wide
// barrier.
//
// Same arithmetic as the staged kernel in k_recur.cuh (page "Recurrent
// operators: RNN, GRU, LSTM", Computation: one accumulator per output, k
// increasing from +0; the gate epilogue in the written order), so both give
// the same bits.  What changes is how h moves between steps:
//
//   * CTAs tile (unit group cu) x (row group cr).  CTA (cu, cr) owns hidden
//     units [u0, u1) (all G gate columns of each) for the batch rows of group
//     cr, so its slice of R serves only its own rows and it fetches only their
//     h: hbuf is laid out [D][2][CR][H][NRP], one contiguous k-major block per
//     row group.
//   * Warp 0 is the loader.  Once per product it waits until every CTA of
//     its row group has published the step (one acquire-polled counter per
//     row group that each CTA increments with a release add), then moves the
//     row group's block of h in a few pieces of several 32-k chunks, one
//     tensor copy (TMA) per piece (plus, when R does not fit in shared
//     memory, one tensor copy of the CTA's R columns per chunk), each piece
//     completing on its slot's "full" mbarrier.  Lane j issues piece j, so
//     the copies of a product go out together.  A ring of slots with "empty"
//     mbarriers lets the loader run ahead.  In global memory and in shared
//     memory a 32-k chunk of a row has a pitch of 36 floats, which keeps the
//     compute warps' 16-byte loads free of bank conflicts.
//   * The other warps compute.  After the gate epilogue they write their h
//     into the next buffer, meet at a named barrier, and one thread adds 1 to
//     the row group's counter (one publication per step, two for GRU with
//     linear_before_reset = 0, whose r (.) h block is published in between).
//     A CTA can publish again only after reading every publication of the
//     others, so the counter reaches target * (unit groups) exactly when
//     every CTA of the row group has published `target` times.
//   Two h buffers suffice: a CTA can only overwrite buffer b after every
//   producer of its row group has published the step that reads b.
//   * With the in-cluster exchange (CL instances) a row group is one
//     thread-block cluster: every CTA keeps the row group's whole h in its own
//     shared memory and writes the h it computes into every peer's copy
//     (distributed shared memory); arrivals on the peers' mbarriers replace
//     the counter, the loader and the tensor copies of h.
//
// Every wait is bounded (globaltimer): a CTA that gives up records
// RNN_ERR_TIMEOUT in the status word; CTAs that see a non-zero status stop.
// The compute warps leave only at a publish barrier, so no warp is left
// waiting on a named barrier, and the loader waits for its own copies in
// flight before it exits.  A CL CTA does not leave early at all: it runs its
// remaining steps without waiting and meets its cluster at the end.
#pragma once

#include <cstdint>
#include <type_traits>

#include "k_recur.cuh"

namespace rnngb {

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Bounded wait on an mbarrier phase.  Gives up (returning false) when the
// CTA is aborting, another CTA reported a failure, or the limit passes.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned parity, int* status, volatile int* abort_flag,
                                          long long limit_ns)
{
    if (mbar_test(bar, parity)) return true;
    if (*abort_flag) return false;
    const unsigned long long t0 = globaltimer_ns();
    unsigned it = 0;
    while (!mbar_test(bar, parity)) {
        if ((++it & 15u) == 0u) {
            if (*abort_flag) return false;
            if (ld_relaxed_s32(status) != 0) { *abort_flag = 1; return false; }
            if ((long long)(globaltimer_ns() - t0) > limit_ns) {
                atomicCAS(status, 0, 6 /* RNN_ERR_TIMEOUT */);
                *abort_flag = 1;
                return false;
            }
        }
    }
    return true;
}

// First hidden unit of unit group cu: groups hold multiples of `quant`
// units, split as evenly as possible.
__device__ __forceinline__ int unit_begin(int cu, int CU, int H, int quant)
{
    const int Q = H / quant;
    return quant * (int)(((long long)cu * Q) / CU);
}

struct DfCtx {
    int d, cu, cr, H, HP, G, GH, CU, CR, u0, U, umax, ugs, NR, NRP, nchunks, cpb, npieces, slots;
    int KR;           // k of each gate row held resident: H, or the leading res_chunks * 32 (0: none)
    int KRP;          // floats between a unit's resident gate rows
    int rpieces;      // pieces whose R is resident (the leading ones); the others stream
    int ctid, ncompute, ul, rb;
    int gi;           // gate split: this thread's share of the gate columns (0: all, or the first share)
    bool active;      // takes part in the products
    bool lead;        // owns the (unit, row tile): gate arithmetic, state, stores
    float* Rs;        // resident R: [umax][ugs] floats (unit-major, gate rows of KR k, KRP apart)
    char* Rring;      // streamed R: slots x rslot bytes, each cpb chunks of [G][umax][36]
    char* Hring;      // slots x hslot bytes, each [cpb][NRP][36] (padded to 128 bytes)
    int rslot, rsub, hslot; // bytes per slot (one piece: cpb chunks of 32 k), per R chunk
    uint64_t* full;
    uint64_t* empty;
    uint64_t* pub;    // completes a phase at each of this CTA's publications
};

// Loader: the pieces of one product (one accumulate pass of the compute
// warps).  `map` describes the h (or r (.) h) exchange buffer, `z` the row
// group's block in it; every producer of the row group must have published
// `target` times before the block may be read.  Streamed R pieces bring the
// ng gate rows from gate g0 on that the product uses (`rmap` has a box of ng
// gates); they land from the start of each chunk's sub-block.
__device__ __forceinline__ bool load_product(const RecParams& p, const DfCtx& x, const CUtensorMap* map, int z,
                                             unsigned target, const unsigned* counter, unsigned& q,
                                             volatile int* abort_flag, int lane, const CUtensorMap* rmap, int g0,
                                             int ng)
{
    // One tensor copy of h per piece of cpb chunks (a box of many small
    // copies lands one after another, a few large boxes land together), and
    // for a streamed piece one of R per chunk.  Pieces are issued by the
    // lanes in parallel, lane j taking piece base + j, in groups no larger
    // than the ring (so no two lanes share a slot).  R does not depend on h:
    // the first group claims its slots and starts its R copies before the
    // wait for the producers, so they run during the exchange.
    const unsigned hbytes = (unsigned)x.NRP * x.cpb * (kDfPitch * 4u);
    const int gsz = min(32, x.slots);
    auto claim = [&](int base, int nmine) -> bool {   // wait for the slots, expect the bytes, copy R
        const bool mine = lane < nmine;
        const unsigned qq = q + (unsigned)lane;
        const int slot = (int)(qq % (unsigned)x.slots);
        const unsigned round = qq / (unsigned)x.slots;
        bool ok = true;
        if (mine) ok = mbar_wait(&x.empty[slot], (round & 1u) ^ 1u, p.status, abort_flag, p.spin_limit_ns);
        if (!__all_sync(0xffffffffu, ok)) return false;
        if (mine) {
            const int c0 = (base + lane) * x.cpb;           // first chunk of the piece
            const int nc = min(x.cpb, x.nchunks - c0);      // R chunks to copy (h: the whole box)
            const bool rstream = base + lane >= x.rpieces;
            const unsigned rbytes = rstream ? (unsigned)(nc * ng * x.umax) * (kDfPitch * 4u) : 0u;
            mbar_arrive_expect_tx(&x.full[slot], hbytes + rbytes);
            if (rstream)
                for (int cl = 0; cl < nc; ++cl)
                    tma_load_4d(x.Rring + (size_t)slot * x.rslot + (size_t)cl * x.rsub, rmap, (c0 + cl) * kRecKC,
                                x.u0, g0, x.d, &x.full[slot]);
        }
        return true;
    };
    auto copy_h = [&](int base, int nmine) {
        if (lane < nmine) {
            const int slot = (int)((q + (unsigned)lane) % (unsigned)x.slots);
            tma_load_4d(x.Hring + (size_t)slot * x.hslot, map, 0, 0, (base + lane) * x.cpb, z, &x.full[slot]);
        }
    };
    const int pre = min(gsz, x.npieces);
    if (!claim(0, pre)) return false;
    if (target > 0) {
        // This CTA's own publication comes first (the counter cannot be
        // complete before it); waiting for it on the mbarrier keeps the
        // loader off the memory pipe while the compute warps work.  Every
        // lane then polls the row group's counter (acquire loads); a proxy
        // fence orders the generic-proxy writes that the acquire made
        // visible before the tensor copies (async proxy) that read them.
        const unsigned qa = q;
        q += (unsigned)pre;   // armed: the exit wait covers these slots
        if (!mbar_wait(x.pub, (target - 1u) & 1u, p.status, abort_flag, p.spin_limit_ns)) return false;
        const unsigned need = target * (unsigned)x.CU;
        bool ready = ld_acquire_u32(counter) >= need;
        if (!__all_sync(0xffffffffu, ready)) {
            const unsigned long long t0 = globaltimer_ns();
            unsigned it = 0;
            while (!__all_sync(0xffffffffu, ready)) {
                if (!ready) ready = ld_acquire_u32(counter) >= need;
                if ((++it & 15u) == 0u) {
                    int bad = 0;
                    if (lane == 0) {
                        if (*abort_flag || ld_relaxed_s32(p.status) != 0) bad = 1;
                        else if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) {
                            atomicCAS(p.status, 0, 6 /* RNN_ERR_TIMEOUT */);
                            bad = 1;
                        }
                    }
                    if (__shfl_sync(0xffffffffu, bad, 0)) {
                        if (lane == 0) *abort_flag = 1;
                        return false;
                    }
                }
            }
        }
        __syncwarp();
        fence_proxy_async_global();
        __syncwarp();
        q = qa;
    }
    copy_h(0, pre);
    q += (unsigned)pre;
    for (int base = pre; base < x.npieces; base += gsz) {
        const int nmine = min(gsz, x.npieces - base);
        if (!claim(base, nmine)) return false;
        copy_h(base, nmine);
        q += (unsigned)nmine;
    }
    return true;
}

// The products of one piece for a thread's TN rows and NC gate columns:
// acc[i][g] += h[row_i][k] * R[gate g][k] over the piece's k, ascending, 4 k
// per vector load.  Operands are loaded PD groups of 4 k ahead (a ring of
// PD + 1 register buffers that runs on across chunk boundaries); the ring
// length divides the 8 groups of a chunk, so every buffer index is a
// compile-time constant.  h rows (and streamed R rows) have a pitch of 36
// floats; chunk cl of a piece is cl * hstep bytes (R: rsub bytes) further on.
template <int TN, int NC, bool EXACT, bool RES>
__device__ __forceinline__ void df_piece(const char* const (&hp)[TN], int hstep, const char* const (&rp)[NC],
                                         int rstep, int ngroups, float (&acc)[TN][NC])
{
    constexpr int PD = TN == 1 ? 3 : 1;
    constexpr int NB = PD + 1;
    static_assert(8 % NB == 0 && PD < 8, "ring length must divide the groups of a chunk");
    float4 hv[NB][TN], rv[NB][NC];
    // group jc (compile-time, 0..7) of the chunk at byte offsets oh / orr
    auto load = [&](int buf, int oh, int orr, int jc) {
#pragma unroll
        for (int i = 0; i < TN; ++i) hv[buf][i] = *reinterpret_cast<const float4*>(hp[i] + oh + jc * 16);
#pragma unroll
        for (int g = 0; g < NC; ++g) rv[buf][g] = *reinterpret_cast<const float4*>(rp[g] + orr + jc * 16);
    };
#pragma unroll
    for (int b = 0; b < PD; ++b)
        if (b < ngroups) load(b, 0, 0, b);
    const int nch = (ngroups + 7) / 8;
    for (int cl = 0; cl < nch; ++cl) {
        const int oh = cl * hstep, orr = cl * rstep;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int jj = cl * 8 + j;
            if (jj >= ngroups) break;
            if (jj + PD < ngroups) {
                if (j + PD < 8) load((j + PD) % NB, oh, orr, j + PD);
                else load((j + PD) % NB, oh + hstep, orr + rstep, j + PD - 8);
            }
            const int b = j % NB;
#pragma unroll
            for (int i = 0; i < TN; ++i)
#pragma unroll
                for (int g = 0; g < NC; ++g) acc[i][g] = mac<EXACT>(acc[i][g], hv[b][i].x, rv[b][g].x);
#pragma unroll
            for (int i = 0; i < TN; ++i)
#pragma unroll
                for (int g = 0; g < NC; ++g) acc[i][g] = mac<EXACT>(acc[i][g], hv[b][i].y, rv[b][g].y);
#pragma unroll
            for (int i = 0; i < TN; ++i)
#pragma unroll
                for (int g = 0; g < NC; ++g) acc[i][g] = mac<EXACT>(acc[i][g], hv[b][i].z, rv[b][g].z);
#pragma unroll
            for (int i = 0; i < TN; ++i)
#pragma unroll
                for (int g = 0; g < NC; ++g) acc[i][g] = mac<EXACT>(acc[i][g], hv[b][i].w, rv[b][g].w);
        }
    }
}

// Compute warps: acc[i][j] += sum_k src[row_i][k] * R[gate col_off + j][k]
// over the product's pieces (k ascending).  Streamed pieces hold the gate
// rows from ring_g0 on.  Returns false once the CTA is aborting (the
// remaining pieces are then skipped, not waited for).
template <int TN, int NC, bool EXACT>
__device__ __forceinline__ bool consume_product(const RecParams& p, const DfCtx& x, int col_off, int ring_g0,
                                                float (&acc)[TN][NC], unsigned& q, volatile int* abort_flag,
                                                int lane, bool live)
{
    bool ok = true;
    for (int pc = 0; pc < x.npieces; ++pc, ++q) {
        const int slot = (int)(q % (unsigned)x.slots);
        const unsigned round = q / (unsigned)x.slots;
        if (ok) ok = mbar_wait(&x.full[slot], round & 1u, p.status, abort_flag, p.spin_limit_ns);
        if (ok && x.active && live) {
            const int k0 = pc * x.cpb * kRecKC;
            const int ngroups = (min(x.cpb * kRecKC, x.H - k0) + 3) / 4;
            const char* hbox = x.Hring + (size_t)slot * x.hslot;
            const char* hp[TN];
#pragma unroll
            for (int i = 0; i < TN; ++i) hp[i] = hbox + (size_t)(x.rb * TN + i) * (kDfPitch * 4);
            const int hstep = x.NRP * kDfPitch * 4;
            const char* rp[NC];
            if (pc < x.rpieces) {
                const float* rbase = x.Rs + (size_t)x.ul * x.ugs + (size_t)col_off * x.KRP + k0;
#pragma unroll
                for (int g = 0; g < NC; ++g) rp[g] = reinterpret_cast<const char*>(rbase + (size_t)g * x.KRP);
                df_piece<TN, NC, EXACT, true>(hp, hstep, rp, kRecKC * 4, ngroups, acc);
            } else {
                const char* rbox = x.Rring + (size_t)slot * x.rslot;
#pragma unroll
                for (int g = 0; g < NC; ++g)
                    rp[g] = rbox + (size_t)((col_off - ring_g0 + g) * x.umax + x.ul) * (kDfPitch * 4);
                df_piece<TN, NC, EXACT, false>(hp, hstep, rp, x.rsub, ngroups, acc);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&x.empty[slot]);
    }
    return ok;
}

// Gate activations: the ones the operator names (FX = false), or the default
// set with its functions called directly (FX = true), which leaves the
// compiler free to interleave the independent gates' chains.
template <bool EXACT>
__device__ __forceinline__ float sigmoid_fn(float v) { return EXACT ? dx_sigmoid(v) : df_sigmoid(v); }
template <bool EXACT>
__device__ __forceinline__ float tanh_fn(float v) { return EXACT ? dx_tanh(v) : df_tanh(v); }

template <int OP, bool EXACT, bool FX>
struct Acts {
    ActSpec f, g, h;
    __device__ __forceinline__ float F(float v) const
    {
        if constexpr (FX) return OP == 0 ? tanh_fn<EXACT>(v) : sigmoid_fn<EXACT>(v);
        else return act<EXACT>(f, v);
    }
    __device__ __forceinline__ float Gf(float v) const
    {
        if constexpr (FX) return tanh_fn<EXACT>(v);
        else return act<EXACT>(g, v);
    }
    __device__ __forceinline__ float Hf(float v) const
    {
        if constexpr (FX) return tanh_fn<EXACT>(v);
        else return act<EXACT>(h, v);
    }
};

// Compute warps meet; one thread publishes (adds 1 to the row group's
// counter).  Returns false (uniformly across the compute warps) when the CTA
// is aborting.
__device__ __forceinline__ bool publish(const DfCtx& x, unsigned* counter, volatile int* abort_flag, bool skip)
{
    named_barrier(1, x.ncompute);
    const bool abort_now = *abort_flag != 0;
    named_barrier(1, x.ncompute);   // everyone has read the abort flag
    if (abort_now) return false;
    if (x.ctid == 0) {
        if (!skip) {
            fence_proxy_async_global();
            red_release_add_u32(counter, 1u);   // the named barrier ordered every compute thread's writes first
        }
        mbar_arrive(x.pub);
    }
    return true;
}

// ---- in-cluster exchange (CL): the CTAs of a row group form one thread-block
// cluster; each keeps the whole h of its rows in its own shared memory (two
// buffers by step parity, plus r (.) h for GRU with linear_before_reset = 0),
// writes the h it computes into every peer's buffer (distributed shared
// memory) and arrives on every peer's barrier for that buffer.

// Bounded wait for the peers' arrivals on one of this CTA's exchange barriers.
__device__ __forceinline__ bool cl_wait(uint64_t* bar, unsigned parity, int* status, volatile int* abort_flag,
                                        long long limit_ns)
{
    if (mbar_test_cluster(bar, parity)) return true;
    if (*abort_flag) return false;
    const unsigned long long t0 = globaltimer_ns();
    unsigned it = 0;
    while (!mbar_test_cluster(bar, parity)) {
        if ((++it & 15u) == 0u) {
            if (*abort_flag) return false;
            if ((long long)(globaltimer_ns() - t0) > limit_ns) {
                atomicCAS(status, 0, 6 /* RNN_ERR_TIMEOUT */);
                *abort_flag = 1;
                return false;
            }
        }
    }
    return true;
}

// This CTA's products from its own copy of h (all chunks, k ascending) and
// its resident R slice.
template <int TN, int NC, bool EXACT>
__device__ __forceinline__ void cl_product(const DfCtx& x, const char* hbox, int col_off, float (&acc)[TN][NC])
{
    const char* hp[TN];
#pragma unroll
    for (int i = 0; i < TN; ++i) hp[i] = hbox + (size_t)(x.rb * TN + i) * (kDfPitch * 4);
    const float* rbase = x.Rs + (size_t)x.ul * x.ugs + (size_t)col_off * x.KRP;
    const char* rp[NC];
#pragma unroll
    for (int g = 0; g < NC; ++g) rp[g] = reinterpret_cast<const char*>(rbase + (size_t)g * x.KRP);
    df_piece<TN, NC, EXACT, true>(hp, x.NRP * kDfPitch * 4, rp, kRecKC * 4, (x.H + 3) / 4, acc);
}

// Each compute thread fences its writes into the peers' buffers at cluster
// scope; once all have met, compute thread r arrives (release, cluster
// scope) on the barrier `bar` of the CTA of rank r.  Measured: one thread
// arriving on all 16 peers in turn took about 2 us a step; spread over the
// lanes the exchange costs about a third of the device-wide one.
__device__ __forceinline__ void cl_publish(const DfCtx& x, uint64_t* bar, bool send)
{
    if (send) fence_acq_rel_cluster();
    named_barrier(1, x.ncompute);
    if (send && x.ctid < x.CU) mbar_arrive_cluster(cluster_map(smem_addr(bar), (unsigned)x.ctid));
}

// Threads per CTA: one row per thread keeps three groups of operands in
// flight (up to 255 registers, 256 threads); wider tiles keep one group in
// flight and more accumulators (up to 168 registers, 384 threads); eight rows
// per thread (32 LSTM accumulators) take up to 255 registers, 256 threads.
template <int TN>
struct DfBounds {
    static constexpr int threads = (TN == 1 || TN == 8) ? 256 : 384;
};

// TWO: GRU with linear_before_reset = 0 (two products per step, the second
// over r (.) h); a separate instance keeps its register allocation apart.
// GS > 1 (one product per step): gate split, GS lanes side by side share a
// (unit, row tile), each taking G / GS of the gate columns over all k in
// ascending order (so every accumulator sees the same operations as
// without the split); the first lane of the group gathers the others'
// sums by shuffles and does the gate arithmetic.  A warp holds 32 / GS such
// groups; with GS = 3 its last two lanes idle.
// CL: in-cluster exchange (the launch makes each row group of a direction
// one cluster of unit_groups CTAs; R is resident; no loader work, no
// counters): no CTA leaves before the whole cluster has met at its end, so
// no peer's shared memory is written after its CTA exits.
template <int OP, int TN, bool EXACT, bool TWO, int GS, bool CL>
__global__ void __launch_bounds__(DfBounds<TN>::threads, 1) rnn_dataflow_kernel(const __grid_constant__ RecParams p)
{
    constexpr int G = OP == 0 ? 1 : (OP == 1 ? 3 : 4);
    static_assert(GS == 1 || (!TWO && G % GS == 0), "gate split: one product per step, whole gate shares");
    static_assert(!CL || GS == 1, "in-cluster exchange without gate split");
    constexpr int NCG = G / GS;       // gate columns per thread
    extern __shared__ __align__(128) unsigned char df_smem[];
    __shared__ __align__(8) uint64_t s_full[kMaxSlots];
    __shared__ __align__(8) uint64_t s_empty[kMaxSlots];
    __shared__ __align__(8) uint64_t s_pub, s_rfill;
    __shared__ __align__(8) uint64_t s_hready[2], s_rhready;   // CL: peers' h / r (.) h landed
    __shared__ int s_abort;

    DfCtx x;
    const int per_dir = p.ctas_per_dir;           // CU * CR
    x.d = blockIdx.x / per_dir;
    const int c = blockIdx.x - x.d * per_dir;
    x.CU = p.unit_groups;
    x.CR = p.row_groups;
    x.cr = c / x.CU;
    x.cu = c - x.cr * x.CU;
    x.H = p.H;
    x.HP = p.hpad;
    x.G = G;
    x.GH = G * p.H;
    x.u0 = unit_begin(x.cu, x.CU, p.H, 1);
    x.U = unit_begin(x.cu + 1, x.CU, p.H, 1) - x.u0;
    x.umax = p.umax;
    x.ugs = p.unit_stride;
    x.NRP = p.npad;                               // padded rows per group
    x.NR = max(0, min(p.N - x.cr * x.NRP, x.NRP));
    x.nchunks = (p.H + kRecKC - 1) / kRecKC;
    x.cpb = p.chunks_per_piece;
    x.npieces = (x.nchunks + x.cpb - 1) / x.cpb;
    x.slots = p.slots;
    x.hslot = (int)df_hslot_bytes(x.NRP, x.cpb);   // 128-byte aligned slot starts
    x.rsub = (int)df_rsub_bytes(x.umax, G);
    x.rslot = p.r_resident ? 0 : x.cpb * x.rsub;
    // R resident in full, or its leading res_chunks 32-k chunks (whole pieces)
    x.KR = p.r_resident ? p.H : p.res_chunks * kRecKC;
    x.KRP = df_gate_stride(x.KR);
    x.rpieces = p.r_resident ? x.npieces : p.res_chunks / x.cpb;
    x.ncompute = blockDim.x - 32;
    x.ctid = (int)threadIdx.x - 32;
    const int RB = x.NRP / TN;
    // t: the thread's (unit, row tile) index; gate split: lane groups of GS
    int t = x.ctid;
    x.gi = 0;
    if (GS > 1 && x.ctid >= 0) {
        constexpr int NG = 32 / GS;
        const int gq = (x.ctid & 31) / GS;
        x.gi = (x.ctid & 31) - gq * GS;
        t = gq < NG ? (x.ctid >> 5) * NG + gq : 1 << 30;
    }
    if (p.unit_fastest) {
        // the lanes of a quarter warp share a row tile (their h loads are
        // broadcasts) and take distinct units (R rows 144 bytes apart)
        x.ul = x.ctid >= 0 ? t % x.umax : 0;
        x.rb = x.ctid >= 0 ? t / x.umax : 0;
    } else {
        x.rb = x.ctid >= 0 ? t % RB : 0;
        x.ul = x.ctid >= 0 ? t / RB : 0;
    }
    x.active = x.ctid >= 0 && x.ul < x.U && x.rb < RB && x.rb * TN < x.NR;
    x.lead = x.active && x.gi == 0;
    // tensor-copy destinations are 128-byte aligned
    unsigned char* base = df_smem + ((128u - (smem_addr(df_smem) & 127u)) & 127u);
    const size_t rres = x.KR > 0 ? (((size_t)x.umax * x.ugs * 4 + 127) / 128) * 128 : 0;
    x.Rs = reinterpret_cast<float*>(base);
    x.Rring = reinterpret_cast<char*>(base + rres);
    x.Hring = reinterpret_cast<char*>(base + rres + (size_t)x.slots * x.rslot);
    // CL: h buffers 0 and 1, then r (.) h, each one row group's block
    const size_t clb = CL ? (((size_t)x.NRP * (x.HP / kRecKC) * kDfPitch * 4 + 127) / 128) * 128 : 0;
    auto clbuf = [&](int i) { return reinterpret_cast<char*>(base + rres + (size_t)i * clb); };
    x.full = s_full;
    x.empty = s_empty;
    x.pub = &s_pub;

    const int lane = threadIdx.x & 31;
    const int d = x.d;
    const bool rev = p.dir_reverse[d] != 0;
    const int nwarps_compute = x.ncompute / 32;
    const size_t blk = (size_t)x.NRP * (x.HP / kRecKC) * kDfPitch;   // one row group's block
    // a unit's slot in a row group's block: [u / 32][row][u % 32], rows of 36
    auto xoff = [&](int rl, int uu) { return ((size_t)(uu / kRecKC) * x.NRP + rl) * kDfPitch + (uu % kRecKC); };
    const int zh0 = (d * 2 + 0) * x.CR + x.cr;                   // tensor-map block index, buffer 0
    auto hblock = [&](int buf) { return p.hbuf + ((size_t)(d * 2 + buf) * x.CR + x.cr) * blk; };
    auto rhblock = [&](int buf) { return p.rhbuf + ((size_t)(d * 2 + buf) * x.CR + x.cr) * blk; };
    unsigned* counter = p.flags + (size_t)(d * x.CR + x.cr);
    constexpr bool two_phase = TWO;

    if (threadIdx.x == 0) {
        for (int i = 0; i < x.slots; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], (unsigned)nwarps_compute);
        }
        mbar_init(&s_pub, 1);
        mbar_init(&s_rfill, 1);
        if (CL) {
            mbar_init(&s_hready[0], (unsigned)x.CU);
            mbar_init(&s_hready[1], (unsigned)x.CU);
            mbar_init(&s_rhready, (unsigned)x.CU);
        }
        s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();
    // CL: every peer's barriers are initialised before any arrival on them
    if constexpr (CL) cluster_sync_all();
    if (x.KR > 0 && threadIdx.x < 32) {
        // R[d][g*H + u][k] -> Rs[(u - u0) * ugs + g*KRP + k], k < KR: one bulk copy of
        // a row of KR floats per (unit, gate), all completing on s_rfill
        // (H is a multiple of 4 and ugs*4 of 16, so every copy is 16-byte
        // aligned at both ends)
        const float* src = p.Rorig + (size_t)d * G * p.H * p.H;
        // CL: also the row group's block of the exchange buffer (h before
        // the first step) into h buffer 0
        const unsigned hb0 = CL ? (unsigned)(x.NRP * (x.HP / kRecKC) * kDfPitch) * 4u : 0u;
        if (lane == 0) mbar_arrive_expect_tx(&s_rfill, (unsigned)(x.U * G * x.KR) * 4u + hb0);
        __syncwarp();
        if (CL && lane == 0) bulk_g2s(clbuf(0), hblock(0), hb0, &s_rfill);
        for (int j = lane; j < x.U * G; j += 32) {
            const int ul = j / G, g = j - ul * G;
            bulk_g2s(x.Rs + (size_t)ul * x.ugs + (size_t)g * x.KRP, src + ((size_t)g * p.H + x.u0 + ul) * p.H,
                     (unsigned)x.KR * 4u, &s_rfill);
        }
    }

    // ------------------------------------------------------------ loader
    if (CL && threadIdx.x < 32) {
        // nothing to stream: wait (bounded) for the fill, then meet the
        // cluster at its end
        if (lane == 0) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_test(&s_rfill, 0u) && (long long)(globaltimer_ns() - t0) <= p.spin_limit_ns) {
            }
        }
        __syncwarp();
        cluster_sync_all();
        return;
    }
    if (threadIdx.x < 32) {
        unsigned q = 0;
        bool ok = true;
        for (int s = 0; s < p.max_len && ok; ++s) {
            const int zh = zh0 + (s & 1) * x.CR;
            if (two_phase) {
                // z and r rows with h, the candidate's rows with r (.) h
                ok = load_product(p, x, &p.hmap, zh, 2u * s, counter, q, &s_abort, lane, &p.rmap, 0, 2);
                if (ok)
                    ok = load_product(p, x, &p.rhmap, zh, 2u * s + 1u, counter, q, &s_abort, lane, &p.rmap2, 2, 1);
            } else {
                ok = load_product(p, x, &p.hmap, zh, (unsigned)s, counter, q, &s_abort, lane, &p.rmap, 0, G);
            }
        }
        // wait (bounded) for this CTA's copies still in flight before leaving
        if (lane == 0 && x.KR > 0) {
            const unsigned long long t0 = globaltimer_ns();
            while (!mbar_test(&s_rfill, 0u) && (long long)(globaltimer_ns() - t0) <= p.spin_limit_ns) {
            }
        }
        if (lane == 0) {
            const unsigned issued = q;
            for (int sl = 0; sl < x.slots && (unsigned)sl < issued; ++sl) {
                const unsigned last = issued - 1u - (unsigned)((issued - 1u - sl) % (unsigned)x.slots);
                const unsigned long long t0 = globaltimer_ns();
                while (!mbar_test(&s_full[last % x.slots], (last / x.slots) & 1u)) {
                    if ((long long)(globaltimer_ns() - t0) > p.spin_limit_ns) break;
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ compute
    const int u = x.u0 + x.ul;
    const ActSpec fA = p.act[d][0], gA = p.act[d][1], hA = p.act[d][2];
    // the operator's default activations (RNN Tanh; GRU Sigmoid, Tanh; LSTM
    // Sigmoid, Tanh, Tanh)
    const bool fixed_acts = OP == 0 ? fA.fn == 1
                                    : (OP == 1 ? fA.fn == 2 && gA.fn == 1 : fA.fn == 2 && gA.fn == 1 && hA.fn == 1);
    float wb[G], rbv[G];
    float pI = 0.f, pO = 0.f, pF = 0.f;
    float hown[TN], cown[TN], xw[TN][G];
    int len[TN];
    // rows: the exchange buffers use the internal row rl of the row group;
    // with sequence_lens the rows are ranked by length (longest first, so a
    // row tile whose first row has finished has finished altogether) and
    // rown[i] is the caller's row behind internal row cr * NRP + rl
    int rown[TN];
    int tile_len = 0;
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
#pragma unroll
    for (int i = 0; i < TN; ++i) {
        const int rl = x.rb * TN + i;
        const bool ok = x.active && rl < x.NR;
        const int ni = x.cr * x.NRP + rl;
        const int n = ok ? (p.perm ? p.perm[ni] : ni) : 0;
        rown[i] = n;
        len[i] = ok ? (p.has_lens ? p.lens[n] : p.S) : 0;
        tile_len = len[i] > tile_len ? len[i] : tile_len;
        hown[i] = (ok && p.has_h0) ? io_load(p.h0, s_index(p, d, n, u), p.io) : 0.f;
        cown[i] = (ok && OP == 2 && p.has_c0) ? io_load(p.c0, s_index(p, d, n, u), p.io) : 0.f;
    }
    const size_t xw_ld = (size_t)p.D * x.GH;
    const size_t xw_col = (size_t)d * x.GH + (size_t)u * G;
    auto xw_row = [&](int s, int i) {
        const int n = rown[i];
        const int t = rev ? len[i] - 1 - s : s;
        const size_t row = p.layout == 0 ? (size_t)t * p.N + n : (size_t)n * p.S + t;
        return p.XW + row * xw_ld + xw_col;
    };
    auto load_xw = [&](int s) {
#pragma unroll
        for (int i = 0; i < TN; ++i) {
            const int rl = x.rb * TN + i;
            if (x.lead && rl < x.NR && s < len[i]) {
                const float* q = xw_row(s, i);
#pragma unroll
                for (int g = 0; g < G; ++g) xw[i][g] = __ldg(q + g);
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) xw[i][g] = 0.f;
            }
        }
    };
    // Wide row tiles (4 or 8 rows per thread) have no registers to spare for
    // the next step's XW during a product: they ask L2 for this step's XW
    // before the product and load it into registers after it.
    constexpr bool XW_LATE = TN >= 4;
    auto prefetch_xw = [&](int s) {
#pragma unroll
        for (int i = 0; i < TN; ++i) {
            const int rl = x.rb * TN + i;
            if (x.lead && rl < x.NR && s < len[i]) prefetch_l2(xw_row(s, i));
        }
    };

    unsigned q = 0;
    const bool skip_first = p.debug_skip_cta == (int)blockIdx.x;
    // the resident R slice must have landed (a failure here sets the abort
    // flag, and the warps leave together at the first publication)
    if (x.KR > 0) mbar_wait(&s_rfill, 0u, p.status, &s_abort, p.spin_limit_ns);
    if (!XW_LATE) load_xw(0);
    for (int s = 0; s < p.max_len; ++s) {
        float xc[TN][G];
        // the step's XW: prefetched into registers during the previous step,
        // or (wide tiles) requested from L2 now and loaded after the product
        auto take_xw = [&]() {
#pragma unroll
            for (int i = 0; i < TN; ++i)
#pragma unroll
                for (int g = 0; g < G; ++g) xc[i][g] = xw[i][g];
        };
        auto next_xw = [&]() {
            if constexpr (XW_LATE) {
                load_xw(s);
                take_xw();
            } else if (s + 1 < p.max_len) {
                load_xw(s + 1);
            }
        };
        if constexpr (XW_LATE) prefetch_xw(s);
        else take_xw();
        float* hdst = hblock((s + 1) & 1);
        // CL: no exchange of the last step's h (nothing reads it)
        const bool cl_send = s + 1 < p.max_len;
        const unsigned cl_h = CL ? smem_addr(clbuf((s + 1) & 1)) : 0u;
        auto put_h = [&](size_t off, float v) {
            if constexpr (CL) {
                if (cl_send)
                    for (int r = 0; r < x.CU; ++r) st_cluster_f32(cluster_map(cl_h + (unsigned)off * 4u, (unsigned)r), v);
            } else {
                hdst[off] = v;
            }
        };
        if constexpr (CL) {
            if (s > 0) cl_wait(&s_hready[s & 1], (unsigned)((s - 1) >> 1) & 1u, p.status, &s_abort, p.spin_limit_ns);
        }
        const bool live = s < tile_len;   // a finished row tile skips its products (its rows stay frozen)

        if constexpr (TWO) {
            {
                float az[TN][2];
#pragma unroll
                for (int i = 0; i < TN; ++i) { az[i][0] = 0.f; az[i][1] = 0.f; }
                if constexpr (CL) {
                    if (x.active && live) cl_product<TN, 2, EXACT>(x, clbuf(s & 1), 0, az);
                } else {
                    consume_product<TN, 2, EXACT>(p, x, 0, 0, az, q, &s_abort, lane, live);
                }
                next_xw();
                float zg[TN];
                float* rh = rhblock(s & 1);
                auto epi_r = [&](auto fx) {
                    constexpr bool FX = decltype(fx)::value;
                    const Acts<OP, EXACT, FX> A{fA, gA, hA};
#pragma unroll
                    for (int i = 0; i < TN; ++i) {
                        const int rl = x.rb * TN + i;
                        zg[i] = 0.f;
                        if (!(x.lead && rl < x.NR)) continue;
                        float rhv = 0.f;
                        if (s < len[i]) {
                            float pz = fadd(xc[i][0], az[i][0]);
                            float pr = fadd(xc[i][1], az[i][1]);
                            if (p.has_B) {
                                pz = fadd(pz, wb[0]); pz = fadd(pz, rbv[0]);
                                pr = fadd(pr, wb[1]); pr = fadd(pr, rbv[1]);
                            }
                            zg[i] = A.F(clipv(p, pz));
                            const float r = A.F(clipv(p, pr));
                            rhv = fmul(r, hown[i]);
                        }
                        if constexpr (CL) {
                            const unsigned a = smem_addr(clbuf(2)) + (unsigned)xoff(rl, u) * 4u;
                            for (int r = 0; r < x.CU; ++r) st_cluster_f32(cluster_map(a, (unsigned)r), rhv);
                        } else {
                            rh[xoff(rl, u)] = rhv;
                        }
                    }
                };
                if (fixed_acts) epi_r(std::true_type{});
                else epi_r(std::false_type{});
                if constexpr (CL) {
                    cl_publish(x, &s_rhready, !(skip_first && s == 0));
                    cl_wait(&s_rhready, (unsigned)s & 1u, p.status, &s_abort, p.spin_limit_ns);
                } else if (!publish(x, counter, &s_abort, skip_first && s == 0)) {
                    return;
                }
                float ah[TN][1];
#pragma unroll
                for (int i = 0; i < TN; ++i) ah[i][0] = 0.f;
                if constexpr (CL) {
                    if (x.active && live) cl_product<TN, 1, EXACT>(x, clbuf(2), 2, ah);
                } else {
                    consume_product<TN, 1, EXACT>(p, x, 2, 2, ah, q, &s_abort, lane, live);
                }
                auto epi = [&](auto fx) {
                    constexpr bool FX = decltype(fx)::value;
                    const Acts<OP, EXACT, FX> A{fA, gA, hA};
#pragma unroll
                    for (int i = 0; i < TN; ++i) {
                        const int rl = x.rb * TN + i;
                        const int n = rown[i];
                        if (!(x.lead && rl < x.NR)) continue;
                        if (s < len[i]) {
                            const int t = rev ? len[i] - 1 - s : s;
                            float ph = fadd(xc[i][2], ah[i][0]);
                            if (p.has_B) { ph = fadd(ph, wb[2]); ph = fadd(ph, rbv[2]); }
                            const float ht = A.Gf(clipv(p, ph));
                            const float hn = fadd(fmul(fsub(1.0f, zg[i]), ht), fmul(zg[i], hown[i]));
                            hown[i] = hn;
                            if (p.Y) io_store(p.Y, y_index(p, t, d, n, u), canon_nan(hn), p.io);
                        } else if (p.Y) {
                            io_store(p.Y, y_index(p, s, d, n, u), 0.f, p.io);
                        }
                        put_h(xoff(rl, u), hown[i]);
                    }
                };
                if (fixed_acts) epi(std::true_type{});
                else epi(std::false_type{});
                if constexpr (CL) cl_publish(x, &s_hready[(s + 1) & 1], cl_send && !(skip_first && s == 0));
                else if (!publish(x, counter, &s_abort, false)) return;
            }
        } else {
            float acc[TN][G];
            {
                float part[TN][NCG];
#pragma unroll
                for (int i = 0; i < TN; ++i)
#pragma unroll
                    for (int g = 0; g < NCG; ++g) part[i][g] = 0.f;
                if constexpr (CL) {
                    if (x.active && live) cl_product<TN, NCG, EXACT>(x, clbuf(s & 1), 0, part);
                } else {
                    consume_product<TN, NCG, EXACT>(p, x, x.gi * NCG, 0, part, q, &s_abort, lane, live);
                }
                // gate split: lane gi of a group holds gates [gi * NCG, (gi + 1) * NCG)
#pragma unroll
                for (int i = 0; i < TN; ++i)
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        if constexpr (GS == 1) acc[i][g] = part[i][g];
                        else if (g < NCG) acc[i][g] = part[i][g];
                        else acc[i][g] = __shfl_down_sync(0xffffffffu, part[i][g % NCG], g / NCG);
                    }
            }
            next_xw();

            auto epi = [&](auto fx) {
                constexpr bool FX = decltype(fx)::value;
                const Acts<OP, EXACT, FX> A{fA, gA, hA};
#pragma unroll
                for (int i = 0; i < TN; ++i) {
                    const int rl = x.rb * TN + i;
                    const int n = rown[i];
                    if (!(x.lead && rl < x.NR)) continue;
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
                            hn = A.F(clipv(p, pre[0]));
                        } else if constexpr (OP == 1) {
                            const float z = A.F(clipv(p, pre[0]));
                            const float r = A.F(clipv(p, pre[1]));
                            float ph;
                            if (p.has_B) ph = fadd(fadd(xc[i][2], fmul(r, fadd(acc[i][2], rbv[2]))), wb[2]);
                            else ph = fadd(xc[i][2], fmul(r, acc[i][2]));
                            const float ht = A.Gf(clipv(p, ph));
                            hn = fadd(fmul(fsub(1.0f, z), ht), fmul(z, hown[i]));
                        } else {
                            float pi = pre[0], po = pre[1], pf = pre[2];
                            const float pc = pre[3];
                            if (p.has_P) {
                                pi = fadd(pi, fmul(pI, cown[i]));
                                pf = fadd(pf, fmul(pF, cown[i]));
                            }
                            const float ig = A.F(clipv(p, pi));
                            const float fg = p.input_forget ? fsub(1.0f, ig) : A.F(clipv(p, pf));
                            const float ct = A.Gf(clipv(p, pc));
                            const float cn = fadd(fmul(fg, cown[i]), fmul(ig, ct));
                            if (p.has_P) po = fadd(po, fmul(pO, cn));
                            const float og = A.F(clipv(p, po));
                            hn = fmul(og, A.Hf(cn));
                            cown[i] = cn;
                        }
                        hown[i] = hn;
                        if (p.Y) io_store(p.Y, y_index(p, t, d, n, u), canon_nan(hn), p.io);
                    } else if (p.Y) {
                        io_store(p.Y, y_index(p, s, d, n, u), 0.f, p.io);
                    }
                    put_h(xoff(rl, u), hown[i]);
                }
            };
            if (fixed_acts) epi(std::true_type{});
            else epi(std::false_type{});
            if constexpr (CL) cl_publish(x, &s_hready[(s + 1) & 1], cl_send && !(skip_first && s == 0));
            else if (!publish(x, counter, &s_abort, skip_first && s == 0)) return;
        }
    }

#pragma unroll
    for (int i = 0; i < TN; ++i) {
        const int rl = x.rb * TN + i;
        const int n = rown[i];
        if (!(x.lead && rl < x.NR)) continue;
        const size_t si = s_index(p, d, n, u);
        if (p.Yh) io_store(p.Yh, si, len[i] > 0 ? canon_nan(hown[i]) : 0.f, p.io);
        if (OP == 2 && p.Yc) io_store(p.Yc, si, len[i] > 0 ? canon_nan(cown[i]) : 0.f, p.io);
    }
    if constexpr (CL) cluster_sync_all();
}

template <int OP, bool TWO>
const void* dataflow_kernel_ptr(int tn, bool exact)
{
    switch (tn * 2 + (exact ? 1 : 0)) {
    case 2: return (const void*)rnn_dataflow_kernel<OP, 1, false, TWO, 1, false>;
    case 3: return (const void*)rnn_dataflow_kernel<OP, 1, true, TWO, 1, false>;
    case 4: return (const void*)rnn_dataflow_kernel<OP, 2, false, TWO, 1, false>;
    case 5: return (const void*)rnn_dataflow_kernel<OP, 2, true, TWO, 1, false>;
    case 8: return (const void*)rnn_dataflow_kernel<OP, 4, false, TWO, 1, false>;
    case 9: return (const void*)rnn_dataflow_kernel<OP, 4, true, TWO, 1, false>;
    case 16: return (const void*)rnn_dataflow_kernel<OP, 8, false, TWO, 1, false>;
    case 17: return (const void*)rnn_dataflow_kernel<OP, 8, true, TWO, 1, false>;
    default: return nullptr;
    }
}

// gs > 1: the gate-split instance (GRU with linear_before_reset = 1, one
// row per thread, a gate column per lane)
template <int OP>
const void* dataflow_kernel_ptr(int tn, bool exact, bool two, int gs)
{
    if (gs != 1) {
        if constexpr (OP == 1) {
            if (gs != 3 || two || tn != 1) return nullptr;
            return exact ? (const void*)rnn_dataflow_kernel<OP, 1, true, false, 3, false>
                         : (const void*)rnn_dataflow_kernel<OP, 1, false, false, 3, false>;
        }
        return nullptr;
    }
    if constexpr (OP == 1) {
        if (two) return dataflow_kernel_ptr<OP, true>(tn, exact);
    }
    return dataflow_kernel_ptr<OP, false>(tn, exact);
}

template <int OP>
cudaError_t launch_dataflow_op(const RecParams& p, bool exact, int threads, size_t smem, cudaStream_t stream)
{
    const void* fn = dataflow_kernel_ptr<OP>(p.rows_per_thread, exact, OP == 1 && p.lbr == 0, p.gate_split);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    void* args[] = {(void*)&p};
    return cudaLaunchCooperativeKernel(fn, dim3(p.D * p.ctas_per_dir), dim3(threads), args, smem, stream);
}

template <int OP>
cudaError_t dataflow_occupancy_op(int tn, bool exact, bool two, int gs, int threads, size_t smem, int* blocks)
{
    const void* fn = dataflow_kernel_ptr<OP>(tn, exact, two, gs);
    if (!fn) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, fn, threads, smem);
}

// In-cluster exchange instances (one or two rows per thread), instantiated
// only by the translation units that launch them.
template <int OP>
const void* cluster_kernel_ptr(int tn, bool exact, bool two)
{
    if constexpr (OP == 1) {
        if (two) {
            if (tn == 1) return exact ? (const void*)rnn_dataflow_kernel<OP, 1, true, true, 1, true>
                                      : (const void*)rnn_dataflow_kernel<OP, 1, false, true, 1, true>;
            if (tn == 2) return exact ? (const void*)rnn_dataflow_kernel<OP, 2, true, true, 1, true>
                                      : (const void*)rnn_dataflow_kernel<OP, 2, false, true, 1, true>;
            return nullptr;
        }
    }
    if (tn == 1) return exact ? (const void*)rnn_dataflow_kernel<OP, 1, true, false, 1, true>
                              : (const void*)rnn_dataflow_kernel<OP, 1, false, false, 1, true>;
    if (tn == 2) return exact ? (const void*)rnn_dataflow_kernel<OP, 2, true, false, 1, true>
                              : (const void*)rnn_dataflow_kernel<OP, 2, false, false, 1, true>;
    return nullptr;
}

// Launch configuration of the in-cluster kernel: clusters of unit_groups CTAs
// (above 8 the non-portable sizes, up to 16).
template <int OP>
cudaError_t cluster_config(const void* fn, int ctas, int cluster, int threads, size_t smem, cudaStream_t stream,
                           cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr)
{
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (cluster > 8) {
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3((unsigned)ctas);
    cfg->blockDim = dim3((unsigned)threads);
    cfg->dynamicSmemBytes = smem;
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg->attrs = attr;
    cfg->numAttrs = 1;
    return cudaSuccess;
}

template <int OP>
cudaError_t launch_cluster_op(const RecParams& p, bool exact, int threads, size_t smem, cudaStream_t stream)
{
    const void* fn = cluster_kernel_ptr<OP>(p.rows_per_thread, exact, OP == 1 && p.lbr == 0);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    cudaError_t e = cluster_config<OP>(fn, p.D * p.ctas_per_dir, p.unit_groups, threads, smem, stream, &cfg, attr);
    if (e != cudaSuccess) return e;
    void* args[] = {(void*)&p};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

// Clusters of the launch that fit on the device at once (0: none fits).
template <int OP>
cudaError_t cluster_occupancy_op(int tn, bool exact, bool two, int ctas, int cluster, int threads, size_t smem,
                                 int* clusters)
{
    const void* fn = cluster_kernel_ptr<OP>(tn, exact, two);
    if (!fn) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    cudaError_t e = cluster_config<OP>(fn, ctas, cluster, threads, smem, nullptr, &cfg, attr);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveClusters(clusters, fn, &cfg);
}

}  // namespace rnngb
