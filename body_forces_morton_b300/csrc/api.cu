// C ABI of the FMM library: plan life cycle, the evaluation pipeline, the
// kick-drift-kick step, statistics and inspection exports.
//
// An evaluation runs in two phases on the caller's stream, with no host wait
// between them:
//   phase 1  root box, keys, radix sort (+ gather), octree levels (the tree
//            kernel records the node count and depth on the device);
//   phase 2  upward pass, dual-tree walk (until its frontier is empty), lists,
//            M2L, L2L (ordered by level), L2P + P2P + scatter, every kernel
//            reading the node count and depth on the device;
//   then one read-back of the small status block.
// Capacities of the node, frontier and pair buffers are estimates; a kernel
// that would exceed one skips the write and sets a bit in the status word, and
// the evaluation is repeated with larger buffers.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/fmm.h"
#include "plan.h"

using namespace bfm;

struct fmm_plan {
    Plan P;
};

namespace {

thread_local std::string g_err;

void set_err(const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
}

#define CUDA_TRY(call)                                                                         \
    do {                                                                                       \
        cudaError_t e_ = (call);                                                               \
        if (e_ != cudaSuccess) {                                                               \
            set_err("%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__, __LINE__); \
            return e_ == cudaErrorMemoryAllocation ? FMM_ERR_OOM : FMM_ERR_CUDA;               \
        }                                                                                      \
    } while (0)

template <class X> cudaError_t dalloc(X *&p, size_t count)
{
    p = nullptr;
    if (count == 0) count = 1;
    return cudaMalloc((void **)&p, count * sizeof(X));
}

void dfree(void *p)
{
    if (p) cudaFree(p);
}

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) cudaSetDevice(dev);
        else prev = -1;
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

constexpr int RS_TILE = 2048;  // the radix sort's smallest tile (flags per pass: tiles x 256 digits)

void free_nodes(Plan &P)
{
    int **ints[] = {&P.node_first, &P.node_count, &P.node_child0, &P.node_nchild, &P.node_parent,
                    &P.node_level, &P.node_done,  &P.m2l_cnt,     &P.p2p_cnt,     &P.m2l_off,
                    &P.p2p_off,    &P.long_seg,    &P.order,       &P.p2p_done};
    for (int **q : ints) { dfree(*q); *q = nullptr; }
    void **vs[] = {&P.node_lo, &P.node_hi, &P.node_c, &P.node_l, &P.node_w, &P.M, &P.Lm2l, &P.L, &P.Mr};
    for (void **q : vs) { dfree(*q); *q = nullptr; }
    dfree(P.flags);
    P.flags = nullptr;
    dfree(P.order_key);
    P.order_key = nullptr;
    dfree(P.p2p_items);
    P.p2p_items = nullptr;
    dfree(P.p2p_nch);
    P.p2p_nch = nullptr;
    dfree(P.node_flag);
    P.node_flag = nullptr;
}

void free_lists(Plan &P)
{
    dfree(P.frontier[0]); dfree(P.frontier[1]);
    dfree(P.m2l_pairs); dfree(P.p2p_pairs); dfree(P.m2l_src); dfree(P.p2p_src);
    P.frontier[0] = P.frontier[1] = nullptr;
    P.m2l_pairs = P.p2p_pairs = nullptr;
    P.m2l_src = P.p2p_src = nullptr;
}

// Node indices are int32 on the device and some node arrays hold two entries
// per node, so the node capacity stays at or below 2^30.
constexpr int64_t kMaxNodeCap = int64_t(1) << 30;

fmm_status alloc_nodes(Plan &P, int64_t cap)
{
    if (cap > kMaxNodeCap) {
        set_err("fmm_eval: the tree needs more than 2^30 nodes");
        return FMM_ERR_CAPACITY;
    }
    free_nodes(P);
    P.cap_nodes = cap;
    const size_t c = (size_t)cap, e = (size_t)P.esize;
    CUDA_TRY(dalloc(P.node_first, c));
    CUDA_TRY(dalloc(P.node_count, c));
    CUDA_TRY(dalloc(P.node_child0, c));
    CUDA_TRY(dalloc(P.node_nchild, c));
    CUDA_TRY(dalloc(P.node_parent, c));
    CUDA_TRY(dalloc(P.node_level, c));
    CUDA_TRY(dalloc(P.node_done, c));
    CUDA_TRY(dalloc(P.m2l_cnt, c));
    CUDA_TRY(dalloc(P.p2p_cnt, c));
    CUDA_TRY(dalloc(P.m2l_off, c + 1));
    CUDA_TRY(dalloc(P.p2p_off, c + 1));
    CUDA_TRY(dalloc(P.long_seg, 2 * c));
    CUDA_TRY(dalloc(P.order, 2 * c));
    CUDA_TRY(dalloc(P.p2p_items, 2 * c));
    CUDA_TRY(dalloc(P.p2p_done, c));
    CUDA_TRY(dalloc(P.p2p_nch, c));
    CUDA_TRY(dalloc(P.node_flag, c));
    CUDA_TRY(cudaMemset(P.node_flag, 0, c * sizeof(unsigned)));
    P.flag_seq = 0;
    CUDA_TRY(dalloc(P.order_key, 2 * c));
    CUDA_TRY(cudaMalloc(&P.node_lo, 3 * c * e));
    CUDA_TRY(cudaMalloc(&P.node_hi, 3 * c * e));
    CUDA_TRY(cudaMalloc(&P.node_c, 4 * c * e));
    CUDA_TRY(cudaMalloc(&P.node_l, 4 * c * e));
    CUDA_TRY(cudaMalloc(&P.node_w, 8 * c * e));
    CUDA_TRY(cudaMalloc(&P.M, (size_t)P.ncp * c * e));
    CUDA_TRY(cudaMalloc(&P.Lm2l, (size_t)P.ncp * c * e));
    CUDA_TRY(cudaMalloc(&P.L, (size_t)P.ncp * c * e));
    CUDA_TRY(cudaMalloc(&P.Mr, (size_t)P.nrp * c * 8));
    CUDA_TRY(cudaMemset(P.m2l_cnt, 0, c * sizeof(int)));
    CUDA_TRY(cudaMemset(P.p2p_cnt, 0, c * sizeof(int)));
    const int64_t tiles_sort = (P.n + RS_TILE - 1) / RS_TILE;
    P.cap_flags = std::max<int64_t>({tiles_sort * 256, cap / 32 + 64, 2 * (cap / 1024) + 64});
    CUDA_TRY(dalloc(P.flags, (size_t)P.cap_flags));
    CUDA_TRY(cudaMemset(P.flags, 0, (size_t)P.cap_flags * sizeof(unsigned long long)));
    P.epoch = 0;
    return FMM_OK;
}

fmm_status alloc_lists(Plan &P, int64_t cap_frontier, int64_t cap_m2l, int64_t cap_p2p)
{
    free_lists(P);
    auto round_up = [](int64_t v) { return (v + kShards - 1) / kShards * kShards; };
    // every shard holds at least one walk tile's worst output: 256 pairs of up to 36 child pairs
    // (a self pair of 8 children) for the frontier, one M2L or P2P pair each for the lists
    // (not under BFM_FMM_FAULT=capacity, which starts every buffer small to exercise regrowth)
    const int64_t ff = P.minimal_caps ? 1 : 36, fl = P.minimal_caps ? 1 : 256;
    cap_frontier = round_up(std::max<int64_t>(cap_frontier, (int64_t)kShards * fl * ff));
    cap_m2l = round_up(std::max<int64_t>(cap_m2l, (int64_t)kShards * fl));
    cap_p2p = round_up(std::max<int64_t>(cap_p2p, (int64_t)kShards * fl));
    P.cap_frontier = cap_frontier;
    P.cap_m2l = cap_m2l;
    P.cap_p2p = cap_p2p;
    CUDA_TRY(dalloc(P.frontier[0], (size_t)cap_frontier));
    CUDA_TRY(dalloc(P.frontier[1], (size_t)cap_frontier));
    CUDA_TRY(dalloc(P.m2l_pairs, (size_t)cap_m2l));
    CUDA_TRY(dalloc(P.p2p_pairs, (size_t)cap_p2p));
    CUDA_TRY(dalloc(P.m2l_src, 2 * (size_t)cap_m2l));
    CUDA_TRY(dalloc(P.p2p_src, 2 * (size_t)cap_p2p));
    return FMM_OK;
}

void free_mutual(Plan &P)
{
    dfree(P.mut_lo); dfree(P.mut_mir_m2l); dfree(P.mut_mir_p2p); dfree(P.mut_base);
    dfree(P.mut_rm2l); dfree(P.mut_lpart); dfree(P.mut_rp2p); dfree(P.mut_own);
    P.mut_lo = P.mut_mir_m2l = P.mut_mir_p2p = nullptr;
    P.mut_base = nullptr;
    P.mut_rm2l = P.mut_lpart = P.mut_rp2p = P.mut_own = nullptr;
    P.mut_for_nodes = 0;
    P.mut_cap_rp = P.mut_cap_em = P.mut_cap_ep = 0;
}

// Buffers of the mutual evaluation. Their sizes follow the lists the walk
// produces, so they are not taken from the list capacities (which grow like
// theta^-3 and can reach 1e9 pairs): they start at estimates (32 partner sums
// per particle, 128 M2L and 48 P2P entries per node, or 1 under
// BFM_FMM_FAULT=capacity), a kernel compares them with the actual sizes, and
// an evaluation that finds one short grows it and repeats. A size <= 0 asks
// for the estimate.
fmm_status ensure_mutual(Plan &P, long long want_rp, long long want_em, long long want_ep)
{
    const size_t e = (size_t)P.esize;
    if (P.mut_for_nodes != P.cap_nodes) {
        dfree(P.mut_lo); dfree(P.mut_base); dfree(P.mut_lpart);
        P.mut_lo = nullptr; P.mut_base = nullptr; P.mut_lpart = nullptr;
        const size_t c = (size_t)P.cap_nodes;
        CUDA_TRY(dalloc(P.mut_lo, 3 * c));
        CUDA_TRY(dalloc(P.mut_base, c + 1));
        CUDA_TRY(cudaMalloc(&P.mut_lpart, (size_t)P.nrp * c * e));
        P.mut_for_nodes = P.cap_nodes;
    }
    if (!P.mut_own) CUDA_TRY(cudaMalloc(&P.mut_own, 4 * (size_t)P.n * e));
    const bool m = P.minimal_caps;
    if (want_rp <= 0) want_rp = m ? 1 : std::max<long long>(32 * (long long)P.n, 65536);
    if (want_em <= 0) want_em = m ? 1 : std::min<long long>(2 * P.cap_m2l, 128 * P.cap_nodes);
    if (want_ep <= 0) want_ep = m ? 1 : std::min<long long>(2 * P.cap_p2p, 48 * P.cap_nodes);
    if (!P.mut_rp2p || P.mut_cap_rp < want_rp) {
        dfree(P.mut_rp2p);
        P.mut_rp2p = nullptr;
        P.mut_cap_rp = 0;
        CUDA_TRY(cudaMalloc(&P.mut_rp2p, 4 * (size_t)want_rp * e));
        P.mut_cap_rp = want_rp;
    }
    if (!P.mut_rm2l || P.mut_cap_em < want_em) {
        dfree(P.mut_rm2l); dfree(P.mut_mir_m2l);
        P.mut_rm2l = nullptr; P.mut_mir_m2l = nullptr;
        P.mut_cap_em = 0;
        CUDA_TRY(dalloc(P.mut_mir_m2l, (size_t)want_em));
        CUDA_TRY(cudaMalloc(&P.mut_rm2l, (size_t)P.nrp * (size_t)want_em * e));
        P.mut_cap_em = want_em;
    }
    if (!P.mut_mir_p2p || P.mut_cap_ep < want_ep) {
        dfree(P.mut_mir_p2p);
        P.mut_mir_p2p = nullptr;
        P.mut_cap_ep = 0;
        CUDA_TRY(dalloc(P.mut_mir_p2p, (size_t)want_ep));
        P.mut_cap_ep = want_ep;
    }
    return FMM_OK;
}

void destroy_plan(Plan &P)
{
    free_nodes(P);
    free_lists(P);
    dfree(P.keys[0]); dfree(P.keys[1]); dfree(P.idx[0]); dfree(P.idx[1]);
    dfree(P.xyzm); dfree(P.far); dfree(P.div); dfree(P.vwin); dfree(P.leaf_of); dfree(P.tree_cc); dfree(P.rel); dfree(P.scratch); dfree(P.ctr); dfree(P.gbar); dfree(P.sort_cnt); dfree(P.sort_big);
    dfree(P.h_pos); dfree(P.h_mass); dfree(P.h_acc); dfree(P.h_pot); dfree(P.acc_cache);
    dfree(P.vjp_acc); dfree(P.vjp_src); dfree(P.Ms); dfree(P.Lsm); dfree(P.Ls);
    free_mutual(P);
    if (P.ctr_host) cudaFreeHost(P.ctr_host);
    for (int i = 0; i < kNumEvents; ++i)
        if (P.ev[i]) cudaEventDestroy(P.ev[i]);
    if (P.ev_done) cudaEventDestroy(P.ev_done);
    if (P.ev_pos) cudaEventDestroy(P.ev_pos);
    if (P.ev_mass) cudaEventDestroy(P.ev_mass);
    if (P.side) cudaStreamDestroy(P.side);
}

// Pair capacities stay at or below 1e9 unordered pairs, so the directed list
// entries (two per pair) index int32 CSR offsets without wrapping; a walk that
// needs more ends in FMM_ERR_CAPACITY after the retries.
int64_t clamp_cap(double v) { return (int64_t)std::min(v, 1.0e9); }

// Node-count and list estimates; the evaluation grows them when exceeded.
int64_t node_estimate(const Plan &P) { return std::min(kMaxNodeCap, std::max<int64_t>(4096, 6 * P.n / P.leaf + 1024)); }

void record(Plan &P, int k, cudaStream_t s) { cudaEventRecord(P.ev[k], s); }

const char *error_bits(unsigned e)
{
    static thread_local char buf[160];
    snprintf(buf, sizeof(buf), "%s%s%s%s%s%s%s%s%s", e & ERR_NONFINITE ? "nonfinite " : "", e & ERR_NODES ? "nodes " : "",
             e & ERR_FRONTIER ? "frontier " : "", e & ERR_M2L_CAP ? "m2l " : "", e & ERR_P2P_CAP ? "p2p " : "",
             e & ERR_SPIN ? "spin-limit " : "", e & ERR_BOUNDS ? "bounds " : "", e & ERR_WALK ? "walk " : "",
             e & ERR_MUT_CAP ? "mutual-buffer " : "");
    return buf;
}

// Wait for the stream by polling an event: the calls block anyway, and a busy
// wait returns as soon as the work is done instead of after the scheduler
// wakes a sleeping thread.
fmm_status wait_stream(Plan &P, cudaStream_t s)
{
    CUDA_TRY(cudaEventRecord(P.ev_done, s));
    cudaError_t e;
    while ((e = cudaEventQuery(P.ev_done)) == cudaErrorNotReady) {
    }
    CUDA_TRY(e);
    return FMM_OK;
}

// Copy the status block back and wait for it.
fmm_status sync_counters(Plan &P, cudaStream_t s)
{
    CUDA_TRY(cudaGetLastError());
    CUDA_TRY(cudaMemcpyAsync(P.ctr_host, P.ctr, sizeof(DevCounters), cudaMemcpyDeviceToHost, s));
    return wait_stream(P, s);
}

fmm_status eval_device(Plan &P, const void *pos, const void *mass, void *acc, void *pot, cudaStream_t s)
{
    if (!pos || !mass || !acc) {
        set_err("fmm_eval: pos, mass and acc_out must be non-NULL device pointers");
        return FMM_ERR_INVALID_ARG;
    }
    P.retries = 0;
    // each attempt that finds a buffer short grows it and repeats; from minimal buffers the node, frontier,
    // list and mutual-evaluation buffers can each take a regrowth or two
    for (int attempt = 0; attempt < 12; ++attempt) {
        P.slot = 0;
        P.launches = 0;
        if (P.mutual) {
            fmm_status sm = ensure_mutual(P, 0, 0, 0);
            if (sm) return sm;
        }
        if (P.epoch > (1u << 24) - 512) {
            CUDA_TRY(cudaMemsetAsync(P.flags, 0, (size_t)P.cap_flags * sizeof(unsigned long long), s));
            P.epoch = 0;
        }
        // ---- phase 1: box, keys, sort, tree (the tree kernel records the node count and depth)
        record(P, 0, s);
        CUDA_TRY(cudaMemsetAsync(P.ctr, 0, sizeof(DevCounters), s));
        CUDA_TRY(cudaMemsetAsync(P.gbar, 0, 3 * sizeof(GridBarrier), s));
        P.launches += launch_keys(P, pos, s);
        record(P, 1, s);
        P.launches += launch_sort(P, pos, mass, s);
        record(P, 2, s);
        P.launches += launch_tree(P, s);
        record(P, 3, s);
        // ---- phase 2, launched without waiting: every kernel reads the node count (and the walk
        // and L2L their extent) on the device, and skips the tree if its build failed
        record(P, 4, s);
        P.launches += launch_upward(P, s);
        record(P, 5, s);
        P.launches += launch_walk(P, 0, s);
        record(P, 6, s);
        P.launches += launch_lists(P, s);
        record(P, 7, s);
        P.launches += launch_m2l(P, s);
        record(P, 8, s);
        P.launches += launch_l2l(P, 0, s);
        record(P, 9, s);
        P.launches += launch_l2p(P, s);
        record(P, 11, s);
        P.launches += launch_p2p(P, acc, pot, s);
        record(P, 10, s);
        fmm_status st = sync_counters(P, s);
        if (st) return st;
        const DevCounters &h = *P.ctr_host;
        if (h.error & ERR_NONFINITE) {
            set_err("fmm_eval: a position is not finite");
            return FMM_ERR_NONFINITE;
        }
        if (h.error & ERR_NODES) {
            // double, up to the cap; a full-size tree that still overflows reports FMM_ERR_CAPACITY
            st = alloc_nodes(P, P.cap_nodes >= kMaxNodeCap ? 2 * P.cap_nodes : std::min(2 * P.cap_nodes, kMaxNodeCap));
            if (st) return st;
            P.retries++;
            continue;
        }
        // the next evaluation's sort: all 8 digits when long runs of equal high words held many keys here
        P.sort_full = P.sort_full || (int64_t)h.sort_long_keys * 64 > P.n;
        P.depth = h.depth;
        P.n_nodes = h.n_nodes;
        const unsigned cap_bits = ERR_FRONTIER | ERR_M2L_CAP | ERR_P2P_CAP;
        if (h.error & cap_bits) {
            // sharded lists: grow to 1.5x the fullest shard (or double), times the shard count
            int64_t cf = P.cap_frontier, cm = P.cap_m2l, cp = P.cap_p2p;
            int mmax = 0, pmax = 0;
            for (int s2 = 0; s2 < kShards; ++s2) {
                mmax = std::max(mmax, h.n_m2l_pairs[s2]);
                pmax = std::max(pmax, h.n_p2p_pairs[s2]);
            }
            if (h.error & ERR_FRONTIER) cf = clamp_cap(std::max(2.0 * cf, 1.5 * kShards * (double)h.frontier_max));
            if (h.error & ERR_M2L_CAP) cm = clamp_cap(std::max(2.0 * cm, 1.5 * kShards * (double)mmax));
            if (h.error & ERR_P2P_CAP) cp = clamp_cap(std::max(2.0 * cp, 1.5 * kShards * (double)pmax));
            st = alloc_lists(P, cf, cm, cp);
            if (st) return st;
            P.retries++;
            continue;
        }
        if (h.error & ERR_MUT_CAP) {
            // a mutual-evaluation buffer was short (its writes were skipped): grow it and repeat
            auto grow = [](long long need) { return need > 0 ? need + need / 4 + 1024 : 0; };
            st = ensure_mutual(P, grow(h.mut_need[0]), grow(h.mut_need[1]), grow(h.mut_need[2]));
            if (st) return st;
            P.retries++;
            continue;
        }
        if (h.error) {
            set_err("fmm_eval: device check failed: %s", error_bits(h.error));
            return FMM_ERR_INTERNAL;
        }
        int64_t m2l_pairs = 0, p2p_pairs = 0;
        for (int s2 = 0; s2 < kShards; ++s2) {
            m2l_pairs += h.n_m2l_pairs[s2];
            p2p_pairs += h.n_p2p_pairs[s2];
        }
        P.n_m2l = 2 * m2l_pairs;
        P.n_p2p_pairs = p2p_pairs;
        P.walk_pairs = h.walk_pairs;
        P.p2p_inter = h.p2p_interactions;
        P.have_eval = true;
        return FMM_OK;
    }
    set_err("fmm_eval: interaction buffers still overflow after %d regrowths", P.retries);
    return FMM_ERR_CAPACITY;
}

}  // namespace

// Node flags (upward pass, L2L) hold the number of the pass that completed the
// node; each pass waits for its own number, so flags left by earlier passes
// need no clearing until the numbers wrap.
unsigned bfm::Plan::next_flag_seq(cudaStream_t s)
{
    if (++flag_seq > 0x7fffffffu) {
        cudaMemsetAsync(node_flag, 0, (size_t)cap_nodes * sizeof(unsigned), s);
        flag_seq = 1;
    }
    return flag_seq;
}

unsigned bfm::Plan::next_epoch()
{
    epoch = (epoch + 1) & 0xffffffu;
    if (epoch == 0) epoch = 1;
    return epoch;
}

extern "C" {

fmm_plan *fmm_plan_create(int64_t n, int p, double theta, int leaf, fmm_dtype dtype)
{
    g_err.clear();
    if (n < 1 || n > (int64_t(1) << 30)) { set_err("fmm_plan_create: n must be in [1, 2^30]"); return nullptr; }
    if (p < 0 || p > kMaxP) { set_err("fmm_plan_create: p must be in [0, 8]"); return nullptr; }
    if (!(theta > 0.0) || theta > 1.0) { set_err("fmm_plan_create: theta must be in (0, 1]"); return nullptr; }
    if (leaf < 1) { set_err("fmm_plan_create: leaf must be >= 1"); return nullptr; }
    if (dtype != FMM_F32 && dtype != FMM_F64) { set_err("fmm_plan_create: unknown dtype"); return nullptr; }
    // Host-side fault injection for tests (no GPU fault is ever provoked):
    //   BFM_FMM_FAULT=alloc     creation fails as if a device allocation had failed;
    //   BFM_FMM_FAULT=capacity  buffers start minimal, so evaluations exercise the regrowth path;
    //   BFM_FMM_FAULT=spin      every L2L wait on a parent runs out its bound (a flag value that no
    //                           pass stores), so evaluations report the expired wait (FMM_ERR_INTERNAL).
    const char *fault = getenv("BFM_FMM_FAULT");
    if (fault && strcmp(fault, "alloc") == 0) {
        set_err("fmm_plan_create: device allocation failed (injected by BFM_FMM_FAULT=alloc)");
        return nullptr;
    }
    const bool minimal = fault && strcmp(fault, "capacity") == 0;
    fmm_plan *h = new (std::nothrow) fmm_plan();
    if (!h) { set_err("fmm_plan_create: out of host memory"); return nullptr; }
    Plan &P = h->P;
    P.n = n; P.p = p; P.theta = theta; P.leaf = leaf; P.dtype = (int)dtype;
    P.minimal_caps = minimal;
    P.fault_spin = fault && strcmp(fault, "spin") == 0;
    P.esize = dtype == FMM_F32 ? 4 : 8;
    P.nc = (p + 1) * (p + 2) * (p + 3) / 6;
    P.ncp = (P.nc + 3) / 4 * 4;
    P.nrc = (p + 1) * (p + 1);
    P.nrp = (P.nrc + 3) / 4 * 4;
    auto fail = [&](fmm_status) -> fmm_plan * {
        destroy_plan(P);
        delete h;
        return nullptr;
    };
    auto ok = [&](cudaError_t e, const char *what) {
        if (e != cudaSuccess) set_err("fmm_plan_create: %s: %s", what, cudaGetErrorString(e));
        return e == cudaSuccess;
    };
    if (!ok(cudaGetDevice(&P.device), "cudaGetDevice")) return fail(FMM_ERR_CUDA);
    if (!ok(cudaDeviceGetAttribute(&P.num_sms, cudaDevAttrMultiProcessorCount, P.device), "SM count"))
        return fail(FMM_ERR_CUDA);
    {
        int coop = 0;
        if (!ok(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, P.device), "cooperative launch"))
            return fail(FMM_ERR_CUDA);
        if (!coop) {
            set_err("fmm_plan_create: the device does not support cooperative launches");
            return fail(FMM_ERR_CUDA);
        }
        // co-resident blocks for the cooperative tree build: up to 4 per SM
        // (grid barriers take up to 2048 blocks)
        P.coop_blocks_tree = std::min(2048, P.num_sms * std::max(1, std::min(4, tree_max_blocks_per_sm())));
        // walk: 8 blocks per SM from N = 2^19 on (large frontiers), 4 below (measured: the smaller grid
        // syncs faster between the small generations of small trees)
        const int wb = n >= (1 << 19) ? 8 : 4;
        P.coop_blocks_walk = std::min(2048, P.num_sms * std::max(1, std::min(wb, walk_max_blocks_per_sm(P.dtype))));
        // the cooperative radix sort runs when all its tiles are co-resident (grid barriers take up to 2048)
        sort_coop_capacity(P.num_sms, P.coop_tiles_sort);
        P.coop_tiles_sort[0] = std::min(2048, P.coop_tiles_sort[0]);
        P.coop_tiles_sort[1] = std::min(2048, P.coop_tiles_sort[1]);
        P.sort_cnt_cap = (size_t)256 * std::max(1, std::max(P.coop_tiles_sort[0], P.coop_tiles_sort[1]));
    }
    const size_t nn = (size_t)n, e = (size_t)P.esize;
    P.sort_big_cap = nn / 33 + 1;  // runs of over 32 keys
    if (!ok(dalloc(P.keys[0], nn), "keys") || !ok(dalloc(P.keys[1], nn), "keys") ||
        !ok(dalloc(P.idx[0], nn), "perm") || !ok(dalloc(P.idx[1], nn), "perm") ||
        !ok(cudaMalloc(&P.xyzm, 4 * nn * e), "particles") || !ok(cudaMalloc(&P.far, 4 * nn * e), "far field") || !ok(dalloc(P.div, nn), "divergence") ||
        !ok(dalloc(P.vwin, nn), "tree windows") || !ok(dalloc(P.leaf_of, nn), "particle leaves") || !ok(dalloc(P.tree_cc, tree_cc_ints(n)), "tree counts") ||
        (P.dtype == 1 && !ok(cudaMalloc(&P.rel, 2 * nn * sizeof(float4)), "leaf-relative particles")) ||
        !ok(cudaMalloc(&P.scratch, 65536), "scratch") || !ok(dalloc(P.ctr, 1), "counters") ||
        !ok(dalloc(P.gbar, 3), "grid barriers") ||
        !ok(dalloc(P.sort_cnt, P.sort_cnt_cap), "sort counts") ||
        !ok(dalloc(P.sort_big, P.sort_big_cap), "sort runs") ||
        !ok(cudaMallocHost((void **)&P.ctr_host, sizeof(DevCounters)), "pinned counters"))
        return fail(FMM_ERR_OOM);
    for (int i = 0; i < kNumEvents; ++i)
        if (!ok(cudaEventCreate(&P.ev[i]), "events")) return fail(FMM_ERR_CUDA);
    if (!ok(cudaEventCreateWithFlags(&P.ev_done, cudaEventDisableTiming), "events")) return fail(FMM_ERR_CUDA);
    const int64_t cap = minimal ? 1024 : node_estimate(P);
    if (alloc_nodes(P, cap) != FMM_OK) return fail(FMM_ERR_OOM);
    // list sizes per node grow like theta^-3 (the pairs a node meets before acceptance); sized for the
    // clustered and Plummer workloads with room to spare, so that evaluations rarely regrow
    const double lf = (minimal ? 1.0 / 16 : 1.0) * std::max(1.0, std::pow(0.7 / theta, 3.0));
    if (alloc_lists(P, clamp_cap(32.0 * lf * cap), clamp_cap(64.0 * lf * cap), clamp_cap(24.0 * lf * cap)) != FMM_OK)
        return fail(FMM_ERR_OOM);
    return h;
}

fmm_status fmm_eval(fmm_plan *plan, const void *pos, const void *mass, void *acc_out, void *pot_out, void *stream)
{
    g_err.clear();
    if (!plan) { set_err("fmm_eval: NULL plan"); return FMM_ERR_INVALID_ARG; }
    DeviceGuard g(plan->P.device);
    plan->P.cache_valid = false;
    return eval_device(plan->P, pos, mass, acc_out, pot_out, (cudaStream_t)stream);
}

fmm_status fmm_eval_host(fmm_plan *plan, const void *pos, const void *mass, void *acc_out, void *pot_out,
                         void *stream)
{
    g_err.clear();
    if (!plan || !pos || !mass || !acc_out) {
        set_err("fmm_eval_host: plan, pos, mass and acc_out must be non-NULL");
        return FMM_ERR_INVALID_ARG;
    }
    Plan &P = plan->P;
    DeviceGuard g(P.device);
    cudaStream_t s = (cudaStream_t)stream;
    const size_t e = (size_t)P.esize, n = (size_t)P.n;
    if (!P.h_pos) {
        CUDA_TRY(cudaMalloc(&P.h_pos, 3 * n * e));
        CUDA_TRY(cudaMalloc(&P.h_mass, n * e));
        CUDA_TRY(cudaMalloc(&P.h_acc, 3 * n * e));
        CUDA_TRY(cudaMalloc(&P.h_pot, n * e));
    }
    if (!P.side) {
        CUDA_TRY(cudaStreamCreateWithFlags(&P.side, cudaStreamNonBlocking));
        CUDA_TRY(cudaEventCreateWithFlags(&P.ev_pos, cudaEventDisableTiming));
        CUDA_TRY(cudaEventCreateWithFlags(&P.ev_mass, cudaEventDisableTiming));
    }
    P.cache_valid = false;
    // positions first, at the full link rate; the masses follow on the side stream, after the positions
    // (so that the two copies do not share the link), while the box, the keys and the radix passes run
    CUDA_TRY(cudaMemcpyAsync(P.h_pos, pos, 3 * n * e, cudaMemcpyHostToDevice, s));
    CUDA_TRY(cudaEventRecord(P.ev_pos, s));
    CUDA_TRY(cudaStreamWaitEvent(P.side, P.ev_pos, 0));
    CUDA_TRY(cudaMemcpyAsync(P.h_mass, mass, n * e, cudaMemcpyHostToDevice, P.side));
    CUDA_TRY(cudaEventRecord(P.ev_mass, P.side));
    P.mass_wait = P.ev_mass;
    fmm_status st = eval_device(P, P.h_pos, P.h_mass, P.h_acc, pot_out ? P.h_pot : nullptr, s);
    P.mass_wait = nullptr;
    if (st) {
        cudaStreamSynchronize(P.side);  // the copy into the plan's buffer ends before the call returns
        return st;
    }
    CUDA_TRY(cudaMemcpyAsync(acc_out, P.h_acc, 3 * n * e, cudaMemcpyDeviceToHost, s));
    if (pot_out) CUDA_TRY(cudaMemcpyAsync(pot_out, P.h_pot, n * e, cudaMemcpyDeviceToHost, s));
    if (fmm_status w = wait_stream(P, s)) return w;
    return FMM_OK;
}

fmm_status fmm_kdk_step(fmm_plan *plan, void *pos, void *vel, const void *mass, double dt, void *stream)
{
    g_err.clear();
    if (!plan || !pos || !vel || !mass) {
        set_err("fmm_kdk_step: plan, pos, vel and mass must be non-NULL");
        return FMM_ERR_INVALID_ARG;
    }
    Plan &P = plan->P;
    DeviceGuard g(P.device);
    cudaStream_t s = (cudaStream_t)stream;
    if (!P.acc_cache) CUDA_TRY(cudaMalloc(&P.acc_cache, 3 * (size_t)P.n * P.esize));
    const bool cached = P.cache_valid && P.cache_pos == pos && P.cache_vel == vel && P.cache_mass == mass;
    P.cache_valid = false;
    int kdk_launches = 0;
    if (!cached) {
        fmm_status st = eval_device(P, pos, mass, P.acc_cache, nullptr, s);
        if (st) return st;
        kdk_launches += P.launches;
    }
    kdk_launches += launch_kick(P, vel, P.acc_cache, 0.5 * dt, s);
    kdk_launches += launch_drift(P, pos, vel, dt, s);
    fmm_status st = eval_device(P, pos, mass, P.acc_cache, nullptr, s);
    if (st) return st;
    kdk_launches += P.launches;
    kdk_launches += launch_kick(P, vel, P.acc_cache, 0.5 * dt, s);
    CUDA_TRY(cudaGetLastError());
    if (fmm_status w = wait_stream(P, s)) return w;
    P.launches = kdk_launches;
    P.cache_valid = true;
    P.cache_pos = pos;
    P.cache_vel = vel;
    P.cache_mass = mass;
    return FMM_OK;
}

fmm_status fmm_kdk_step_lattice(fmm_plan *plan, void *pos, void *vel, const void *mass, double dt, int pos_exp,
                                int vel_exp, void *stream)
{
    g_err.clear();
    if (!plan || !pos || !vel || !mass) {
        set_err("fmm_kdk_step_lattice: plan, pos, vel and mass must be non-NULL");
        return FMM_ERR_INVALID_ARG;
    }
    Plan &P = plan->P;
    if (pos_exp < -1000 || pos_exp > 100 || vel_exp < -1000 || vel_exp > 100) {
        set_err("fmm_kdk_step_lattice: lattice exponents out of range");
        return FMM_ERR_INVALID_ARG;
    }
    DeviceGuard g(P.device);
    cudaStream_t s = (cudaStream_t)stream;
    if (!P.acc_cache) CUDA_TRY(cudaMalloc(&P.acc_cache, 3 * (size_t)P.n * P.esize));
    const bool cached = P.cache_valid && P.cache_pos == pos && P.cache_vel == vel && P.cache_mass == mass;
    P.cache_valid = false;
    int launches = 0;
    // put the state on its lattices (a no-op once it lies there): x += 0, v += 0 rounded
    launches += launch_lattice_axpy(P, pos, nullptr, 0.0, pos_exp, pos_exp, s);
    launches += launch_lattice_axpy(P, vel, nullptr, 0.0, vel_exp, vel_exp, s);
    if (!cached) {
        fmm_status st = eval_device(P, pos, mass, P.acc_cache, nullptr, s);
        if (st) return st;
        launches += P.launches;
    }
    launches += launch_lattice_axpy(P, vel, P.acc_cache, 0.5 * dt, vel_exp, vel_exp, s);
    launches += launch_lattice_axpy(P, pos, vel, dt, pos_exp, pos_exp, s);
    fmm_status st = eval_device(P, pos, mass, P.acc_cache, nullptr, s);
    if (st) return st;
    launches += P.launches;
    launches += launch_lattice_axpy(P, vel, P.acc_cache, 0.5 * dt, vel_exp, vel_exp, s);
    CUDA_TRY(cudaGetLastError());
    if (fmm_status w = wait_stream(P, s)) return w;
    P.launches = launches;
    P.cache_valid = true;
    P.cache_pos = pos;
    P.cache_vel = vel;
    P.cache_mass = mass;
    return FMM_OK;
}

void fmm_kdk_reset(fmm_plan *plan)
{
    if (plan) plan->P.cache_valid = false;
}

fmm_status fmm_plan_set_f64_ieee(fmm_plan *plan, int on)
{
    g_err.clear();
    if (!plan) { set_err("fmm_plan_set_f64_ieee: NULL plan"); return FMM_ERR_INVALID_ARG; }
    if (plan->P.dtype != FMM_F64 && on) {
        set_err("fmm_plan_set_f64_ieee: only fp64 plans have a double-float mode to switch off");
        return FMM_ERR_INVALID_ARG;
    }
    plan->P.f64_ieee = on != 0;
    plan->P.cache_valid = false;
    return FMM_OK;
}

fmm_status fmm_plan_set_m2l_rotation(fmm_plan *plan, int on)
{
    g_err.clear();
    if (!plan) { set_err("fmm_plan_set_m2l_rotation: NULL plan"); return FMM_ERR_INVALID_ARG; }
    if (on && plan->P.mutual) {
        set_err("fmm_plan_set_m2l_rotation: a mutual plan uses the reduced Cartesian operator");
        return FMM_ERR_INVALID_ARG;
    }
    plan->P.m2l_rotation = on != 0;
    plan->P.cache_valid = false;
    return FMM_OK;
}

fmm_status fmm_plan_set_mutual(fmm_plan *plan, int on)
{
    g_err.clear();
    if (!plan) { set_err("fmm_plan_set_mutual: NULL plan"); return FMM_ERR_INVALID_ARG; }
    if (on && plan->P.m2l_rotation) {
        set_err("fmm_plan_set_mutual: the mutual M2L uses the reduced Cartesian operator; switch the rotation off first");
        return FMM_ERR_INVALID_ARG;
    }
    plan->P.mutual = on != 0;
    plan->P.cache_valid = false;
    return FMM_OK;
}

fmm_status fmm_vjp(fmm_plan *plan, const void *pos, const void *mass, const void *acc_bar, const void *pot_bar,
                   void *pos_bar, void *mass_bar, void *stream)
{
    g_err.clear();
    if (!plan || !pos || !mass || !acc_bar || !pos_bar || !mass_bar) {
        set_err("fmm_vjp: plan, pos, mass, acc_bar, pos_bar and mass_bar must be non-NULL");
        return FMM_ERR_INVALID_ARG;
    }
    Plan &P = plan->P;
    DeviceGuard g(P.device);
    cudaStream_t s = (cudaStream_t)stream;
    P.cache_valid = false;
    const size_t e = (size_t)P.esize, n = (size_t)P.n;
    if (!P.vjp_acc) {
        CUDA_TRY(cudaMalloc(&P.vjp_acc, 3 * n * e));
        CUDA_TRY(cudaMalloc(&P.vjp_src, 4 * n * e));
    }
    // the forward evaluation: tree, lists, complete locals and accelerations
    fmm_status st = eval_device(P, pos, mass, P.vjp_acc, nullptr, s);
    if (st) return st;
    const int fwd_launches = P.launches;
    if (P.vjp_cap_nodes < P.cap_nodes) {
        dfree(P.Ms); dfree(P.Lsm); dfree(P.Ls);
        P.Ms = P.Lsm = P.Ls = nullptr;
        P.vjp_cap_nodes = 0;
        const size_t bytes = (size_t)P.cap_nodes * P.ncp * e;
        CUDA_TRY(cudaMalloc(&P.Ms, bytes));
        CUDA_TRY(cudaMalloc(&P.Lsm, bytes));
        CUDA_TRY(cudaMalloc(&P.Ls, bytes));
        P.vjp_cap_nodes = P.cap_nodes;
    }
    const int vjp_launches = launch_vjp(P, acc_bar, pot_bar, pos_bar, mass_bar, s);
    st = sync_counters(P, s);
    if (st) return st;
    if (P.ctr_host->error) {
        set_err("fmm_vjp: device check failed: %s", error_bits(P.ctr_host->error));
        return FMM_ERR_INTERNAL;
    }
    P.launches = fwd_launches + vjp_launches;
    return FMM_OK;
}

void fmm_destroy(fmm_plan *plan)
{
    if (!plan) return;
    DeviceGuard g(plan->P.device);
    cudaDeviceSynchronize();
    destroy_plan(plan->P);
    delete plan;
}

const char *fmm_last_error(void) { return g_err.c_str(); }

fmm_status fmm_plan_stats(const fmm_plan *plan, fmm_stats *out)
{
    g_err.clear();
    if (!plan || !out) { set_err("fmm_plan_stats: NULL argument"); return FMM_ERR_INVALID_ARG; }
    const Plan &P = plan->P;
    memset(out, 0, sizeof(*out));
    out->n = P.n;
    out->p = P.p;
    if (!P.have_eval) return FMM_OK;
    DeviceGuard g(P.device);
    out->n_nodes = P.n_nodes;
    out->depth = P.depth;
    out->n_m2l = P.n_m2l;
    out->n_p2p_interactions = P.p2p_inter;
    out->walk_pairs = P.walk_pairs;
    out->launches = P.launches;
    out->retries = P.retries;
    // every leaf has exactly one self pair, counted once in the directed lists
    int64_t leaves = 0;
    {
        std::vector<int> nch((size_t)P.n_nodes);
        if (cudaMemcpy(nch.data(), P.node_nchild, nch.size() * sizeof(int), cudaMemcpyDeviceToHost) == cudaSuccess)
            for (int v : nch) leaves += v == 0;
    }
    out->n_leaves = leaves;
    out->n_p2p = 2 * P.n_p2p_pairs - leaves;
    static const int a[FMM_N_STAGES] = {0, 1, 2, 4, 5, 6, 7, 8, 9, 11};
    static const int b[FMM_N_STAGES] = {1, 2, 3, 5, 6, 7, 8, 9, 11, 10};
    for (int k = 0; k < FMM_N_STAGES; ++k) {
        float ms = 0.f;
        cudaEventElapsedTime(&ms, P.ev[a[k]], P.ev[b[k]]);
        out->stage_ms[k] = ms;
    }
    float tot = 0.f;
    cudaEventElapsedTime(&tot, P.ev[0], P.ev[10]);
    out->total_ms = tot;
    return FMM_OK;
}

int64_t fmm_plan_export_size(const fmm_plan *plan, int what)
{
    if (!plan) return -1;
    const Plan &P = plan->P;
    const int64_t nn = P.have_eval ? P.n_nodes : 0, e = P.esize;
    switch (what) {
    case FMM_EXPORT_KEYS: return 8 * P.n;
    case FMM_EXPORT_PERM: return 4 * P.n;
    case FMM_EXPORT_NODE_FIRST: case FMM_EXPORT_NODE_COUNT: case FMM_EXPORT_NODE_CHILD0:
    case FMM_EXPORT_NODE_NCHILD: case FMM_EXPORT_NODE_PARENT: case FMM_EXPORT_NODE_LEVEL: return 4 * nn;
    case FMM_EXPORT_LEVEL_OFF: return 4 * (kMaxLevel + 2);
    case FMM_EXPORT_NODE_LO: case FMM_EXPORT_NODE_HI: case FMM_EXPORT_NODE_CENTRE: case FMM_EXPORT_NODE_HALF:
        return 3 * e * nn;
    case FMM_EXPORT_MULTIPOLE: case FMM_EXPORT_LOCAL_M2L: case FMM_EXPORT_LOCAL: return (int64_t)P.nc * e * nn;
    case FMM_EXPORT_M2L_OFF: case FMM_EXPORT_P2P_OFF: return 4 * (nn + 1);
    case FMM_EXPORT_M2L_SRC: case FMM_EXPORT_P2P_SRC: {
        if (!P.have_eval) return 0;
        int total = 0;
        const int *off = what == FMM_EXPORT_M2L_SRC ? P.m2l_off : P.p2p_off;
        if (cudaMemcpy(&total, off + nn, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
        return 4 * (int64_t)total;
    }
    default: return -1;
    }
}

fmm_status fmm_plan_export(const fmm_plan *plan, int what, void *dst, int64_t bytes)
{
    g_err.clear();
    const int64_t need = fmm_plan_export_size(plan, what);
    if (!plan || !dst || need < 0 || bytes < need) {
        set_err("fmm_plan_export: bad plan, selector or buffer size (need %lld bytes)", (long long)need);
        return FMM_ERR_INVALID_ARG;
    }
    const Plan &P = plan->P;
    DeviceGuard g(P.device);
    CUDA_TRY(cudaDeviceSynchronize());
    const int64_t nn = P.n_nodes, e = P.esize;
    auto copy = [&](const void *src) -> fmm_status {
        CUDA_TRY(cudaMemcpy(dst, src, (size_t)need, cudaMemcpyDeviceToHost));
        return FMM_OK;
    };
    switch (what) {
    case FMM_EXPORT_KEYS: return copy(P.keys[0]);
    case FMM_EXPORT_PERM: return copy(P.idx[0]);
    case FMM_EXPORT_NODE_FIRST: return copy(P.node_first);
    case FMM_EXPORT_NODE_COUNT: return copy(P.node_count);
    case FMM_EXPORT_NODE_CHILD0: return copy(P.node_child0);
    case FMM_EXPORT_NODE_NCHILD: return copy(P.node_nchild);
    case FMM_EXPORT_NODE_PARENT: return copy(P.node_parent);
    case FMM_EXPORT_NODE_LEVEL: return copy(P.node_level);
    case FMM_EXPORT_LEVEL_OFF: memcpy(dst, P.ctr_host->level_off, (size_t)need); return FMM_OK;
    case FMM_EXPORT_NODE_LO: return copy(P.node_lo);
    case FMM_EXPORT_NODE_HI: return copy(P.node_hi);
    case FMM_EXPORT_M2L_OFF: return copy(P.m2l_off);
    case FMM_EXPORT_P2P_OFF: return copy(P.p2p_off);
    case FMM_EXPORT_M2L_SRC: return copy(P.m2l_src);
    case FMM_EXPORT_P2P_SRC: return copy(P.p2p_src);
    case FMM_EXPORT_NODE_CENTRE: case FMM_EXPORT_NODE_HALF: {
        std::vector<char> tmp((size_t)(4 * e * nn));
        CUDA_TRY(cudaMemcpy(tmp.data(), what == FMM_EXPORT_NODE_CENTRE ? P.node_c : P.node_l, tmp.size(),
                            cudaMemcpyDeviceToHost));
        for (int64_t a = 0; a < nn; ++a) memcpy((char *)dst + 3 * e * a, tmp.data() + 4 * e * a, (size_t)(3 * e));
        return FMM_OK;
    }
    case FMM_EXPORT_MULTIPOLE: case FMM_EXPORT_LOCAL_M2L: case FMM_EXPORT_LOCAL: {
        const void *src = what == FMM_EXPORT_MULTIPOLE ? P.M : (what == FMM_EXPORT_LOCAL_M2L ? P.Lm2l : P.L);
        std::vector<char> tmp((size_t)(P.ncp * e * nn));
        CUDA_TRY(cudaMemcpy(tmp.data(), src, tmp.size(), cudaMemcpyDeviceToHost));
        for (int64_t a = 0; a < nn; ++a)
            memcpy((char *)dst + P.nc * e * a, tmp.data() + P.ncp * e * a, (size_t)(P.nc * e));
        return FMM_OK;
    }
    default: break;
    }
    set_err("fmm_plan_export: unknown selector %d", what);
    return FMM_ERR_INVALID_ARG;
}

}  // extern "C"
