// Host-side plan of the FMM library: device buffers, capacities and the
// launchers each kernel file provides.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace bfm {

constexpr int kNumEvents = 12;

struct Plan {
    // parameters
    int64_t n = 0;
    int p = 4;
    int nc = 35;        // coefficients per expansion
    int ncp = 36;       // padded row stride (multiple of 4 elements)
    int nrc = 25;       // reduced coefficients (p + 1)^2
    int nrp = 28;       // their padded row stride (multiple of 4)
    double theta = 0.7;
    int leaf = 32;
    int dtype = 0;      // 0 f32, 1 f64
    bool f64_ieee = false;  // fp64 plans: every stage in IEEE fp64 (default: the ALU-bound stages in double-float)
    bool m2l_rotation = false;  // M2L by rotation to the z axis in solid harmonics (default: reduced Cartesian)
    bool mutual = false;        // M2L and P2P once per unordered pair, both directions (plain arithmetic)
    int esize = 4;      // bytes per real
    int device = 0;
    int num_sms = 148;
    int coop_blocks_tree = 148;   // grids of the cooperative launches (co-resident blocks)
    int coop_blocks_walk = 148;
    int coop_tiles_sort[2] = {0, 0};  // co-resident tiles of the cooperative radix sort (small, large tiles)

    // capacities
    int64_t cap_nodes = 0, cap_frontier = 0, cap_m2l = 0, cap_p2p = 0, cap_flags = 0;
    bool minimal_caps = false;     // BFM_FMM_FAULT=capacity: buffers start at their minimum
    bool fault_spin = false;       // BFM_FMM_FAULT=spin: the level-ordered L2L kernel (also in fp32 plans)
                                   // waits for a flag value that no pass stores

    // particle buffers
    uint64_t *keys[2] = {nullptr, nullptr};
    uint32_t *idx[2] = {nullptr, nullptr};
    void *xyzm = nullptr;          // sorted particles, vec4<T> (x, y, z, m)
    void *far = nullptr;           // far field at the sorted particles, vec4<T> (phi, ax, ay, az)
    uint8_t *div = nullptr;        // divergence level of consecutive sorted keys
    uint8_t *vwin = nullptr;       // per sorted position: the deepest level whose run around it holds > leaf keys
    int *leaf_of = nullptr;        // per sorted particle: its leaf (written by the direct L2L)
    int *tree_cc = nullptr;        // per level and chunk of positions: node counts, then their offsets
    void *rel = nullptr;           // fp64 plans: leaf-relative particles as double-float float4 [2][N]

    // node buffers
    int *node_first = nullptr, *node_count = nullptr, *node_child0 = nullptr, *node_nchild = nullptr;
    int *node_parent = nullptr, *node_level = nullptr, *node_done = nullptr;
    void *node_lo = nullptr, *node_hi = nullptr;  // T[3] per node
    void *node_c = nullptr, *node_l = nullptr;    // vec4<T>: (cx, cy, cz, |l|^2), (lx, ly, lz, 0)
    void *node_w = nullptr;  // the walk's node records, 2 vec4<T>: (cx, cy, cz, nchild), (lx, ly, lz, child0), ints as bits
    void *M = nullptr, *Lm2l = nullptr, *L = nullptr;  // T[ncp] per node
    void *Mr = nullptr;            // reduced (n_z <= 1) moments for M2L, [nrp] 8-byte slots per node: T for
                                   // fp32 and fp64 p >= 5, double-float pairs in level units for fp64 p <= 4

    // walk and lists
    int2 *frontier[2] = {nullptr, nullptr};
    int2 *m2l_pairs = nullptr, *p2p_pairs = nullptr;
    int *m2l_cnt = nullptr, *p2p_cnt = nullptr;    // per receiver counts (also fill cursors)
    int *m2l_off = nullptr, *p2p_off = nullptr;    // CSR offsets [cap_nodes + 1]
    int *m2l_src = nullptr, *p2p_src = nullptr;    // CSR sources [2 * cap]
    int *long_seg = nullptr;                       // receivers whose lists are too long for the warp sort
    int *order = nullptr;                          // [2][cap_nodes] receivers by decreasing work (M2L in [1])
    int2 *p2p_items = nullptr;                     // [2 cap_nodes] P2P work items (receiver, chunk | chunks << 8)
    int *p2p_done = nullptr;                       // [cap_nodes] chunks of a receiver applied so far
    uint8_t *p2p_nch = nullptr;                    // [cap_nodes] P2P chunks of every receiver
    unsigned *node_flag = nullptr;                 // [cap_nodes] number of the last pass that completed the node
    unsigned flag_seq = 0;                         // the last pass number handed out (0: none)
    uint8_t *order_key = nullptr;                  // [2][cap_nodes] work bucket of every node

    void *scratch = nullptr;       // 64 KiB for small per-block partials

    // chained-scan flags
    unsigned long long *flags = nullptr;
    unsigned epoch = 0;
    int slot = 0;                  // next ticket counter

    // status
    DevCounters *ctr = nullptr;      // device
    GridBarrier *gbar = nullptr;     // device: barriers of the cooperative tree [0], walk [1] and sort [2]
    unsigned *sort_cnt = nullptr;    // device: per tile and digit, the cooperative sort's counts and offsets
    size_t sort_cnt_cap = 0;         // its entries
    int2 *sort_big = nullptr;        // device: (start, length) of the runs of equal high key words longer than one
                                     // thread sorts
    size_t sort_big_cap = 0;         // its entries (such runs hold over 32 keys each)
    bool sort_full = false;          // sort all 8 key digits: the last evaluation found many keys in long runs
    bool mr_fresh = false;           // the upward pass wrote the reduced rows of this evaluation's moments
    DevCounters *ctr_host = nullptr; // pinned mirror

    // host-buffer staging (fmm_eval_host), allocated on first use
    void *h_pos = nullptr, *h_mass = nullptr, *h_acc = nullptr, *h_pot = nullptr;

    // VJP (fmm_vjp), allocated on first use: the forward accelerations (caller's order), the sources
    // (pbar, -abar) in the tree's order, and the source moments, M2L locals and complete locals
    void *vjp_acc = nullptr, *vjp_src = nullptr;
    void *Ms = nullptr, *Lsm = nullptr, *Ls = nullptr;
    int64_t vjp_cap_nodes = 0;

    // mutual evaluation (fmm_plan_set_mutual), allocated on first use and grown when an evaluation reports
    // one short: per node the lower-part lengths of the M2L and P2P lists and the start of the P2P upper
    // part [3][cap_nodes], the P2P share slots [cap_nodes + 1] and the own reduced M2L share [cap_nodes]
    // rows; per M2L list entry the mirrored entry and the partner's reduced share (a row) [mut_cap_em]; per
    // P2P list entry the mirrored entry [mut_cap_ep]; the partners' P2P sums [mut_cap_rp] and the own P2P
    // sums [n]
    int *mut_lo = nullptr, *mut_mir_m2l = nullptr, *mut_mir_p2p = nullptr;
    long long *mut_base = nullptr;
    void *mut_rm2l = nullptr, *mut_lpart = nullptr, *mut_rp2p = nullptr, *mut_own = nullptr;
    long long mut_cap_rp = 0, mut_cap_em = 0, mut_cap_ep = 0;
    int64_t mut_for_nodes = 0;     // node capacity the per-node buffers were sized for

    // KDK acceleration cache, caller's order
    void *acc_cache = nullptr;
    bool cache_valid = false;
    const void *cache_pos = nullptr, *cache_vel = nullptr, *cache_mass = nullptr;

    // timing and stats of the last evaluation
    cudaEvent_t ev[kNumEvents] = {};
    cudaEvent_t ev_done = nullptr;   // completion of the status read-back (polled)
    // host-buffer evaluations: the mass upload runs on a side stream while the keys and the first
    // radix passes run; the pass that gathers the masses waits on mass_wait when it is set
    cudaStream_t side = nullptr;
    cudaEvent_t ev_pos = nullptr, ev_mass = nullptr, mass_wait = nullptr;
    int ev_stage[kNumEvents] = {};
    int n_ev = 0;
    int launches = 0;
    int retries = 0;
    int depth = 0;
    int64_t n_nodes = 0, n_leaves = 0, n_m2l = 0, n_p2p = 0, n_p2p_pairs = 0, p2p_inter = 0, walk_pairs = 0;
    bool have_eval = false;
    double stage_ms[16] = {};
    double total_ms = 0;

    unsigned next_epoch();
    unsigned next_flag_seq(cudaStream_t s);  // a fresh, nonzero node_flag value for one pass
    int next_slot() { return slot++; }
};

// ---- launchers (one per kernel file) ----------------------------------------
// Each returns the number of kernels it launched.
int launch_keys(Plan &P, const void *pos, cudaStream_t s);
int launch_sort(Plan &P, const void *pos, const void *mass, cudaStream_t s);
int launch_tree(Plan &P, cudaStream_t s);
size_t tree_cc_ints(int64_t n);  // size of Plan::tree_cc for n particles
void sort_coop_capacity(int num_sms, int tiles[2]);  // co-resident tiles of the cooperative sort
int tree_max_blocks_per_sm();
int walk_max_blocks_per_sm(int dtype);
int launch_upward(Plan &P, cudaStream_t s);
int launch_walk(Plan &P, int depth, cudaStream_t s);
int launch_lists(Plan &P, cudaStream_t s);
int launch_m2l(Plan &P, cudaStream_t s);
int launch_m2l_df(Plan &P, cudaStream_t s);  // fp64 plans, p <= kMaxPDf
int launch_m2l_plain(Plan &P, const void *M, void *Lout, cudaStream_t s);  // plain arithmetic, given buffers
int launch_mutual_index(Plan &P, cudaStream_t s);  // mutual plans: lower parts, mirrored entries, P2P slots
int launch_p2p_mutual(Plan &P, void *acc, void *pot, cudaStream_t s);
int launch_vjp(Plan &P, const void *abar, const void *pbar, void *pos_bar, void *mass_bar, cudaStream_t s);
constexpr int kMaxPDf = 4;
int launch_l2l(Plan &P, int depth, cudaStream_t s);
int launch_l2p(Plan &P, cudaStream_t s);
int launch_p2p(Plan &P, void *acc, void *pot, cudaStream_t s);
int launch_p2p_df(Plan &P, void *acc, void *pot, cudaStream_t s);
int launch_l2p_df(Plan &P, cudaStream_t s);  // fp64 plans, p <= kMaxPL2pDf
constexpr int kMaxPL2pDf = 6;
int launch_kick(Plan &P, void *vel, const void *acc, double h, cudaStream_t s);
int launch_drift(Plan &P, void *pos, const void *vel, double dt, cudaStream_t s);
int launch_lattice_axpy(Plan &P, void *y, const void *x, double h, int e_y, int e_inc, cudaStream_t s);

inline int grid_for(const Plan &P, int per_sm = 8) { return P.num_sms * per_sm; }

}  // namespace bfm
