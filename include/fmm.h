/*
 * fmm.h -- C ABI of the B300 Fast Multipole Method library (libbfm_fmm.so).
 *
 * One call of fmm_eval computes, for N particles, the Newtonian potential
 *     Phi_i = -G sum_{j != i} m_j / |x_i - x_j|
 * and the acceleration a_i = -grad Phi_i (G = 1, no softening, self-interaction
 * and other zero-separation pairs omitted), approximated by the Fast Multipole
 * Method (JZ-FMM page, sections "From particle pairs to node pairs" and
 * "Combining near and far interactions"):
 *   1. Morton keys on 21 bits per axis of the root cube and a stable radix sort;
 *   2. an octree over the sorted keys, a node splitting while it holds more than
 *      `leaf` particles (at most 21 levels), children stored contiguously
 *      ("Why this works well on GPUs");
 *   3. Cartesian multipole moments M_n = sum m s^n / n! up to order p at the
 *      leaves (P2M) and translated to the parents (M2M) ("Describing the source
 *      and the receiving region", moment eqs.);
 *   4. a symmetric dual-tree walk accepting a node pair (A, B) when
 *      |l_A + l_B| < theta |c_A - c_B| (the opening-criterion eq.; c is the
 *      centre, l the per-axis half-width of the node's tight box), which emits
 *      M2L and P2P interaction lists;
 *   5. multipole-to-local translation (M2L) keeping every term of total degree
 *      |n| + |k| <= p ("Calculating a node-node interaction", Phi_B and
 *      grad Phi_B eqs.; "terms through total degree p", demo caption);
 *   6. the downward pass: L2L to the children and L2P at the particles
 *      (Taylor eq.), plus the direct near-field sum P2P over the P2P lists.
 * fmm_kdk_step adds a kick-drift-kick leapfrog step built on that force
 * (Jaxion post, section "Implementation": half kick, drift, half kick).
 *
 * Conventions for every call:
 *  - Array arguments of fmm_eval / fmm_kdk_step are DEVICE pointers owned by the
 *    caller, in the plan's dtype (float for FMM_F32, double for FMM_F64):
 *    pos, vel, acc are N x 3 row-major (x, y, z per particle), mass and pot have
 *    N entries. Outputs come back in the caller's particle order.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream). All GPU work is enqueued on it. The calls are blocking: they
 *    return once the results are complete and checked. Every kernel reads the
 *    tree's size from device memory, so the stream is synchronised once per
 *    evaluation, at the end, to read back the device-side status word (an
 *    evaluation that overflowed a buffer is then repeated with grown buffers).
 *  - A plan is not thread-safe: one call in flight per plan.
 *  - Errors are returned as status codes, never as a process abort; the reason
 *    is available from fmm_last_error() on the calling thread.
 *  - Results are reproducible: the same plan, inputs and device give bitwise
 *    identical outputs (no floating-point atomics; fixed summation orders).
 */
#ifndef BFM_FMM_H
#define BFM_FMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Arithmetic type of a plan: positions, masses, expansions and accumulators.
 * FMM_F32 computes every stage in fp32. FMM_F64 takes and returns fp64; its
 * two ALU-bound stages, P2P and (for p <= 4) M2L, run in double-float
 * arithmetic (unevaluated sums of two fp32 numbers, ~2^-48 relative) on the
 * FP32 pipe, whose rate on this GPU is far above the FP64 pipe's, in
 * power-of-two units of the root box and total mass; near-field pairs closer
 * than 2^-8 of their leaf pair's extent, and M2L pairs outside those units'
 * range, are evaluated in fp64. The other stages compute in fp64.
 */
typedef enum { FMM_F32 = 0, FMM_F64 = 1 } fmm_dtype;

typedef enum {
    FMM_OK = 0,
    FMM_ERR_INVALID_ARG = 1, /* bad size, order, angle, leaf size, pointer or dtype */
    FMM_ERR_OOM = 2,         /* device or host allocation failed */
    FMM_ERR_CUDA = 3,        /* a CUDA runtime call failed (message has the CUDA error) */
    FMM_ERR_CAPACITY = 4,    /* lists still overflow after the retries, or over 2^30 nodes / 1e9 pairs */
    FMM_ERR_NONFINITE = 5,   /* a position is NaN or infinite */
    FMM_ERR_INTERNAL = 6     /* a device-side consistency check failed */
} fmm_status;

/* Stages timed by the plan (CUDA events on the plan's stream). */
enum {
    FMM_STAGE_KEYS = 0,  /* root box, Morton keys, digit histograms */
    FMM_STAGE_SORT = 1,  /* radix sort passes + gather into sorted SoA */
    FMM_STAGE_TREE = 2,  /* octree levels */
    FMM_STAGE_UP = 3,    /* node boxes, P2M, M2M */
    FMM_STAGE_WALK = 4,  /* dual-tree walk */
    FMM_STAGE_LISTS = 5, /* interaction lists into per-receiver CSR, canonical order */
    FMM_STAGE_M2L = 6,
    FMM_STAGE_L2L = 7,
    FMM_STAGE_L2P = 8,   /* local expansions at the leaves' particles */
    FMM_STAGE_P2P = 9,   /* near field + far field, scattered to the caller's order */
    FMM_N_STAGES = 10
};

typedef struct fmm_plan fmm_plan;

/* Counts and timings of the last completed evaluation of a plan. */
typedef struct {
    int64_t n;                  /* particles */
    int64_t n_nodes;            /* octree nodes */
    int64_t n_leaves;
    int32_t depth;              /* deepest level (root = 0) */
    int32_t p;                  /* expansion order */
    int64_t n_m2l;              /* directed M2L list entries (receiver <- source node) */
    int64_t n_p2p;              /* directed P2P list entries (receiver leaf <- source leaf) */
    int64_t n_p2p_interactions; /* particle pairs evaluated by P2P, sum |A||B| over entries */
    int64_t walk_pairs;         /* node pairs visited by the walk */
    double stage_ms[FMM_N_STAGES];
    double total_ms;            /* first stage start to last stage end, device time */
    int32_t launches;           /* kernels this library launched for the evaluation */
    int32_t retries;            /* capacity regrowths during the evaluation */
} fmm_stats;

/*
 * Create a plan for `n` particles (n >= 1), expansion order p in [0, 8],
 * opening angle theta in (0, 1], leaf size leaf >= 1, arithmetic `dtype`.
 * Allocates the device scratch for n particles on the current CUDA device.
 * Returns NULL on failure (fmm_last_error() says why).
 */
fmm_plan *fmm_plan_create(int64_t n, int p, double theta, int leaf, fmm_dtype dtype);

/*
 * One evaluation. pos [n x 3], mass [n] (device, read only); acc_out [n x 3]
 * (device, written); pot_out [n] (device, written) or NULL to skip the potential.
 * Returns FMM_OK, FMM_ERR_INVALID_ARG (NULL pos/mass/acc), FMM_ERR_NONFINITE,
 * FMM_ERR_CAPACITY, FMM_ERR_CUDA or FMM_ERR_INTERNAL; outputs are undefined on error.
 */
fmm_status fmm_eval(fmm_plan *plan, const void *pos, const void *mass, void *acc_out, void *pot_out,
                    void *stream);

/*
 * Same evaluation with HOST buffers (pageable or pinned): the call copies pos and
 * mass to plan-owned device memory, evaluates, and copies acc (and pot, unless
 * NULL) back before returning. The mass copy runs on a plan-owned side stream,
 * ordered after the position copy, while the first stages run on `stream`; both
 * have ended when the call returns, on success and on error.
 */
fmm_status fmm_eval_host(fmm_plan *plan, const void *pos, const void *mass, void *acc_out, void *pot_out,
                         void *stream);

/*
 * One kick-drift-kick step of length dt (dt < 0 steps backwards), in place on the
 * device arrays pos [n x 3] and vel [n x 3]; mass [n] is read only:
 *     v += a(x) dt/2;  x += v dt;  v += a(x) dt/2.
 * The acceleration at the end of a step is cached in the plan and reused as the
 * first half kick of the next step when the next call passes the same pos, vel
 * and mass pointers and no other call has used the plan in between; the caller
 * must not modify pos between such calls (use fmm_kdk_reset otherwise).
 */
fmm_status fmm_kdk_step(fmm_plan *plan, void *pos, void *vel, const void *mass, double dt, void *stream);

/*
 * The same step on an integer lattice (JZ-FMM page, "Why reversibility
 * matters"): positions live on the lattice 2^pos_exp Z, velocities on
 * 2^vel_exp Z, and every kick and drift increment is rounded to its lattice
 * (round half to even, so the increment of -dt is exactly minus that of dt).
 * The force stays floating point and is reproduced bit for bit at a revisited
 * state, so a step with -dt undoes a step with dt exactly, whatever the
 * dynamics. pos and vel are first rounded to their lattices (a no-op once they
 * lie there). The values must stay below 2^(mantissa bits) lattice units
 * (|x| < 2^(53 + pos_exp) in fp64) for the sums to be exact. Shares the
 * acceleration cache of fmm_kdk_step.
 */
fmm_status fmm_kdk_step_lattice(fmm_plan *plan, void *pos, void *vel, const void *mass, double dt, int pos_exp,
                                int vel_exp, void *stream);

/*
 * Arithmetic of an fp64 plan. By default (on = 0) the ALU-bound stages of an
 * fp64 plan -- M2L for p <= 4, L2P and the leaf P2M for p <= 6, and P2P --
 * compute in double-float (pairs of fp32 values, about 48 significant bits) on
 * the FP32 pipe, because the B300's FP64 rate is about 1/64 of its FP32 rate;
 * the results stay within 1e-12 of the fp64 oracle. on = 1 runs every stage in
 * IEEE fp64 instead (slower; the pages' own precision). Applies to the next
 * evaluation. FMM_ERR_INVALID_ARG for a NULL plan or on = 1 on an fp32 plan.
 */
fmm_status fmm_plan_set_f64_ieee(fmm_plan *plan, int on);

/*
 * M2L operator of the plan. on = 0 (default): the reduced (trace-free)
 * Cartesian contraction, the derivative tensor of 1/r built by recurrence per
 * pair. on = 1: the rotation-based M2L of jaccpot issue 152 (item 1, "An
 * on-chip-rotation ... M2L kernel"): in real solid harmonics, each source
 * multipole is rotated so that the separation lies on the z axis, translated
 * along z (a translation that only couples equal orders m), and the local is
 * rotated back, the rotations built on chip from the separation. Both keep
 * every term of total degree <= p, so they give the same result up to
 * rounding; the per-pair work differs (O(p^3) here against the reduced
 * contraction's O(p^4), with larger constants, so the Cartesian form is the
 * faster one for p <= 8). fp64 plans with rotation run their M2L in IEEE fp64.
 * Applies to the next evaluation; FMM_ERR_INVALID_ARG for a NULL plan or, with
 * on != 0, a mutual plan.
 */
fmm_status fmm_plan_set_m2l_rotation(fmm_plan *plan, int on);

/*
 * Mutual (symmetric) evaluation of the interaction lists (jaccpot issue 152,
 * "Mutual FMM"): each unordered accepted pair of nodes is evaluated once for
 * both receivers, one derivative tensor per M2L pair (D^m(-R) = (-1)^{|m|}
 * D^m(R)) and one separation and reciprocal square root per particle pair with
 * equal and opposite forces. The result is the same truncation as the default
 * evaluation, equal to it up to rounding. Sums stay deterministic (bit for bit
 * from run to run): the receiver with the lower node index evaluates the pair,
 * the partner's share goes to a buffer slot and is added by a second pass in
 * list order. M2L and P2P then run in plain arithmetic of the plan's dtype
 * (IEEE fp64 in fp64 plans). The plan allocates the buffers on first use: about
 * 2 x (M2L list capacity) x (p+1)^2 reals plus 32 particle sums per particle,
 * grown and the evaluation repeated when that is short. on != 0 switches it on.
 * FMM_ERR_INVALID_ARG for a NULL plan or together with the rotation-based M2L
 * (the mutual M2L uses the reduced Cartesian operator). Applies to the next
 * evaluation.
 */
fmm_status fmm_plan_set_mutual(fmm_plan *plan, int on);

/*
 * Vector-Jacobian product of one evaluation (JZ-FMM page, "Differentiating the
 * force calculation": one contribution from the next higher derivative of the
 * original evaluation, one from an FMM with the force sensitivities acting as
 * dipole moments). For the loss l = sum_i acc_bar_i . a_i + pot_bar_i phi_i it
 * writes pos_bar = dl/dx [n x 3] and mass_bar = dl/dm [n]:
 *     pos_bar_k  = m_k grad Phi_s(x_k) - Hess Phi(x_k) acc_bar_k - pot_bar_k a_k
 *     mass_bar_k = Phi_s(x_k),
 * Phi the forward potential, Phi_s the potential of sources at every particle
 * with monopole pot_bar_j and dipole -acc_bar_j (self terms omitted), both on the
 * forward evaluation's tree, centres and lists: the exact derivatives of the
 * evaluation with the tree and the expansion centres held fixed (moving a
 * particle that bounds a node's box also moves that node's centre, which this
 * does not differentiate; the effect is of the order of the FMM's error).
 * Arguments are DEVICE arrays in the plan's dtype and the caller's particle
 * order; pot_bar may be NULL (zero). The call runs the forward evaluation
 * first (it does not reuse an earlier one), allocates the plan's VJP buffers on
 * first use, blocks until done and returns FMM_ERR_INTERNAL if a device check
 * failed. It invalidates the kick-drift-kick acceleration cache.
 */
fmm_status fmm_vjp(fmm_plan *plan, const void *pos, const void *mass, const void *acc_bar, const void *pot_bar,
                   void *pos_bar, void *mass_bar, void *stream);

/* Drop the cached acceleration of fmm_kdk_step (the next step evaluates it afresh). */
void fmm_kdk_reset(fmm_plan *plan);

/* Release the plan and its device memory. NULL is accepted. */
void fmm_destroy(fmm_plan *plan);

/* Message of the last failure on the calling thread ("" if none). */
const char *fmm_last_error(void);

/* Counts and per-stage device times of the plan's last evaluation. */
fmm_status fmm_plan_stats(const fmm_plan *plan, fmm_stats *out);

/*
 * Inspection of intermediate results of the last evaluation (tests and tools).
 * `what` selects an array; fmm_plan_export_size gives its size in bytes (or -1
 * for an unknown selector) and fmm_plan_export copies it into the HOST buffer
 * `dst` of `bytes` bytes (FMM_ERR_INVALID_ARG when too small). Layouts:
 *   KEYS       uint64 [n]        sorted Morton keys
 *   PERM       uint32 [n]        sorted slot -> caller's particle index
 *   NODE_FIRST, NODE_COUNT, NODE_CHILD0, NODE_NCHILD, NODE_PARENT, NODE_LEVEL
 *              int32 [n_nodes]   breadth-first node order, children contiguous
 *                                (child0 = -1 and nchild = 0 at leaves, parent of the root = -1)
 *   LEVEL_OFF  int32 [23]        nodes of level l are [LEVEL_OFF[l], LEVEL_OFF[l+1])
 *   NODE_LO, NODE_HI, NODE_CENTRE, NODE_HALF
 *              dtype [n_nodes x 3]  tight box, c = (lo+hi)/2, l = (hi-lo)/2
 *   MULTIPOLE, LOCAL_M2L, LOCAL
 *              dtype [n_nodes x ncoef]  ncoef = (p+1)(p+2)(p+3)/6, graded order
 *                                (degree d = 0..p; within a degree x exponent
 *                                descending, then y exponent descending);
 *                                LOCAL_M2L holds the M2L terms only, LOCAL the
 *                                complete local expansion after L2L
 *   M2L_OFF, P2P_OFF  int32 [n_nodes + 1]  CSR offsets by receiver node
 *   M2L_SRC, P2P_SRC  int32 [n_m2l], [n_p2p] source nodes, ascending per receiver
 */
enum {
    FMM_EXPORT_KEYS = 0,
    FMM_EXPORT_PERM = 1,
    FMM_EXPORT_NODE_FIRST = 2,
    FMM_EXPORT_NODE_COUNT = 3,
    FMM_EXPORT_NODE_CHILD0 = 4,
    FMM_EXPORT_NODE_NCHILD = 5,
    FMM_EXPORT_NODE_PARENT = 6,
    FMM_EXPORT_NODE_LEVEL = 7,
    FMM_EXPORT_LEVEL_OFF = 8,
    FMM_EXPORT_NODE_LO = 9,
    FMM_EXPORT_NODE_HI = 10,
    FMM_EXPORT_NODE_CENTRE = 11,
    FMM_EXPORT_NODE_HALF = 12,
    FMM_EXPORT_MULTIPOLE = 13,
    FMM_EXPORT_LOCAL_M2L = 14,
    FMM_EXPORT_LOCAL = 15,
    FMM_EXPORT_M2L_OFF = 16,
    FMM_EXPORT_M2L_SRC = 17,
    FMM_EXPORT_P2P_OFF = 18,
    FMM_EXPORT_P2P_SRC = 19,
    FMM_EXPORT_COUNT = 20
};
int64_t fmm_plan_export_size(const fmm_plan *plan, int what);
fmm_status fmm_plan_export(const fmm_plan *plan, int what, void *dst, int64_t bytes);

/*
 * Root box and Morton keys without any device allocation (the pages have no
 * counterpart; this is a library convenience).
 *
 * For callers that cannot allocate device memory when they need the keys: code
 * working within a fixed memory budget handed out by its own allocator, a
 * library embedded in a host application that forbids device allocation after
 * start-up, or a real-time loop that must not take the driver's allocation
 * locks. It needs no plan: the caller passes pos [n x 3] (device,
 * `dtype` reals) and keys_out [n] (device, uint64, written in the caller's
 * particle order) and optionally box_out [4] (device doubles: the root cube's
 * lower corner x, y, z and its side). The keys are the same as the plan path's
 * (21-bit quantisation against the root cube, x highest in each 3-bit digit).
 *
 * Scratch: a fixed 48 KiB array in the library's device image (one partial box
 * per 2048 particles, for at most 1024 blocks), held by every GPU that loads
 * the library until the process exits. Hence n must be in [1, 2^21]; larger n
 * (or NULL pos/keys_out, or an unknown dtype) returns FMM_ERR_INVALID_ARG
 * without touching the GPU. The first call on a device looks the array's
 * device address up (once per device, with that device current); make that
 * first call before any stream capture. Every call clears the words that must
 * start at zero; calls that overlap on the GPU (two streams, or two host
 * threads on one device) share the array and race. The call blocks until the
 * keys are written and returns FMM_ERR_NONFINITE if a coordinate is NaN or
 * infinite. It calls no allocating routine.
 */
fmm_status fmm_morton_keys_noalloc(const void *pos, int64_t n, fmm_dtype dtype, uint64_t *keys_out,
                                   double *box_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BFM_FMM_H */
