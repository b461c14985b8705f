// Shared device utilities of the FMM library: vector types, exactly rounded
// scalar operations for the geometry, the device status word, a decoupled
// look-back chained scan and warp helpers.
#pragma once

#include <cuda/atomic>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bfm {

constexpr int kMaxLevel = 21;        // Morton keys carry 21 bits per axis
constexpr int kMaxP = 8;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kShards = 64;          // the walk's outputs are split into this many independently counted shards
// P2P work of one receiver leaf is split into up to kMaxChunks chunks of its
// source list, taken by different warps, when it is above the largest of
// kChunkWork interactions, the total over the node capacity (which bounds the
// number of chunks) and the total over kShareDiv per SM (about a third of an
// even share of the resident warps, so that no single receiver's warp is left
// running alone at the end of the near field).
// fp64 plans keep a floor of 2^20: a double-float pair costs several fp32 pairs,
// and their chunk waits cost more than the tail they would cut.
constexpr long long kChunkWork = 1ll << 16;
constexpr long long kChunkWorkF64 = 1ll << 20;
constexpr int kShareDiv = 64;
constexpr int kMaxChunks = 64;
constexpr unsigned kSpinLimit = 1u << 22;  // iterations of any bounded wait
// polls of a chunk-turn wait (wait_turn), the first 4096 64 ns apart and the rest 1 us apart: about
// 17 s. The earlier chunk of a receiving leaf of thousands of particles can take most of a second in
// double-float arithmetic, since a chunk's first round waits for the earlier chunk's every round
constexpr unsigned kTurnSpinLimit = 1u << 24;

// ---- device status word bits (ORed by kernels, read by the host) ----------
enum : unsigned {
    ERR_NONFINITE = 1u << 0,  // a NaN / Inf position
    ERR_NODES = 1u << 1,      // node capacity exceeded
    ERR_FRONTIER = 1u << 2,   // walk frontier capacity exceeded
    ERR_M2L_CAP = 1u << 3,    // M2L pair capacity exceeded
    ERR_P2P_CAP = 1u << 4,    // P2P pair capacity exceeded
    ERR_SPIN = 1u << 5,       // a bounded wait gave up
    ERR_BOUNDS = 1u << 6,     // an index check failed (skipped access)
    ERR_WALK = 1u << 7,       // walk did not terminate in the expected iterations
    ERR_MUT_CAP = 1u << 8,    // a mutual-evaluation buffer too small (needed sizes in mut_need)
};

// ---- per-evaluation device counters (zeroed at the start of every evaluation)
struct DevCounters {
    unsigned error;
    int n_nodes;
    int depth;
    int bbox_done;
    int level_off[kMaxLevel + 3];
    double box[4];                 // root box min corner (x, y, z) and side, in the plan's dtype widened
    unsigned hist[8][256];         // radix digit histograms, one row per pass
    unsigned tile_ctr[96];         // one ticket counter per chained-scan use
    int frontier_cnt[3][64];       // walk frontier sizes per shard (cycled over 3 generations)
    int frontier_max;              // largest shard fill seen by the walk
    int n_m2l_pairs[64];           // unordered M2L pairs per shard
    int n_p2p_pairs[64];           // unordered P2P pairs per shard (self pairs included)
    long long walk_pairs;
    long long p2p_interactions;
    int n_long;                    // list segments too long for the warp sort
    int n_sort_groups;             // runs of equal high key words too long for one thread
    int sort_long_keys;            // the keys in those runs
    long long mut_need[3];         // mutual buffers needed (set with ERR_MUT_CAP): P2P share slots, M2L
                                   // list entries, P2P list entries
    int order_cnt[2][64];          // work buckets (0: P2P receivers, 1: M2L receivers)
    int order_cur[2][64];
    int work_ctr[4];               // dynamic work counters
};

// ---- vector types ---------------------------------------------------------
struct __align__(32) dbl4 { double x, y, z, w; };
template <class T> struct V4;
template <> struct V4<float> { using type = float4; };
template <> struct V4<double> { using type = dbl4; };
template <class T> using vec4 = typename V4<T>::type;

template <class T> __device__ __forceinline__ vec4<T> make4(T x, T y, T z, T w)
{
    vec4<T> v;
    v.x = x; v.y = y; v.z = z; v.w = w;
    return v;
}

// ---- exactly rounded scalar ops (never contracted into FMA) ----------------
__device__ __forceinline__ float add_rn(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ double add_rn(double a, double b) { return __dadd_rn(a, b); }
__device__ __forceinline__ float sub_rn(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ double sub_rn(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ float mul_rn(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ double mul_rn(double a, double b) { return __dmul_rn(a, b); }
__device__ __forceinline__ float div_rn(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ double div_rn(double a, double b) { return __ddiv_rn(a, b); }

// |v|^2 as ((x*x + y*y) + z*z), every step rounded
template <class T> __device__ __forceinline__ T norm2_rn(T x, T y, T z)
{
    return add_rn(add_rn(mul_rn(x, x), mul_rn(y, y)), mul_rn(z, z));
}

// ---- loads that bypass L1 (data written by other blocks of the same kernel)
template <class T> __device__ __forceinline__ T ld_cg(const T *p) { return __ldcg(p); }
__device__ __forceinline__ dbl4 ld_cg(const dbl4 *p)
{
    const double2 *q = reinterpret_cast<const double2 *>(p);
    double2 a = __ldcg(q), b = __ldcg(q + 1);
    dbl4 r;
    r.x = a.x; r.y = a.y; r.z = b.x; r.w = b.y;
    return r;
}

__device__ __forceinline__ void set_error(DevCounters *c, unsigned bit) { atomicOr(&c->error, bit); }

// Node count for the kernels after the tree build, read on the device (they are
// launched without the host waiting for the tree): 0 when the tree build failed
// (node capacity exceeded or a non-finite position), so that every later stage
// skips the inconsistent tree and the evaluation retries or reports the error.
__device__ __forceinline__ int phase2_nodes(const DevCounters *ctr)
{
    return (ctr->error & (ERR_NODES | ERR_NONFINITE)) ? 0 : ctr->n_nodes;
}

// ---- chunked receivers: chunk c of a receiver applies its partial sums after
// chunk c - 1 (which an earlier warp took). Lane 0 waits, bounded, for the
// receiver's counter to reach c; the warp barrier passes the ordering on.
__device__ __forceinline__ void wait_turn(int *flag, int want, DevCounters *ctr)
{
    if ((threadIdx.x & 31) == 0) {
        cuda::atomic_ref<int, cuda::thread_scope_device> r(*flag);
        unsigned spins = 0;
        while (r.load(cuda::memory_order_acquire) != want) {
            if (++spins > kTurnSpinLimit) {
                set_error(ctr, ERR_SPIN);
                break;
            }
            __nanosleep(spins < 4096 ? 64 : 1024);
        }
    }
    __syncwarp();
}

// After every lane's writes of chunk c: publish them and pass the turn on.
__device__ __forceinline__ void pass_turn(int *flag, int next)
{
    __threadfence();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        cuda::atomic_ref<int, cuda::thread_scope_device> r(*flag);
        r.store(next, cuda::memory_order_release);
    }
}

// ---- grid-wide barrier of a cooperative launch (all blocks co-resident) -----
// One arrival counter per launch, on its own 128-byte line; it only grows:
// barrier number k of a kernel completes when it reaches (k + 1) * gridDim.x.
// Thread 0 of each block arrives with release semantics (after the block
// barrier, so it publishes the whole block's writes) and waits with acquire
// loads, bounded; the block barrier then passes the ordering on to the block's
// other threads. Returns false, with ERR_SPIN set, if the wait gave up; every
// block's wait is bounded the same way. (A two-level arrival tree measured no
// faster at these grid sizes.)
struct __align__(128) GridBarrier {
    unsigned count;
    unsigned pad[31];
};

__device__ __forceinline__ bool grid_barrier(GridBarrier *gb, unsigned k, DevCounters *ctr)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        cuda::atomic_ref<unsigned, cuda::thread_scope_device> c(gb->count);
        c.fetch_add(1u, cuda::memory_order_release);
        const unsigned target = (k + 1) * gridDim.x;
        unsigned spins = 0;
        while (c.load(cuda::memory_order_acquire) < target) {
            if (++spins > (1u << 22)) {
                set_error(ctr, ERR_SPIN);
                ok = 0;
                break;
            }
            __nanosleep(20);
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// ---- chained scan with decoupled look-back ---------------------------------
// Flag word: [63:40] epoch, [39:38] state (1 = aggregate, 2 = inclusive prefix), [37:0] value.
constexpr unsigned long long kFlagValueMask = (1ull << 38) - 1;

__device__ __forceinline__ unsigned long long flag_pack(unsigned epoch, unsigned state, unsigned long long v)
{
    return ((unsigned long long)(epoch & 0xffffffu) << 40) | ((unsigned long long)state << 38) | (v & kFlagValueMask);
}

__device__ __forceinline__ void flag_store(unsigned long long *p, unsigned long long v)
{
    cuda::atomic_ref<unsigned long long, cuda::thread_scope_device> r(*p);
    r.store(v, cuda::memory_order_release);
}

__device__ __forceinline__ unsigned long long flag_load(unsigned long long *p)
{
    cuda::atomic_ref<unsigned long long, cuda::thread_scope_device> r(*p);
    return r.load(cuda::memory_order_acquire);
}

// Relaxed flag read: the flag word carries its value, nothing else is read on
// its strength, so no acquire ordering is needed (and several can be in flight).
__device__ __forceinline__ unsigned long long flag_load_relaxed(unsigned long long *p)
{
    cuda::atomic_ref<unsigned long long, cuda::thread_scope_device> r(*p);
    return r.load(cuda::memory_order_relaxed);
}

// Exclusive prefix of `aggregate` over the tiles before `tile` in one chained
// scan. flags[t * stride] is tile t's word. Called by one thread per scanned
// quantity. Every tile with a lower index was taken earlier from the same ticket
// counter, so it is running or done and the wait ends; the spin is bounded all the
// same and reports ERR_SPIN (returning a partial prefix) if it ever gives up.
__device__ __forceinline__ unsigned long long chained_exclusive(unsigned long long *flags, int stride, int tile,
                                                                unsigned long long aggregate, unsigned epoch,
                                                                DevCounters *ctr)
{
    if (tile == 0) {
        flag_store(flags, flag_pack(epoch, 2, aggregate));
        return 0;
    }
    flag_store(flags + (size_t)tile * stride, flag_pack(epoch, 1, aggregate));
    unsigned long long excl = 0;
    int t = tile - 1;
    unsigned spins = 0;
    const unsigned long long ep = (unsigned long long)(epoch & 0xffffffu);
    while (t >= 0) {
        unsigned long long f = flag_load(flags + (size_t)t * stride);
        unsigned state = (unsigned)((f >> 38) & 3u);
        if ((f >> 40) != ep || state == 0) {
            if (++spins > kSpinLimit) {
                set_error(ctr, ERR_SPIN);
                break;
            }
            continue;
        }
        excl += f & kFlagValueMask;
        if (state == 2) break;
        --t;
    }
    flag_store(flags + (size_t)tile * stride, flag_pack(epoch, 2, excl + aggregate));
    return excl;
}

// The same exclusive prefix for one thread, reading W predecessors' flags per
// round (independent loads, so one round costs about one load latency): their
// values are added from the nearest back until an inclusive prefix; a flag not
// yet published ends the round and the next round starts at it. Bounded like
// chained_exclusive.
template <int W>
__device__ __forceinline__ unsigned long long chained_exclusive_wide(unsigned long long *flags, int stride, int tile,
                                                                     unsigned long long aggregate, unsigned epoch,
                                                                     DevCounters *ctr)
{
    if (tile == 0) {
        flag_store(flags, flag_pack(epoch, 2, aggregate));
        return 0;
    }
    flag_store(flags + (size_t)tile * stride, flag_pack(epoch, 1, aggregate));
    unsigned long long excl = 0;
    int t = tile - 1;
    unsigned spins = 0;
    const unsigned long long ep = (unsigned long long)(epoch & 0xffffffu);
    while (t >= 0) {
        unsigned long long f[W];
#pragma unroll
        for (int i = 0; i < W; ++i) f[i] = t - i >= 0 ? flag_load_relaxed(flags + (size_t)(t - i) * stride) : 0ull;
        bool done = false, stalled = false;
#pragma unroll
        for (int i = 0; i < W; ++i) {
            if (done || stalled || t < 0) continue;
            const unsigned state = (unsigned)((f[i] >> 38) & 3u);
            if ((f[i] >> 40) != ep || state == 0) {
                stalled = true;
                continue;
            }
            excl += f[i] & kFlagValueMask;
            if (state == 2) done = true;
            --t;
        }
        if (done) break;
        if (stalled && ++spins > kSpinLimit) {
            set_error(ctr, ERR_SPIN);
            break;
        }
    }
    flag_store(flags + (size_t)tile * stride, flag_pack(epoch, 2, excl + aggregate));
    return excl;
}

// The same exclusive prefix computed by a whole warp (every lane calls it, lane
// 0's `aggregate` counts): each round reads 32 W predecessors' flags at once
// (lane l, slot k holds tile - 1 - l - 32 k; relaxed loads, the flag carries
// its value) and adds them up to the nearest inclusive prefix, so the look-back
// advances 32 W tiles per round without an inclusive prefix -- and, when all
// tiles run at once, inclusive prefixes spread 32 W tiles per round. Returns
// the prefix to every lane. Bounded like chained_exclusive.
template <int W = 1>
__device__ __forceinline__ unsigned long long chained_exclusive_warp(unsigned long long *flags, int stride, int tile,
                                                                     unsigned long long aggregate, unsigned epoch,
                                                                     DevCounters *ctr)
{
    const int lane = threadIdx.x & 31;
    if (tile == 0) {
        if (lane == 0) flag_store(flags, flag_pack(epoch, 2, aggregate));
        return 0;
    }
    if (lane == 0) flag_store(flags + (size_t)tile * stride, flag_pack(epoch, 1, aggregate));
    const unsigned long long ep = (unsigned long long)(epoch & 0xffffffu);
    unsigned long long excl = 0;
    int t = tile - 1;
    unsigned spins = 0;
    for (;;) {
        unsigned state[W];
        unsigned long long v[W];
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const int idx = t - lane - 32 * k;
            state[k] = 2;  // before tile 0: an inclusive prefix of 0
            v[k] = 0;
            if (idx >= 0) {
                const unsigned long long f = flag_load_relaxed(flags + (size_t)idx * stride);
                state[k] = (f >> 40) == ep ? (unsigned)((f >> 38) & 3u) : 0u;
                v[k] = f & kFlagValueMask;
            }
        }
        // nearest inclusive prefix in the window: slot kstop, lane stop
        int kstop = W, stop = 31;
#pragma unroll
        for (int k = W - 1; k >= 0; --k) {
            const unsigned incl = __ballot_sync(kFull, state[k] == 2);
            if (incl) {
                kstop = k;
                stop = __ffs(incl) - 1;
            }
        }
        bool wait = false;
#pragma unroll
        for (int k = 0; k < W; ++k) {
            const unsigned need = k < kstop ? kFull : (k == kstop ? (stop == 31 ? kFull : ((2u << stop) - 1u)) : 0u);
            wait |= (__ballot_sync(kFull, state[k] == 0) & need) != 0u;
        }
        if (wait) {
            if (++spins > kSpinLimit) {
                if (lane == 0) set_error(ctr, ERR_SPIN);
                break;
            }
            continue;
        }
        unsigned long long sum = 0;
#pragma unroll
        for (int k = 0; k < W; ++k)
            if (k < kstop || (k == kstop && lane <= stop)) sum += v[k];
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
        excl += sum;
        if (kstop < W) break;
        t -= 32 * W;
    }
    if (lane == 0) flag_store(flags + (size_t)tile * stride, flag_pack(epoch, 2, excl + aggregate));
    return excl;
}

// ---- warp helpers ------------------------------------------------------------
__device__ __forceinline__ unsigned lanemask_lt()
{
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <class T> __device__ __forceinline__ T warp_sum_xor(T v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// inclusive scan over the warp of an int
__device__ __forceinline__ int warp_incl_scan(int v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(kFull, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Sum v over the 32 lanes and hand the NC sums to store(k, sum): three halving
// steps (offsets 16, 8, 4) leave each lane NR/8 partial sums of its own
// coefficient block, two butterfly steps (2, 1) finish them; lane 4 j then
// stores its block. Fixed order, so reproducible, and the same lane always
// stores the same k.
template <class T, int NR, int NC, class F>
__device__ __forceinline__ void reduce_apply(T (&v)[NR], int lane, F &&store)
{
    constexpr int H1 = NR / 2, H2 = NR / 4, H3 = NR / 8;
    T a[H1], b[H2], c[H3];
    const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4;
#pragma unroll
    for (int i = 0; i < H1; ++i) {
        const T send = u4 ? v[i] : v[i + H1], keep = u4 ? v[i + H1] : v[i];
        a[i] = keep + __shfl_xor_sync(kFull, send, 16);
    }
#pragma unroll
    for (int i = 0; i < H2; ++i) {
        const T send = u3 ? a[i] : a[i + H2], keep = u3 ? a[i + H2] : a[i];
        b[i] = keep + __shfl_xor_sync(kFull, send, 8);
    }
#pragma unroll
    for (int i = 0; i < H3; ++i) {
        const T send = u2 ? b[i] : b[i + H3], keep = u2 ? b[i + H3] : b[i];
        c[i] = keep + __shfl_xor_sync(kFull, send, 4);
    }
#pragma unroll
    for (int i = 0; i < H3; ++i) {
        c[i] += __shfl_xor_sync(kFull, c[i], 2);
        c[i] += __shfl_xor_sync(kFull, c[i], 1);
    }
    if ((lane & 3) == 0) {
        const int base = (u4 ? H1 : 0) + (u3 ? H2 : 0) + (u2 ? H3 : 0);
#pragma unroll
        for (int i = 0; i < H3; ++i)
            if (base + i < NC) store(base + i, c[i]);
    }
}

// The same over the 8 lanes of an aligned lane group (j = lane & 7): three
// halving steps (offsets 4, 2, 1) leave lane j the NR/8 sums of its block.
template <class T, int NR, int NC, class F>
__device__ __forceinline__ void reduce_apply8(T (&v)[NR], int j, F &&store)
{
    constexpr int H1 = NR / 2, H2 = NR / 4, H3 = NR / 8;
    T a[H1], b[H2], c[H3];
    const bool u4 = j & 4, u2 = j & 2, u1 = j & 1;
#pragma unroll
    for (int i = 0; i < H1; ++i) {
        const T send = u4 ? v[i] : v[i + H1], keep = u4 ? v[i + H1] : v[i];
        a[i] = keep + __shfl_xor_sync(kFull, send, 4);
    }
#pragma unroll
    for (int i = 0; i < H2; ++i) {
        const T send = u2 ? a[i] : a[i + H2], keep = u2 ? a[i + H2] : a[i];
        b[i] = keep + __shfl_xor_sync(kFull, send, 2);
    }
#pragma unroll
    for (int i = 0; i < H3; ++i) {
        const T send = u1 ? b[i] : b[i + H3], keep = u1 ? b[i + H3] : b[i];
        c[i] = keep + __shfl_xor_sync(kFull, send, 1);
    }
    const int base = (u4 ? H1 : 0) + (u2 ? H2 : 0) + (u1 ? H3 : 0);
#pragma unroll
    for (int i = 0; i < H3; ++i)
        if (base + i < NC) store(base + i, c[i]);
}

template <class T, int NR, int NC>
__device__ __forceinline__ void reduce_store(T (&v)[NR], int lane, T *__restrict__ dst)
{
    reduce_apply<T, NR, NC>(v, lane, [dst](int k, const T &x) { dst[k] = x; });
}

template <class T> __device__ __forceinline__ T pos_inf();
template <> __device__ __forceinline__ float pos_inf<float>() { return __int_as_float(0x7f800000); }
template <> __device__ __forceinline__ double pos_inf<double>() { return __longlong_as_double(0x7ff0000000000000ll); }

// Asynchronous global-to-shared copies (cp.async, L1-allocating): a warp's
// staging issues every copy of a tile before waiting once, instead of paying
// one load latency per 32 elements (a load, then a store that waits for it).
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst_smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(dst_smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 16;\n" ::"r"(d), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Groups of asynchronous copies: commit closes the thread's copies issued so
// far into a group; wait_group<N> returns once at most N of the thread's
// groups are still in flight (so with one group per pipeline stage, N = 1
// waits for all but the newest).
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace bfm
