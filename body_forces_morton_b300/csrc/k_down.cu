// Downward pass: L2L level by level, then L2P + P2P at the leaves.
//
// JZ-FMM page, "Combining near and far interactions", stage 3: translate each
// parent's local Taylor expansion to its children, evaluate the expansions at
// the particle positions (Taylor eq.: Phi(c + dx) = sum_k L_k dx^k / k!,
// a = -grad Phi) and calculate the remaining nearby interactions directly
// (direct gravity eq.: Phi_i += -G m_j / r, a_i += G m_j (x_j - x_i) / r^3,
// skipping zero separations, i.e. the particle itself).
//
// Leaf kernel: one warp per receiving leaf. The particles of its source leaves
// are staged through shared memory (32 list entries and up to a chunk of
// particles at a time) and read back as warp-wide broadcasts; the lane mapping
// keeps all 32 lanes busy for small leaves by splitting the sources. Results
// are written straight to the caller's particle order.
#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

template <class T, int P>
__global__ __launch_bounds__(256) void k_l2l(int level, const DevCounters *__restrict__ ctr,
                                             const int *__restrict__ parent, const vec4<T> *__restrict__ nc,
                                             const T *__restrict__ Lm2l, T *__restrict__ L, int ncp)
{
    constexpr int NC = Exp<P>::NC;
    const int lo = ctr->level_off[level], hi = ctr->level_off[level + 1];
    for (int a = lo + blockIdx.x * blockDim.x + threadIdx.x; a < hi; a += gridDim.x * blockDim.x) {
        T out[NC];
        const T *own = Lm2l + (size_t)a * ncp;
#pragma unroll
        for (int k = 0; k < NC; ++k) out[k] = own[k];
        if (level > 0) {
            const int par = parent[a];
            T lp[NC];
            const T *pr = L + (size_t)par * ncp;
#pragma unroll
            for (int k = 0; k < NC; ++k) lp[k] = pr[k];
            const vec4<T> c = nc[a], cp = nc[par];
            Exp<P>::template l2l<T>(lp, c.x - cp.x, c.y - cp.y, c.z - cp.z, out);
        }
        T *dst = L + (size_t)a * ncp;
#pragma unroll
        for (int k = 0; k < NC; ++k) dst[k] = out[k];
    }
}

template <class T>
__device__ __forceinline__ void p2p_one(const vec4<T> &s, T x, T y, T z, T &phi, T &ax, T &ay, T &az)
{
    const T dx = s.x - x, dy = s.y - y, dz = s.z - z;
    const T r2 = dx * dx + dy * dy + dz * dz;
    T rinv = rsqrt_t(r2);
    rinv = r2 > T(0) ? rinv : T(0);  // zero separation: the particle itself (or an exact duplicate)
    const T mr = s.w * rinv;
    const T mr3 = mr * rinv * rinv;
    ax += mr3 * dx;
    ay += mr3 * dy;
    az += mr3 * dz;
    phi -= mr;
}

constexpr int LF_WARPS = 4;                            // warps per block of the leaf kernel
template <class T> struct LeafChunk { static constexpr int value = 256; };   // staged source particles per warp
template <> struct LeafChunk<double> { static constexpr int value = 128; };

// Stage up to CH particles of the concatenated source leaves [g0, g0 + CH) of
// the current group of (at most 32) list entries into shared memory.
// Lane i holds the group's i-th leaf: first particle fb, count cb, exclusive
// prefix ex of the counts.
template <class T, int CH>
__device__ __forceinline__ int stage_sources(vec4<T> *buf, const vec4<T> *__restrict__ xyzm, int fb, int ex,
                                             int tot, int g0, int lane)
{
    const int n_here = min(CH, tot - g0);
    for (int k0 = 0; k0 < n_here; k0 += 32) {  // warp-uniform: every lane takes part in the shuffles
        const int k = k0 + lane;
        const int g = g0 + k;
        // the leaf holding particle g of the group: last lane with ex <= g (ex ascends over the lanes)
        int lo = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const int exm = __shfl_sync(kFull, ex, lo + step);
            lo = exm <= g ? lo + step : lo;
        }
        const int f = __shfl_sync(kFull, fb, lo);
        const int e = __shfl_sync(kFull, ex, lo);
        if (k < n_here) buf[k] = xyzm[f + (g - e)];
    }
    return n_here;
}

// L2P + P2P for one receiver leaf per warp.
//  count <= 32: lane = (r, q), r < 2^k >= count the receiver, q one of 32 / 2^k
//               source strides; the strides are summed by a fixed butterfly.
//  count > 32:  each lane takes receivers lane and lane + 32 of a 64-particle
//               round, so every staged source feeds two interactions.
template <class T, int P>
__global__ __launch_bounds__(LF_WARPS * 32) void k_leaf(int n_nodes, const int *__restrict__ first,
                                                        const int *__restrict__ count,
                                                        const int *__restrict__ nchild,
                                                        const vec4<T> *__restrict__ xyzm,
                                                        const uint32_t *__restrict__ perm,
                                                        const vec4<T> *__restrict__ nc, const T *__restrict__ L,
                                                        int ncp, const int *__restrict__ off,
                                                        const int *__restrict__ src, T *__restrict__ acc,
                                                        T *__restrict__ pot)
{
    constexpr int CH = LeafChunk<T>::value;
    __shared__ vec4<T> s_src[LF_WARPS][CH];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    vec4<T> *buf = s_src[w];
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a];
        const vec4<T> ca = nc[a];
        const int beg = off[a], end = off[a + 1];
        const T *La = L + (size_t)a * ncp;
        if (c <= 32) {
            int lg = 0;
            while ((1 << lg) < c) ++lg;
            const int r = lane & ((1 << lg) - 1), q = lane >> lg, S = 32 >> lg;
            const bool active = r < c;
            const vec4<T> pi = xyzm[f + (active ? r : 0)];
            T phi = T(0), ax = T(0), ay = T(0), az = T(0);
            for (int lb = beg; lb < end; lb += 32) {
                const int e = lb + lane;
                int fb = 0, cb = 0;
                if (e < end) {
                    const int b = src[e];
                    fb = first[b];
                    cb = count[b];
                }
                const int incl = warp_incl_scan(cb);
                const int tot = __shfl_sync(kFull, incl, 31);
                const int ex = incl - cb;
                for (int g0 = 0; g0 < tot; g0 += CH) {
                    __syncwarp();
                    const int n_here = stage_sources<T, CH>(buf, xyzm, fb, ex, tot, g0, lane);
                    __syncwarp();
                    int j = q;
                    for (; j + 3 * S < n_here; j += 4 * S) {
                        p2p_one<T>(buf[j], pi.x, pi.y, pi.z, phi, ax, ay, az);
                        p2p_one<T>(buf[j + S], pi.x, pi.y, pi.z, phi, ax, ay, az);
                        p2p_one<T>(buf[j + 2 * S], pi.x, pi.y, pi.z, phi, ax, ay, az);
                        p2p_one<T>(buf[j + 3 * S], pi.x, pi.y, pi.z, phi, ax, ay, az);
                    }
                    for (; j < n_here; j += S) p2p_one<T>(buf[j], pi.x, pi.y, pi.z, phi, ax, ay, az);
                }
            }
            // sum the source strides: lanes with the same r, fixed order
            for (int o = 1 << lg; o < 32; o <<= 1) {
                phi += __shfl_xor_sync(kFull, phi, o);
                ax += __shfl_xor_sync(kFull, ax, o);
                ay += __shfl_xor_sync(kFull, ay, o);
                az += __shfl_xor_sync(kFull, az, o);
            }
            if (active && q == 0) {
                Exp<P>::template l2p<T>(La, pi.x - ca.x, pi.y - ca.y, pi.z - ca.z, phi, ax, ay, az);
                const uint32_t o = perm[f + r];
                acc[3 * (size_t)o] = ax;
                acc[3 * (size_t)o + 1] = ay;
                acc[3 * (size_t)o + 2] = az;
                if (pot) pot[o] = phi;
            }
        } else {
            for (int r0 = 0; r0 < c; r0 += 64) {
                const bool act0 = r0 + lane < c, act1 = r0 + 32 + lane < c;
                const vec4<T> p0 = xyzm[f + r0 + (act0 ? lane : 0)];
                const vec4<T> p1 = xyzm[f + r0 + (act1 ? 32 + lane : 0)];
                T phi0 = T(0), ax0 = T(0), ay0 = T(0), az0 = T(0);
                T phi1 = T(0), ax1 = T(0), ay1 = T(0), az1 = T(0);
                for (int lb = beg; lb < end; lb += 32) {
                    const int e = lb + lane;
                    int fb = 0, cb = 0;
                    if (e < end) {
                        const int b = src[e];
                        fb = first[b];
                        cb = count[b];
                    }
                    const int incl = warp_incl_scan(cb);
                    const int tot = __shfl_sync(kFull, incl, 31);
                    const int ex = incl - cb;
                    for (int g0 = 0; g0 < tot; g0 += CH) {
                        __syncwarp();
                        const int n_here = stage_sources<T, CH>(buf, xyzm, fb, ex, tot, g0, lane);
                        __syncwarp();
                        int j = 0;
                        for (; j + 1 < n_here; j += 2) {
                            const vec4<T> s0 = buf[j], s1 = buf[j + 1];
                            p2p_one<T>(s0, p0.x, p0.y, p0.z, phi0, ax0, ay0, az0);
                            p2p_one<T>(s0, p1.x, p1.y, p1.z, phi1, ax1, ay1, az1);
                            p2p_one<T>(s1, p0.x, p0.y, p0.z, phi0, ax0, ay0, az0);
                            p2p_one<T>(s1, p1.x, p1.y, p1.z, phi1, ax1, ay1, az1);
                        }
                        if (j < n_here) {
                            p2p_one<T>(buf[j], p0.x, p0.y, p0.z, phi0, ax0, ay0, az0);
                            p2p_one<T>(buf[j], p1.x, p1.y, p1.z, phi1, ax1, ay1, az1);
                        }
                    }
                }
                if (act0) {
                    Exp<P>::template l2p<T>(La, p0.x - ca.x, p0.y - ca.y, p0.z - ca.z, phi0, ax0, ay0, az0);
                    const uint32_t o = perm[f + r0 + lane];
                    acc[3 * (size_t)o] = ax0;
                    acc[3 * (size_t)o + 1] = ay0;
                    acc[3 * (size_t)o + 2] = az0;
                    if (pot) pot[o] = phi0;
                }
                if (act1) {
                    Exp<P>::template l2p<T>(La, p1.x - ca.x, p1.y - ca.y, p1.z - ca.z, phi1, ax1, ay1, az1);
                    const uint32_t o = perm[f + r0 + 32 + lane];
                    acc[3 * (size_t)o] = ax1;
                    acc[3 * (size_t)o + 1] = ay1;
                    acc[3 * (size_t)o + 2] = az1;
                    if (pot) pot[o] = phi1;
                }
            }
        }
    }
}

template <class T, int P>
int launch_l2l_tp(Plan &P_, int depth, cudaStream_t s)
{
    for (int level = 0; level <= depth; ++level)
        k_l2l<T, P><<<P_.num_sms * 4, 256, 0, s>>>(level, P_.ctr, P_.node_parent, (const vec4<T> *)P_.node_c,
                                                   (const T *)P_.Lm2l, (T *)P_.L, P_.ncp);
    return depth + 1;
}

template <class T, int P>
int launch_leaf_tp(Plan &P_, void *acc, void *pot, cudaStream_t s)
{
    k_leaf<T, P><<<P_.num_sms * 16, LF_WARPS * 32, 0, s>>>((int)P_.n_nodes, P_.node_first, P_.node_count, P_.node_nchild,
                                                (const vec4<T> *)P_.xyzm, P_.idx[0], (const vec4<T> *)P_.node_c,
                                                (const T *)P_.L, P_.ncp, P_.p2p_off, P_.p2p_src, (T *)acc, (T *)pot);
    return 1;
}

#define BFM_DISPATCH_P(fn, T, ...)                        \
    switch (P.p) {                                        \
    case 0: return fn<T, 0>(P, __VA_ARGS__);              \
    case 1: return fn<T, 1>(P, __VA_ARGS__);              \
    case 2: return fn<T, 2>(P, __VA_ARGS__);              \
    case 3: return fn<T, 3>(P, __VA_ARGS__);              \
    case 4: return fn<T, 4>(P, __VA_ARGS__);              \
    case 5: return fn<T, 5>(P, __VA_ARGS__);              \
    case 6: return fn<T, 6>(P, __VA_ARGS__);              \
    case 7: return fn<T, 7>(P, __VA_ARGS__);              \
    default: return fn<T, 8>(P, __VA_ARGS__);             \
    }

template <class T> int launch_l2l_t(Plan &P, int depth, cudaStream_t s) { BFM_DISPATCH_P(launch_l2l_tp, T, depth, s) }
template <class T> int launch_leaf_t(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    BFM_DISPATCH_P(launch_leaf_tp, T, acc, pot, s)
}

}  // namespace

int launch_l2l(Plan &P, int depth, cudaStream_t s)
{
    return P.dtype == 0 ? launch_l2l_t<float>(P, depth, s) : launch_l2l_t<double>(P, depth, s);
}

int launch_leaf(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    return P.dtype == 0 ? launch_leaf_t<float>(P, acc, pot, s) : launch_leaf_t<double>(P, acc, pot, s);
}

}  // namespace bfm
