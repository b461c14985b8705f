// Downward pass: L2L level by level, then L2P + P2P at the leaves.
//
// JZ-FMM page, "Combining near and far interactions", stage 3: translate each
// parent's local Taylor expansion to its children, evaluate the expansions at
// the particle positions (Taylor eq.: Phi(c + dx) = sum_k L_k dx^k / k!,
// a = -grad Phi) and calculate the remaining nearby interactions directly
// (direct gravity eq.: Phi_i += -G m_j / r, a_i += G m_j (x_j - x_i) / r^3,
// skipping zero separations, i.e. the particle itself).
//
// Leaf kernel: one warp per leaf, a lane per receiving particle; the particles
// of every source leaf in the P2P list are staged through shared memory 32 at a
// time and read back as warp-wide broadcasts. Results are written straight to
// the caller's particle order.
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
    rinv = r2 > T(0) ? rinv : T(0);
    const T mr = s.w * rinv;
    const T mr3 = mr * rinv * rinv;
    ax += mr3 * dx;
    ay += mr3 * dy;
    az += mr3 * dz;
    phi -= mr;
}

template <class T, int P>
__global__ __launch_bounds__(256) void k_leaf(int n_nodes, const int *__restrict__ first, const int *__restrict__ count,
                                              const int *__restrict__ nchild, const vec4<T> *__restrict__ xyzm,
                                              const uint32_t *__restrict__ perm, const vec4<T> *__restrict__ nc,
                                              const T *__restrict__ L, int ncp, const int *__restrict__ off,
                                              const int *__restrict__ src, T *__restrict__ acc, T *__restrict__ pot)
{
    __shared__ vec4<T> s_src[8][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a];
        const vec4<T> ca = nc[a];
        const int beg = off[a], end = off[a + 1];
        for (int r0 = 0; r0 < c; r0 += 32) {
            const bool active = r0 + lane < c;
            const int i = f + r0 + (active ? lane : 0);
            const vec4<T> q = xyzm[i];
            T phi = T(0), ax = T(0), ay = T(0), az = T(0);
            Exp<P>::template l2p<T>(L + (size_t)a * ncp, q.x - ca.x, q.y - ca.y, q.z - ca.z, phi, ax, ay, az);
            for (int e = beg; e < end; ++e) {
                const int b = src[e];
                const int fb = first[b], cb = count[b];
                for (int s0 = 0; s0 < cb; s0 += 32) {
                    __syncwarp();
                    if (s0 + lane < cb) s_src[w][lane] = xyzm[fb + s0 + lane];
                    __syncwarp();
                    const int ns = cb - s0 < 32 ? cb - s0 : 32;
                    if (ns == 32) {
#pragma unroll 8
                        for (int k = 0; k < 32; ++k) p2p_one<T>(s_src[w][k], q.x, q.y, q.z, phi, ax, ay, az);
                    } else {
                        for (int k = 0; k < ns; ++k) p2p_one<T>(s_src[w][k], q.x, q.y, q.z, phi, ax, ay, az);
                    }
                }
            }
            if (active) {
                const uint32_t o = perm[i];
                acc[3 * (size_t)o] = ax;
                acc[3 * (size_t)o + 1] = ay;
                acc[3 * (size_t)o + 2] = az;
                if (pot) pot[o] = phi;
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
    k_leaf<T, P><<<P_.num_sms * 8, 256, 0, s>>>((int)P_.n_nodes, P_.node_first, P_.node_count, P_.node_nchild,
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
