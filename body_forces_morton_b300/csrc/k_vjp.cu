// Vector-Jacobian product of one FMM evaluation.
//
// JZ-FMM page, "Differentiating the force calculation": the VJP of the FMM
// has one contribution from the next higher derivative of the original
// evaluation and one from an FMM in which the force sensitivities act as
// dipole moments. With cotangents abar_i (accelerations) and pbar_i
// (potentials, optional) the loss sensitivities are
//   xbar_k = m_k grad Phi_s(x_k) - Hess Phi(x_k) abar_k - pbar_k a_k,
//   mbar_k = Phi_s(x_k),
// with Phi the forward potential and Phi_s the potential of sources at every
// particle with monopole pbar_j and dipole -abar_j. Both run on the forward
// evaluation's tree, centres and lists, so these are the exact derivatives of
// the evaluation with the tree and the expansion centres held fixed (the pair
// kernel of the total-degree truncation is symmetric in its two particles).
//
// Stages after the forward evaluation (which leaves the tree, the lists, the
// complete forward locals L and the accelerations):
//   k_vjp_sources   the cotangents in the tree's particle order, as the
//                   sources' (monopole, dipole) = (pbar, -abar);
//   k_vjp_up        per level, deepest first: a leaf's moments from its
//                   particles (Exp<P>::p2m_dip), an internal node's from its
//                   children (m2m), in a fixed order;
//   M2L and L2L     the forward kernels on the source moments (plain
//                   arithmetic in the plan's dtype);
//   k_vjp_leaf      per leaf, a lane per particle: Phi_s and its gradient from
//                   the source locals, the forward Hessian from L
//                   (Exp<P>::l2p_hess), plus the direct terms of every pair in
//                   the leaf's P2P list, sources staged in shared memory; the
//                   result combined as above and written in the caller's order.
#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

constexpr int VJP_WARPS = 4;
constexpr int VJP_CH = 64;  // staged source particles per warp

template <class T>
__global__ __launch_bounds__(256) void k_vjp_sources(int n, const uint32_t *__restrict__ perm,
                                                     const T *__restrict__ abar, const T *__restrict__ pbar,
                                                     vec4<T> *__restrict__ src)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t o = perm[i];
        src[i] = make4<T>(pbar ? pbar[o] : T(0), -abar[3 * (size_t)o], -abar[3 * (size_t)o + 1],
                          -abar[3 * (size_t)o + 2]);
    }
}

// Source moments of the nodes of one level (a thread per node).
template <class T, int P>
__global__ __launch_bounds__(128) void k_vjp_up(const DevCounters *__restrict__ ctr, int level,
                                                const int *__restrict__ first, const int *__restrict__ count,
                                                const int *__restrict__ child0, const int *__restrict__ nchild,
                                                const vec4<T> *__restrict__ nc, const vec4<T> *__restrict__ xyzm,
                                                const vec4<T> *__restrict__ src, T *__restrict__ Ms, int ncp)
{
    constexpr int NC = Exp<P>::NC;
    const int n_nodes = phase2_nodes(ctr);
    const int lo = min(ctr->level_off[level], n_nodes), hi = min(ctr->level_off[level + 1], n_nodes);
    for (int a = lo + blockIdx.x * blockDim.x + threadIdx.x; a < hi; a += gridDim.x * blockDim.x) {
        T M[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) M[k] = T(0);
        const vec4<T> c = nc[a];
        const int nch = nchild[a];
        if (nch == 0) {
            const int f = first[a], e = f + count[a];
            for (int i = f; i < e; ++i) {
                const vec4<T> x = xyzm[i], s = src[i];
                Exp<P>::template p2m_dip<T>(x.x - c.x, x.y - c.y, x.z - c.z, s.x, s.y, s.z, s.w, M);
            }
        } else {
            const int c0 = child0[a];
            for (int ch = c0; ch < c0 + nch; ++ch) {
                const vec4<T> cc = nc[ch];
                Exp<P>::template m2m<T>(Ms + (size_t)ch * ncp, cc.x - c.x, cc.y - c.y, cc.z - c.z, M);
            }
        }
        T *dst = Ms + (size_t)a * ncp;
#pragma unroll
        for (int k = 0; k < NC; ++k) dst[k] = M[k];
    }
}

// The leaves: a warp per leaf, a lane per receiving particle (rounds of 32).
template <class T, int P>
__global__ __launch_bounds__(VJP_WARPS * 32) void k_vjp_leaf(
    const DevCounters *__restrict__ ctr, const int *__restrict__ first, const int *__restrict__ count,
    const int *__restrict__ nchild, const vec4<T> *__restrict__ nc, const vec4<T> *__restrict__ xyzm,
    const vec4<T> *__restrict__ src, const uint32_t *__restrict__ perm, const T *__restrict__ L,
    const T *__restrict__ Ls, int ncp, const int *__restrict__ off, const int *__restrict__ lsrc,
    const T *__restrict__ acc_fwd, T *__restrict__ pos_bar, T *__restrict__ mass_bar)
{
    __shared__ vec4<T> s_x[VJP_WARPS][VJP_CH];
    __shared__ vec4<T> s_s[VJP_WARPS][VJP_CH];
    const int n_nodes = phase2_nodes(ctr);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a];
        const vec4<T> ca = nc[a];
        const int beg = off[a], end = off[a + 1];
        for (int r0 = 0; r0 < c; r0 += 32) {
            const int i = f + r0 + lane;
            const bool mine = r0 + lane < c;
            const vec4<T> xi = xyzm[mine ? i : f];
            const T dx = xi.x - ca.x, dy = xi.y - ca.y, dz = xi.z - ca.z;
            // far field: Phi_s and -grad Phi_s from the source locals, the forward Hessian from L
            T phis = T(0), ngx = T(0), ngy = T(0), ngz = T(0);
            Exp<P>::template l2p<T>(Ls + (size_t)a * ncp, dx, dy, dz, phis, ngx, ngy, ngz);
            T H[6] = {T(0), T(0), T(0), T(0), T(0), T(0)};
            Exp<P>::template l2p_hess<T>(L + (size_t)a * ncp, dx, dy, dz, H);
            T gx = -ngx, gy = -ngy, gz = -ngz;
            // near field over the leaf's P2P list (the leaf itself included; zero separations skipped)
            for (int q = beg; q < end; ++q) {
                const int b = lsrc[q];
                const int fb = first[b], cb = count[b];
                for (int g0 = 0; g0 < cb; g0 += VJP_CH) {
                    const int nh = min(VJP_CH, cb - g0);
                    __syncwarp();
                    for (int k = lane; k < nh; k += 32) {
                        s_x[w][k] = xyzm[fb + g0 + k];
                        s_s[w][k] = src[fb + g0 + k];
                    }
                    __syncwarp();
                    for (int k = 0; k < nh; ++k) {
                        const vec4<T> xj = s_x[w][k], sj = s_s[w][k];
                        const T ux = xi.x - xj.x, uy = xi.y - xj.y, uz = xi.z - xj.z;
                        const T r2 = ux * ux + uy * uy + uz * uz;
                        if (r2 == T(0)) continue;
                        const T ri = rsqrt_t(r2);
                        const T ir2 = ri * ri, ir3 = ri * ir2, ir5 = ir3 * ir2;
                        // forward: Hessian of -m_j / r is m_j (r^2 delta - 3 u u) / r^5
                        const T m3 = xj.w * ir3, m5 = T(3) * xj.w * ir5;
                        H[0] += m3 - m5 * ux * ux;
                        H[1] -= m5 * ux * uy;
                        H[2] -= m5 * ux * uz;
                        H[3] += m3 - m5 * uy * uy;
                        H[4] -= m5 * uy * uz;
                        H[5] += m3 - m5 * uz * uz;
                        // sources (monopole q = sj.x, dipole d = sj.yzw): Phi_s += -q / r - d.u / r^3,
                        // grad Phi_s += q u / r^3 - d / r^3 + 3 (d.u) u / r^5
                        const T du = sj.y * ux + sj.z * uy + sj.w * uz;
                        phis -= sj.x * ri + du * ir3;
                        const T cu = sj.x * ir3 + T(3) * du * ir5;
                        gx += cu * ux - sj.y * ir3;
                        gy += cu * uy - sj.z * ir3;
                        gz += cu * uz - sj.w * ir3;
                    }
                }
            }
            if (mine) {
                const uint32_t o = perm[i];
                const vec4<T> si = src[i];
                const T abx = -si.y, aby = -si.z, abz = -si.w;  // the particle's own cotangent abar
                const T hx = H[0] * abx + H[1] * aby + H[2] * abz;
                const T hy = H[1] * abx + H[3] * aby + H[4] * abz;
                const T hz = H[2] * abx + H[4] * aby + H[5] * abz;
                const T *ai = acc_fwd + 3 * (size_t)o;
                pos_bar[3 * (size_t)o] = xi.w * gx - hx - si.x * ai[0];
                pos_bar[3 * (size_t)o + 1] = xi.w * gy - hy - si.x * ai[1];
                pos_bar[3 * (size_t)o + 2] = xi.w * gz - hz - si.x * ai[2];
                mass_bar[o] = phis;
            }
        }
    }
}

template <class T, int P>
int launch_vjp_tp(Plan &P_, const void *abar, const void *pbar, void *pos_bar, void *mass_bar, cudaStream_t s)
{
    const int n = (int)P_.n;
    k_vjp_sources<T><<<P_.num_sms * 4, 256, 0, s>>>(n, P_.idx[0], (const T *)abar, (const T *)pbar,
                                                     (vec4<T> *)P_.vjp_src);
    int launches = 1;
    for (int l = P_.depth; l >= 0; --l) {
        k_vjp_up<T, P><<<P_.num_sms * 2, 128, 0, s>>>(P_.ctr, l, P_.node_first, P_.node_count, P_.node_child0,
                                                      P_.node_nchild, (const vec4<T> *)P_.node_c,
                                                      (const vec4<T> *)P_.xyzm, (const vec4<T> *)P_.vjp_src,
                                                      (T *)P_.Ms, P_.ncp);
        ++launches;
    }
    // the M2L and L2L kernels take their receivers from work counters that the forward evaluation
    // ran to the end: start them afresh
    cudaMemsetAsync(P_.ctr->work_ctr, 0, sizeof(P_.ctr->work_ctr), s);
    launches += launch_m2l_plain(P_, P_.Ms, P_.Lsm, s);
    // L2L of the source locals: the forward kernel on the source buffers
    void *fwd_lm2l = P_.Lm2l, *fwd_l = P_.L;
    P_.Lm2l = P_.Lsm;
    P_.L = P_.Ls;
    launches += launch_l2l(P_, P_.depth, s);
    P_.Lm2l = fwd_lm2l;
    P_.L = fwd_l;
    k_vjp_leaf<T, P><<<P_.num_sms * 8, VJP_WARPS * 32, 0, s>>>(
        P_.ctr, P_.node_first, P_.node_count, P_.node_nchild, (const vec4<T> *)P_.node_c, (const vec4<T> *)P_.xyzm,
        (const vec4<T> *)P_.vjp_src, P_.idx[0], (const T *)P_.L, (const T *)P_.Ls, P_.ncp, P_.p2p_off, P_.p2p_src,
        (const T *)P_.vjp_acc, (T *)pos_bar, (T *)mass_bar);
    return launches + 1;
}

template <class T>
int launch_vjp_t(Plan &P, const void *abar, const void *pbar, void *pos_bar, void *mass_bar, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_vjp_tp<T, 0>(P, abar, pbar, pos_bar, mass_bar, s);
    case 1: return launch_vjp_tp<T, 1>(P, abar, pbar, pos_bar, mass_bar, s);
    case 2: return launch_vjp_tp<T, 2>(P, abar, pbar, pos_bar, mass_bar, s);
    case 3: return launch_vjp_tp<T, 3>(P, abar, pbar, pos_bar, mass_bar, s);
    case 4: return launch_vjp_tp<T, 4>(P, abar, pbar, pos_bar, mass_bar, s);
    case 5: return launch_vjp_tp<T, 5>(P, abar, pbar, pos_bar, mass_bar, s);
    case 6: return launch_vjp_tp<T, 6>(P, abar, pbar, pos_bar, mass_bar, s);
    case 7: return launch_vjp_tp<T, 7>(P, abar, pbar, pos_bar, mass_bar, s);
    default: return launch_vjp_tp<T, 8>(P, abar, pbar, pos_bar, mass_bar, s);
    }
}

}  // namespace

int launch_vjp(Plan &P, const void *abar, const void *pbar, void *pos_bar, void *mass_bar, cudaStream_t s)
{
    return P.dtype == 0 ? launch_vjp_t<float>(P, abar, pbar, pos_bar, mass_bar, s)
                        : launch_vjp_t<double>(P, abar, pbar, pos_bar, mass_bar, s);
}

}  // namespace bfm
