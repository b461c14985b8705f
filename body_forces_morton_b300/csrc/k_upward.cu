// Upward pass: node boxes, centres, half-widths, P2M at the leaves and M2M to
// the parents, in one kernel.
//
// JZ-FMM page, "Combining near and far interactions", stage 1: calculate the
// moments of the leaves, then translate and combine the children's moments
// around their parent centres. Moments M_n = sum m s^n / n! about the centre
// c = (lo + hi) / 2 of the node's tight box; l = (hi - lo) / 2 is the per-axis
// half-width of the opening criterion.
//
// fp32 plans: one cooperative launch: first every leaf (a warp each: box, then P2M with a
// fixed butterfly reduction over the lanes), then the internal nodes level by
// level from the deepest up, a grid barrier before each level. A warp takes
// four parents at a time, a lane per child (at most 8): the parent's box is
// the union of the children's boxes and its moments the sum of the children's
// M2M translations, reduced in a fixed order over the 8-lane group.
#include "dfloat.cuh"
#include "expansions_gen.cuh"
#include "plan.h"

#include <algorithm>

namespace bfm {

namespace {

template <class T> __device__ __forceinline__ T tmin(T a, T b) { return b < a ? b : a; }
template <class T> __device__ __forceinline__ T tmax(T a, T b) { return b > a ? b : a; }

template <class T>
__device__ __forceinline__ void store_geometry(int a, const T lo[3], const T hi[3], T *__restrict__ node_lo,
                                               T *__restrict__ node_hi, vec4<T> *__restrict__ nc,
                                               vec4<T> *__restrict__ nl, T c[3], bool writer)
{
    T l[3];
    for (int k = 0; k < 3; ++k) {
        c[k] = mul_rn(add_rn(lo[k], hi[k]), T(0.5));
        l[k] = mul_rn(sub_rn(hi[k], lo[k]), T(0.5));
    }
    if (writer) {
        for (int k = 0; k < 3; ++k) {
            node_lo[3 * a + k] = lo[k];
            node_hi[3 * a + k] = hi[k];
        }
        nc[a] = make4<T>(c[0], c[1], c[2], norm2_rn(l[0], l[1], l[2]));
        nl[a] = make4<T>(l[0], l[1], l[2], T(0));
    }
}

template <int NC> struct Padded { static constexpr int value = (NC + 7) / 8 * 8; };

template <class T, int P>
__global__ __launch_bounds__(256) void k_upward_all(GridBarrier *gb, DevCounters *ctr, const vec4<T> *__restrict__ xyzm,
                                                    const int *__restrict__ first, const int *__restrict__ count,
                                                    const int *__restrict__ child0, const int *__restrict__ nchild,
                                                    T *node_lo, T *node_hi, vec4<T> *nc, vec4<T> *nl, T *M, int ncp)
{
    constexpr int NC = Exp<P>::NC;
    constexpr int NR = Padded<NC>::value;
    const int n_nodes = phase2_nodes(ctr);
    if (n_nodes == 0) return;
    const int depth = ctr->depth;
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    for (int a = wid; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        // ---- leaf: box, centre, P2M
        const int f = first[a], c = count[a];
        T lo[3], hi[3], cen[3];
        for (int k = 0; k < 3; ++k) { lo[k] = pos_inf<T>(); hi[k] = -pos_inf<T>(); }
        for (int i = f + lane; i < f + c; i += 32) {
            vec4<T> q = xyzm[i];
            lo[0] = tmin(lo[0], q.x); hi[0] = tmax(hi[0], q.x);
            lo[1] = tmin(lo[1], q.y); hi[1] = tmax(hi[1], q.y);
            lo[2] = tmin(lo[2], q.z); hi[2] = tmax(hi[2], q.z);
        }
        for (int o = 16; o > 0; o >>= 1)
            for (int k = 0; k < 3; ++k) {
                lo[k] = tmin(lo[k], __shfl_xor_sync(kFull, lo[k], o));
                hi[k] = tmax(hi[k], __shfl_xor_sync(kFull, hi[k], o));
            }
        store_geometry<T>(a, lo, hi, node_lo, node_hi, nc, nl, cen, lane == 0);
        T m[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) m[k] = T(0);
        for (int i = f + lane; i < f + c; i += 32) {
            vec4<T> q = xyzm[i];
            Exp<P>::template p2m<T>(q.x - cen[0], q.y - cen[1], q.z - cen[2], q.w, m);
        }
        reduce_store<T, NR, NC>(m, lane, M + (size_t)a * ncp);
    }
    // ---- internal nodes, deepest level first; the children's data was written by other
    // blocks before the barrier and is read through L2
    const int g = lane >> 3, j = lane & 7;
    for (int level = depth - 1; level >= 0; --level) {
        if (!grid_barrier(gb, (unsigned)(depth - 1 - level), ctr)) return;
        const int lo_l = ctr->level_off[level], hi_l = min(ctr->level_off[level + 1], n_nodes);
        for (int p0 = lo_l + 4 * wid; p0 < hi_l; p0 += 4 * nwarps) {
            const int par = p0 + g;
            const int nch = par < hi_l ? nchild[par] : 0;
            const bool has = j < nch;
            const int ch = has ? child0[par] + j : 0;
            T lo[3], hi[3], cen[3];
            for (int k = 0; k < 3; ++k) {
                lo[k] = has ? ld_cg(node_lo + 3 * ch + k) : pos_inf<T>();
                hi[k] = has ? ld_cg(node_hi + 3 * ch + k) : -pos_inf<T>();
            }
            for (int o = 4; o > 0; o >>= 1)
                for (int k = 0; k < 3; ++k) {
                    lo[k] = tmin(lo[k], __shfl_xor_sync(kFull, lo[k], o));
                    hi[k] = tmax(hi[k], __shfl_xor_sync(kFull, hi[k], o));
                }
            store_geometry<T>(par, lo, hi, node_lo, node_hi, nc, nl, cen, j == 0 && nch > 0);
            T m[NR];
#pragma unroll
            for (int k = 0; k < NR; ++k) m[k] = T(0);
            if (has) {
                T mc[NC];
#pragma unroll
                for (int k = 0; k < NC; ++k) mc[k] = ld_cg(M + (size_t)ch * ncp + k);
                const vec4<T> cc = ld_cg(nc + ch);
                Exp<P>::template m2m<T>(mc, cc.x - cen[0], cc.y - cen[1], cc.z - cen[2], m);
            }
            T *dst = M + (size_t)par * ncp;
            reduce_apply8<T, NR, NC>(m, j, [&](int k, const T &x) {
                if (nch > 0) dst[k] = x;
            });
        }
    }
}

// The fp64 plans' upward pass: one warp per leaf; when a warp finishes a node
// it takes a ticket on the parent, and the warp holding the parent's last
// ticket goes on with the parent (all its children are complete), so no warp
// waits. It keeps the FP64-bound M2M work spread over the whole pass, where
// the level-synchronous kernel would run each level's alone.
template <class T, int P>
__global__ __launch_bounds__(256, 2) void k_upward_ticket(const DevCounters *__restrict__ nctr, const vec4<T> *__restrict__ xyzm,
                                                const int *__restrict__ first, const int *__restrict__ count,
                                                const int *__restrict__ child0, const int *__restrict__ nchild,
                                                const int *__restrict__ parent, int *done, T *node_lo, T *node_hi,
                                                vec4<T> *nc, vec4<T> *nl, T *M, int ncp)
{
    const int n_nodes = phase2_nodes(nctr);
    constexpr int NC = Exp<P>::NC;
    constexpr int NR = Padded<NC>::value;
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        // ---- leaf: box, centre, P2M
        const int f = first[a], c = count[a];
        T lo[3], hi[3], cen[3];
        for (int k = 0; k < 3; ++k) { lo[k] = pos_inf<T>(); hi[k] = -pos_inf<T>(); }
        for (int i = f + lane; i < f + c; i += 32) {
            vec4<T> q = xyzm[i];
            lo[0] = tmin(lo[0], q.x); hi[0] = tmax(hi[0], q.x);
            lo[1] = tmin(lo[1], q.y); hi[1] = tmax(hi[1], q.y);
            lo[2] = tmin(lo[2], q.z); hi[2] = tmax(hi[2], q.z);
        }
        for (int o = 16; o > 0; o >>= 1)
            for (int k = 0; k < 3; ++k) {
                lo[k] = tmin(lo[k], __shfl_xor_sync(kFull, lo[k], o));
                hi[k] = tmax(hi[k], __shfl_xor_sync(kFull, hi[k], o));
            }
        store_geometry<T>(a, lo, hi, node_lo, node_hi, nc, nl, cen, lane == 0);
        if constexpr (sizeof(T) == 8 && P <= kMaxPL2pDf) {
            // P2M in double-float, in the leaf's own power-of-two units: lengths in 2^eh >= its
            // largest half-width, masses in 2^em >= its mass (the FP64 pipe only forms the offsets)
            T msum = T(0);
            for (int i = f + lane; i < f + c; i += 32) msum += xyzm[i].w;
            for (int o = 16; o > 0; o >>= 1) msum += __shfl_xor_sync(kFull, msum, o);
            int eh, em;
            frexp(tmax(tmax(hi[0] - lo[0], hi[1] - lo[1]), hi[2] - lo[2]) * T(0.5), &eh);
            frexp(msum, &em);
            df m[NR];
#pragma unroll
            for (int k = 0; k < NR; ++k) m[k] = df(0.0f, 0.0f);
            for (int i = f + lane; i < f + c; i += 32) {
                const vec4<T> q = xyzm[i];
                Exp<P>::template p2m<df>(df_from(scale2(q.x - cen[0], -eh)), df_from(scale2(q.y - cen[1], -eh)),
                                         df_from(scale2(q.z - cen[2], -eh)), df_from(scale2(q.w, -em)), m);
            }
            T *dst = M + (size_t)a * ncp;
            reduce_apply<df, NR, NC>(m, lane, [&](int k, const df &x) {
                dst[k] = scale2(df_to(x), em + eh * coef_degree(k));
            });
        } else {
            T m[NR];
#pragma unroll
            for (int k = 0; k < NR; ++k) m[k] = T(0);
            for (int i = f + lane; i < f + c; i += 32) {
                vec4<T> q = xyzm[i];
                Exp<P>::template p2m<T>(q.x - cen[0], q.y - cen[1], q.z - cen[2], q.w, m);
            }
            reduce_store<T, NR, NC>(m, lane, M + (size_t)a * ncp);
        }
        // ---- climb while this warp completes the parent's last child
        int cur = a;
        for (;;) {
            // every lane's stores of this node (geometry by lane 0, moment blocks by lanes 0, 4, ...)
            // are visible before lane 0 takes the parent's ticket
            __threadfence();
            __syncwarp();
            const int par = parent[cur];
            if (par < 0) break;
            int ticket = 0;
            if (lane == 0) ticket = atomicAdd(&done[par], 1);
            ticket = __shfl_sync(kFull, ticket, 0);
            if (ticket != nchild[par] - 1) break;
            __threadfence();
            const int c0 = child0[par], nch = nchild[par];
            for (int k = 0; k < 3; ++k) { lo[k] = pos_inf<T>(); hi[k] = -pos_inf<T>(); }
            if (lane < nch) {
                for (int k = 0; k < 3; ++k) {
                    lo[k] = ld_cg(node_lo + 3 * (c0 + lane) + k);
                    hi[k] = ld_cg(node_hi + 3 * (c0 + lane) + k);
                }
            }
            for (int o = 16; o > 0; o >>= 1)
                for (int k = 0; k < 3; ++k) {
                    lo[k] = tmin(lo[k], __shfl_xor_sync(kFull, lo[k], o));
                    hi[k] = tmax(hi[k], __shfl_xor_sync(kFull, hi[k], o));
                }
            store_geometry<T>(par, lo, hi, node_lo, node_hi, nc, nl, cen, lane == 0);
            T m[NR];
#pragma unroll
            for (int k = 0; k < NR; ++k) m[k] = T(0);
            if (lane < nch) {
                const int ch = c0 + lane;
                T mc[NC];
#pragma unroll
                for (int k = 0; k < NC; ++k) mc[k] = ld_cg(M + (size_t)ch * ncp + k);
                vec4<T> cc = ld_cg(nc + ch);
                Exp<P>::template m2m<T>(mc, cc.x - cen[0], cc.y - cen[1], cc.z - cen[2], m);
            }
            // children sit in lanes 0..7, the other lanes hold zeros
            reduce_store<T, NR, NC>(m, lane, M + (size_t)par * ncp);
            cur = par;
        }
    }
}

template <class T, int P>
int launch_upward_tp(Plan &P_, cudaStream_t s)
{
    if constexpr (sizeof(T) == 8) {
        cudaMemsetAsync(P_.node_done, 0, (size_t)P_.cap_nodes * sizeof(int), s);
        k_upward_ticket<T, P><<<P_.num_sms * 8, 256, 0, s>>>(
            P_.ctr, (const vec4<T> *)P_.xyzm, P_.node_first, P_.node_count, P_.node_child0, P_.node_nchild,
            P_.node_parent, P_.node_done, (T *)P_.node_lo, (T *)P_.node_hi, (vec4<T> *)P_.node_c,
            (vec4<T> *)P_.node_l, (T *)P_.M, P_.ncp);
        return 1;
    } else {
        static const int occ = [] {
            int b = 0;
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_upward_all<T, P>, 256, 0);
            return b;
        }();
        const int blocks = std::min(2048, P_.num_sms * std::max(1, std::min(8, occ)));
        GridBarrier *gb = P_.gbar + 3;
        const vec4<T> *xyzm = (const vec4<T> *)P_.xyzm;
        T *lo = (T *)P_.node_lo, *hi = (T *)P_.node_hi, *M = (T *)P_.M;
        vec4<T> *nc = (vec4<T> *)P_.node_c, *nl = (vec4<T> *)P_.node_l;
        int ncp = P_.ncp;
        void *args[] = {&gb, &P_.ctr, (void *)&xyzm, &P_.node_first, &P_.node_count, &P_.node_child0, &P_.node_nchild,
                        (void *)&lo, (void *)&hi, (void *)&nc, (void *)&nl, (void *)&M, &ncp};
        cudaLaunchCooperativeKernel((const void *)k_upward_all<T, P>, dim3(blocks), dim3(256), args, 0, s);
        return 1;
    }
}

template <class T>
int launch_upward_t(Plan &P, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_upward_tp<T, 0>(P, s);
    case 1: return launch_upward_tp<T, 1>(P, s);
    case 2: return launch_upward_tp<T, 2>(P, s);
    case 3: return launch_upward_tp<T, 3>(P, s);
    case 4: return launch_upward_tp<T, 4>(P, s);
    case 5: return launch_upward_tp<T, 5>(P, s);
    case 6: return launch_upward_tp<T, 6>(P, s);
    case 7: return launch_upward_tp<T, 7>(P, s);
    default: return launch_upward_tp<T, 8>(P, s);
    }
}

}  // namespace

int launch_upward(Plan &P, cudaStream_t s)
{
    return P.dtype == 0 ? launch_upward_t<float>(P, s) : launch_upward_t<double>(P, s);
}

}  // namespace bfm
