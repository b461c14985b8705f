// Upward pass: node boxes, centres, half-widths, P2M at the leaves and M2M to
// the parents, in one kernel.
//
// JZ-FMM page, "Combining near and far interactions", stage 1: calculate the
// moments of the leaves, then translate and combine the children's moments
// around their parent centres. Moments M_n = sum m s^n / n! about the centre
// c = (lo + hi) / 2 of the node's tight box; l = (hi - lo) / 2 is the per-axis
// half-width of the opening criterion.
//
// fp32 plans: one launch, deepest level first, a node's eight lanes waiting on
// its children's flags (k_upward_flags): a leaf's box and P2M from its
// particles, an internal node's box the union of its children's boxes and its
// moments the sum of their M2M translations, both reduced in a fixed order
// over the 8-lane group. fp64 plans: k_upward_ticket, below.
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

// fp32 plans' upward pass in one launch, without grid barriers: warps take
// chunks of four nodes of one level from a shared counter, deepest level
// first, eight lanes per node. A leaf's group bounds and expands its own
// particles (P2M); an internal node's group waits, bounded, until each child's
// flag holds this pass's number (stored with release semantics once the
// child's box and moments are written), then unites the children's boxes and
// sums their M2M translations. Both kinds meet in the same fixed-order 8-lane
// reductions, so no lane waits inside a shuffle. A chunk never spans two
// levels, so no lane waits for its own warp; every child lies in an earlier
// chunk, taken by a running warp, so the earliest unfinished chunk can always
// finish.
template <class T, int P>
__global__ __launch_bounds__(256) void k_upward_flags(DevCounters *ctr, const vec4<T> *__restrict__ xyzm,
                                                      const int *__restrict__ first, const int *__restrict__ count,
                                                      const int *__restrict__ child0, const int *__restrict__ nchild,
                                                      T *node_lo, T *node_hi, vec4<T> *nc, vec4<T> *nl, T *M, int ncp,
                                                      unsigned *flag, unsigned seq, T *Mr)
{
    constexpr int NC = Exp<P>::NC;
    constexpr int NR = Padded<NC>::value;
    __shared__ int s_off[kMaxLevel + 2];
    const int n_nodes = phase2_nodes(ctr);
    if (n_nodes == 0) return;
    const int depth = ctr->depth;
    for (int l = threadIdx.x; l <= depth + 1; l += blockDim.x) s_off[l] = min(ctr->level_off[l], n_nodes);
    __syncthreads();
    const int lane = threadIdx.x & 31, g = lane >> 3, j = lane & 7;
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[3], 1);
        t = __shfl_sync(kFull, t, 0);
        int lo_n = 0, hi_n = -1;
        for (int l = depth; l >= 0; --l) {  // chunk t -> four nodes of one level, deepest level first
            const int nch = (s_off[l + 1] - s_off[l] + 3) >> 2;
            if (t < nch) {
                lo_n = s_off[l] + 4 * t;
                hi_n = min(s_off[l + 1], lo_n + 4);
                break;
            }
            t -= nch;
        }
        if (hi_n < 0) break;
        const int a = lo_n + g;
        const bool valid = a < hi_n;
        const int nch = valid ? nchild[a] : 0;
        const bool leaf = valid && nch == 0;
        const int f = leaf ? first[a] : 0, c = leaf ? count[a] : 0;
        const bool has = j < nch;
        const int ch = has ? child0[a] + j : 0;
        T lo[3], hi[3], cen[3];
        for (int k = 0; k < 3; ++k) { lo[k] = pos_inf<T>(); hi[k] = -pos_inf<T>(); }
        if (leaf) {
            for (int i = f + j; i < f + c; i += 8) {
                const vec4<T> q = xyzm[i];
                lo[0] = tmin(lo[0], q.x); hi[0] = tmax(hi[0], q.x);
                lo[1] = tmin(lo[1], q.y); hi[1] = tmax(hi[1], q.y);
                lo[2] = tmin(lo[2], q.z); hi[2] = tmax(hi[2], q.z);
            }
        } else if (has) {
            cuda::atomic_ref<unsigned, cuda::thread_scope_device> fl(flag[ch]);
            unsigned spins = 0;
            while (fl.load(cuda::memory_order_acquire) != seq) {
                if (++spins > kSpinLimit) {
                    set_error(ctr, ERR_SPIN);
                    break;
                }
                __nanosleep(32);
            }
            for (int k = 0; k < 3; ++k) {
                lo[k] = ld_cg(node_lo + 3 * ch + k);
                hi[k] = ld_cg(node_hi + 3 * ch + k);
            }
        }
        for (int o = 4; o > 0; o >>= 1)
            for (int k = 0; k < 3; ++k) {
                lo[k] = tmin(lo[k], __shfl_xor_sync(kFull, lo[k], o));
                hi[k] = tmax(hi[k], __shfl_xor_sync(kFull, hi[k], o));
            }
        store_geometry<T>(a, lo, hi, node_lo, node_hi, nc, nl, cen, valid && j == 0);
        T m[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) m[k] = T(0);
        if (leaf) {
            for (int i = f + j; i < f + c; i += 8) {
                const vec4<T> q = xyzm[i];
                Exp<P>::template p2m<T>(q.x - cen[0], q.y - cen[1], q.z - cen[2], q.w, m);
            }
        } else if (has) {
            T mc[NC];
            if constexpr (sizeof(T) == 4) {
                // the child's row in 16-byte pieces through L2 (rows are padded to a multiple of 4)
                const float4 *v = reinterpret_cast<const float4 *>(M + (size_t)ch * ncp);
#pragma unroll
                for (int q = 0; q < (NC + 3) / 4; ++q) {
                    const float4 x = __ldcg(v + q);
                    const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int h = 0; h < 4; ++h)
                        if (4 * q + h < NC) mc[4 * q + h] = e[h];
                }
            } else {
#pragma unroll
                for (int k = 0; k < NC; ++k) mc[k] = ld_cg(M + (size_t)ch * ncp + k);
            }
            const vec4<T> cc = ld_cg(nc + ch);
            Exp<P>::template m2m<T>(mc, cc.x - cen[0], cc.y - cen[1], cc.z - cen[2], m);
        }
        T *dst = M + (size_t)a * ncp;
        reduce_apply8<T, NR, NC>(m, j, [&](int k, const T &x) {
            if (valid) dst[k] = x;
        });
        // publish the group's box and moments, then the node's flag
        __threadfence();
        __syncwarp();
        if (valid && j == 0) {
            cuda::atomic_ref<unsigned, cuda::thread_scope_device>(flag[a]).store(seq, cuda::memory_order_release);
            if (Mr != nullptr) {  // the reduced row the M2L reads, off the parents' wait
                constexpr int NRC = Exp<P>::NRC, NRP = (NRC + 3) / 4 * 4;
                T mk[NC], r[NRP];
                if constexpr (sizeof(T) == 4) {
                    const float4 *v = reinterpret_cast<const float4 *>(dst);
#pragma unroll
                    for (int q = 0; q < (NC + 3) / 4; ++q) {
                        const float4 x = v[q];
                        const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int h = 0; h < 4; ++h)
                            if (4 * q + h < NC) mk[4 * q + h] = e[h];
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < NC; ++k) mk[k] = dst[k];
                }
#pragma unroll
                for (int k = NRC; k < NRP; ++k) r[k] = T(0);
                Exp<P>::template reduce_m<T>(mk, r);
                if constexpr (sizeof(T) == 4) {
                    float4 *v = reinterpret_cast<float4 *>(Mr + (size_t)a * NRP);
#pragma unroll
                    for (int q = 0; q < NRP / 4; ++q) v[q] = make_float4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                } else {
#pragma unroll
                    for (int k = 0; k < NRP; ++k) Mr[(size_t)a * NRP + k] = r[k];
                }
            }
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
                                                vec4<T> *nc, vec4<T> *nl, T *M, int ncp, bool use_df)
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
        if (sizeof(T) == 8 && P <= kMaxPL2pDf && use_df) {
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
            (vec4<T> *)P_.node_l, (T *)P_.M, P_.ncp, !P_.f64_ieee);
        P_.mr_fresh = false;
        return 1;
    } else {
        const unsigned seq = P_.next_flag_seq(s);
        k_upward_flags<T, P><<<P_.num_sms * 4, 256, 0, s>>>(
            P_.ctr, (const vec4<T> *)P_.xyzm, P_.node_first, P_.node_count, P_.node_child0, P_.node_nchild,
            (T *)P_.node_lo, (T *)P_.node_hi, (vec4<T> *)P_.node_c, (vec4<T> *)P_.node_l, (T *)P_.M, P_.ncp,
            P_.node_flag, seq, P_.m2l_rotation ? (T *)nullptr : (T *)P_.Mr);
        P_.mr_fresh = !P_.m2l_rotation;  // the reduced rows of this evaluation's moments are written
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
