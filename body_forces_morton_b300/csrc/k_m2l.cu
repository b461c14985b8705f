// Multipole-to-local translation over the M2L lists.
//
// JZ-FMM page, "Calculating a node-node interaction": with R = c_A - c_B, the
// local Taylor coefficients of receiver A gain
//     L_k += -G sum_{|n| <= p - |k|} (-1)^{|n|} M_n(B) D^{n+k}(R),  D^m = d^m (1/r),
// whose k = 0 and |k| = 1 terms through the dipole are the page's Phi_B and
// grad Phi_B equations. Only the moments and the separation are needed, never
// the source particles; the derivative tensor is built on chip for every pair
// (no per-pair operator data in memory).
//
// The contraction runs on reduced (trace-free) coefficients: D^m is harmonic,
// so the moments with n_z >= 2 fold into those with n_z <= 1 once per node
// (k_moments_r, Exp<P>::reduce_m) and only the locals with k_z <= 1 are
// accumulated, the others following from the same identity when the receiver's
// row is written (Exp<P>::expand_l): (p+1)^2 instead of C(p+3,3) coefficients
// each side, 155 instead of 210 terms at p = 4.
//
// One warp per receiver, receivers taken from a shared counter in decreasing
// order of list length; lane j takes the receiver's sources j, j+32, ... in
// list order (ascending source index) and keeps a private partial L in
// registers. The reduced multipoles of each round of 32 sources are staged
// through shared memory with coalesced 16-byte loads; a fixed reduction sums
// the lanes, so the result is reproducible.
#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

constexpr int M2L_WARPS = 4;

template <class T> struct Vec16;
template <> struct Vec16<float> { using type = float4; static constexpr int n = 4; };
template <> struct Vec16<double> { using type = double2; static constexpr int n = 2; };

template <class T, int P> struct M2LShape {
    static constexpr int NC = Exp<P>::NC;
    static constexpr int NCP = (NC + 3) / 4 * 4;      // row stride of M and L in global memory
    static constexpr int NRC = Exp<P>::NRC;           // reduced coefficients
    static constexpr int NRP = (NRC + 3) / 4 * 4;     // row stride of the reduced moments
    static constexpr int STR = NRP + 1;               // odd row stride in shared memory
    static constexpr int V = Vec16<T>::n;             // elements per 16-byte load
    static constexpr int NV = NRP / V;
    static constexpr int NR = (NRC + 7) / 8 * 8;      // accumulators, padded for the halving reduction
    static constexpr size_t smem = sizeof(T) * M2L_WARPS * (32 * STR + NRC);
};

// Reduced moments of every node: Mr[b] = reduce_m(M[b]), padding zeroed.
template <class T, int P>
__global__ __launch_bounds__(256) void k_moments_r(const DevCounters *__restrict__ nctr, const T *__restrict__ M, T *__restrict__ Mr)
{
    const int n_nodes = phase2_nodes(nctr);
    using S = M2LShape<T, P>;
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < n_nodes; b += gridDim.x * blockDim.x) {
        T r[S::NRP];
#pragma unroll
        for (int i = S::NRC; i < S::NRP; ++i) r[i] = T(0);
        Exp<P>::template reduce_m<T>(M + (size_t)b * S::NCP, r);
#pragma unroll
        for (int i = 0; i < S::NRP; ++i) Mr[(size_t)b * S::NRP + i] = r[i];
    }
}

template <class T, int P>
__global__ __launch_bounds__(M2L_WARPS * 32) void k_m2l(const DevCounters *__restrict__ nctr, const int *__restrict__ order,
                                                        const int *__restrict__ off,
                                                        const int *__restrict__ src, const vec4<T> *__restrict__ nc,
                                                        const T *__restrict__ Mr, T *__restrict__ Lout,
                                                        DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    using S = M2LShape<T, P>;
    using V16 = typename Vec16<T>::type;
    extern __shared__ __align__(16) unsigned char m2l_smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T *rows = reinterpret_cast<T *>(m2l_smem) + (size_t)w * 32 * S::STR;
    T *lred = reinterpret_cast<T *>(m2l_smem) + (size_t)M2L_WARPS * 32 * S::STR + (size_t)w * S::NRC;
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[1], 1);
        t = __shfl_sync(kFull, t, 0);
        if (t >= n_nodes) break;
        const int a = order[t];
        const int beg = off[a], end = off[a + 1];
        const vec4<T> ca = nc[a];
        T L[S::NR];
#pragma unroll
        for (int k = 0; k < S::NR; ++k) L[k] = T(0);
        for (int q0 = beg; q0 < end; q0 += 32) {
            const int q = q0 + lane;
            const bool valid = q < end;
            const int b = valid ? src[q] : 0;
            const int nsrc = min(32, end - q0);
            __syncwarp();
            // stage the reduced multipole rows of this round's sources (16-byte loads, one row per source)
            for (int t0 = 0; t0 < nsrc * S::NV; t0 += 32) {
                const int tt = t0 + lane;
                const int row = tt / S::NV, col = tt - row * S::NV;
                const int bb = __shfl_sync(kFull, b, row & 31);
                if (tt < nsrc * S::NV) {
                    const V16 x = __ldg(reinterpret_cast<const V16 *>(Mr + (size_t)bb * S::NRP) + col);
                    const T *xs = reinterpret_cast<const T *>(&x);
#pragma unroll
                    for (int i = 0; i < S::V; ++i) rows[row * S::STR + col * S::V + i] = xs[i];
                }
            }
            __syncwarp();
            if (valid) {
                const vec4<T> cb = nc[b];
                Exp<P>::template m2l_r<T>(rows + lane * S::STR, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L);
            }
        }
        reduce_apply<T, S::NR, S::NRC>(L, lane, [&](int k, const T &x) { lred[k] = x; });
        __syncwarp();
        if (lane == 0) Exp<P>::template expand_l<T>(lred, Lout + (size_t)a * S::NCP);
    }
}

template <class T, int P>
int launch_m2l_tp(Plan &P_, cudaStream_t s)
{
    using S = M2LShape<T, P>;
    static_assert(S::NRP % S::V == 0, "row stride must be a whole number of 16-byte loads");
    k_moments_r<T, P><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, (const T *)P_.M, (T *)P_.Mr);
    cudaFuncSetAttribute(k_m2l<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::smem);
    k_m2l<T, P><<<P_.num_sms * 16, M2L_WARPS * 32, S::smem, s>>>(
        P_.ctr, P_.order + P_.cap_nodes, P_.m2l_off, P_.m2l_src, (const vec4<T> *)P_.node_c,
        (const T *)P_.Mr, (T *)P_.Lm2l, P_.ctr);
    return 2;
}

template <class T>
int launch_m2l_t(Plan &P, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_m2l_tp<T, 0>(P, s);
    case 1: return launch_m2l_tp<T, 1>(P, s);
    case 2: return launch_m2l_tp<T, 2>(P, s);
    case 3: return launch_m2l_tp<T, 3>(P, s);
    case 4: return launch_m2l_tp<T, 4>(P, s);
    case 5: return launch_m2l_tp<T, 5>(P, s);
    case 6: return launch_m2l_tp<T, 6>(P, s);
    case 7: return launch_m2l_tp<T, 7>(P, s);
    default: return launch_m2l_tp<T, 8>(P, s);
    }
}

}  // namespace

int launch_m2l(Plan &P, cudaStream_t s)
{
    if (P.dtype == 0) return launch_m2l_t<float>(P, s);
    return P.p <= kMaxPDf ? launch_m2l_df(P, s) : launch_m2l_t<double>(P, s);
}

}  // namespace bfm
