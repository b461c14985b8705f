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
// One warp per receiver; lane j takes the receiver's sources j, j+32, ... in
// list order (ascending source index) and keeps a private partial L in
// registers; a fixed butterfly sums the lanes, so the result is reproducible.
#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

template <class T, int P>
__global__ __launch_bounds__(256) void k_m2l(int n_nodes, const int *__restrict__ off, const int *__restrict__ src,
                                             const vec4<T> *__restrict__ nc, const T *__restrict__ M, int ncp,
                                             T *__restrict__ Lout)
{
    constexpr int NC = Exp<P>::NC;
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        const int beg = off[a], end = off[a + 1];
        const vec4<T> ca = nc[a];
        T L[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) L[k] = T(0);
        for (int q = beg + lane; q < end; q += 32) {
            const int b = src[q];
            const vec4<T> cb = nc[b];
            T mb[NC];
            const T *row = M + (size_t)b * ncp;
#pragma unroll
            for (int k = 0; k < NC; ++k) mb[k] = __ldg(row + k);
            Exp<P>::template m2l<T>(mb, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L);
        }
        if (end - beg > 0) {
#pragma unroll
            for (int k = 0; k < NC; ++k) L[k] = warp_sum_xor(L[k]);
        }
        if (lane == 0) {
            T *dst = Lout + (size_t)a * ncp;
#pragma unroll
            for (int k = 0; k < NC; ++k) dst[k] = L[k];
        }
    }
}

template <class T, int P>
int launch_m2l_tp(Plan &P_, cudaStream_t s)
{
    k_m2l<T, P><<<P_.num_sms * 8, 256, 0, s>>>((int)P_.n_nodes, P_.m2l_off, P_.m2l_src, (const vec4<T> *)P_.node_c,
                                               (const T *)P_.M, P_.ncp, (T *)P_.Lm2l);
    return 1;
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
    return P.dtype == 0 ? launch_m2l_t<float>(P, s) : launch_m2l_t<double>(P, s);
}

}  // namespace bfm
