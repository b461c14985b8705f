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
// registers. Each lane copies its own source's reduced multipole row into
// shared memory with 16-byte asynchronous copies, one round of 32 sources
// ahead of the round it computes (double buffer, one copy group per round),
// and reads it back with 16-byte loads; rows sit an odd number of 16-byte
// units apart, so the lanes' reads of their own rows are free of bank
// conflicts. No lane touches another lane's row, so the pipeline needs no
// warp synchronisation. A fixed reduction sums the lanes, so the result is
// reproducible.
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
    static constexpr int V = Vec16<T>::n;             // elements per 16-byte load
    static constexpr int NV = NRP / V;                // 16-byte units per row
    static constexpr int SU = NV | 1;                 // row stride in shared memory, in 16-byte units (odd)
    static constexpr int STR = SU * V;                // the same in elements
    static constexpr bool REG = NRP * sizeof(T) <= 128;  // rows small enough to read into registers
    static constexpr int NR = (NRC + 7) / 8 * 8;      // accumulators, padded for the halving reduction
    static constexpr size_t smem = sizeof(T) * M2L_WARPS * (2 * 32 * STR + NRC);
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

// One source of the current round: its reduced row (in this lane's shared
// slot) translated to the receiver's centre ca and added to L.
template <class T, int P>
__device__ __forceinline__ void m2l_apply_row(const T *row, const vec4<T> &ca, const vec4<T> &cb,
                                              T (&L)[M2LShape<T, P>::NR])
{
    using S = M2LShape<T, P>;
    using V16 = typename Vec16<T>::type;
    if constexpr (S::REG) {
        T m[S::NRP];
#pragma unroll
        for (int c = 0; c < S::NV; ++c) *reinterpret_cast<V16 *>(m + c * S::V) = reinterpret_cast<const V16 *>(row)[c];
        Exp<P>::template m2l_r<T>(m, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L);
    } else {
        Exp<P>::template m2l_r<T>(row, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L);
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
    extern __shared__ __align__(16) unsigned char m2l_smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T *const slot = reinterpret_cast<T *>(m2l_smem) + (size_t)w * 2 * 32 * S::STR + lane * S::STR;  // buffer 0
    T *const slot1 = slot + 32 * S::STR;                                                                 // buffer 1
    T *lred = reinterpret_cast<T *>(m2l_smem) + (size_t)M2L_WARPS * 2 * 32 * S::STR + (size_t)w * S::NRC;
    // copy source q's row (if q is in the list) into dst; returns its centre
    auto stage = [&](int q, int end, T *dst, bool &valid) {
        valid = q < end;
        vec4<T> cb = make4<T>(T(0), T(0), T(0), T(0));
        if (valid) {
            const int b = src[q];
            cb = nc[b];
            const T *g = Mr + (size_t)b * S::NRP;
#pragma unroll
            for (int c = 0; c < S::NV; ++c) cp_async16(dst + c * S::V, g + c * S::V);
        }
        cp_async_commit();
        return cb;
    };
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
        bool valid;
        vec4<T> cb = stage(beg + lane, end, slot, valid);
        int cur = 0;
        for (int q0 = beg; q0 < end; q0 += 32) {
            bool valid_n;
            const vec4<T> cb_n = stage(q0 + 32 + lane, end, cur ? slot : slot1, valid_n);
            cp_async_wait_group<1>();  // this lane's copies of the current round have landed
            if (valid) m2l_apply_row<T, P>(cur ? slot1 : slot, ca, cb, L);
            valid = valid_n;
            cb = cb_n;
            cur ^= 1;
        }
        cp_async_wait_all();
        reduce_apply<T, S::NR, S::NRC>(L, lane, [&](int k, const T &x) { lred[k] = x; });
        __syncwarp();
        if (lane == 0) Exp<P>::template expand_l<T>(lred, Lout + (size_t)a * S::NCP);
        __syncwarp();
    }
}

template <class T, int P>
int launch_m2l_tp(Plan &P_, const void *M, void *Lout, cudaStream_t s)
{
    using S = M2LShape<T, P>;
    static_assert(S::NRP % S::V == 0, "row stride must be a whole number of 16-byte loads");
    static_assert(S::smem <= 227 * 1024, "M2L staging exceeds shared memory");
    k_moments_r<T, P><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, (const T *)M, (T *)P_.Mr);
    cudaFuncSetAttribute(k_m2l<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::smem);
    k_m2l<T, P><<<P_.num_sms * 16, M2L_WARPS * 32, S::smem, s>>>(
        P_.ctr, P_.order + P_.cap_nodes, P_.m2l_off, P_.m2l_src, (const vec4<T> *)P_.node_c,
        (const T *)P_.Mr, (T *)Lout, P_.ctr);
    return 2;
}

template <class T>
int launch_m2l_t(Plan &P, const void *M, void *Lout, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_m2l_tp<T, 0>(P, M, Lout, s);
    case 1: return launch_m2l_tp<T, 1>(P, M, Lout, s);
    case 2: return launch_m2l_tp<T, 2>(P, M, Lout, s);
    case 3: return launch_m2l_tp<T, 3>(P, M, Lout, s);
    case 4: return launch_m2l_tp<T, 4>(P, M, Lout, s);
    case 5: return launch_m2l_tp<T, 5>(P, M, Lout, s);
    case 6: return launch_m2l_tp<T, 6>(P, M, Lout, s);
    case 7: return launch_m2l_tp<T, 7>(P, M, Lout, s);
    default: return launch_m2l_tp<T, 8>(P, M, Lout, s);
    }
}

}  // namespace

int launch_m2l(Plan &P, cudaStream_t s)
{
    if (P.dtype == 0) return launch_m2l_t<float>(P, P.M, P.Lm2l, s);
    return P.p <= kMaxPDf && !P.f64_ieee ? launch_m2l_df(P, s) : launch_m2l_t<double>(P, P.M, P.Lm2l, s);
}

int launch_m2l_plain(Plan &P, const void *M, void *Lout, cudaStream_t s)
{
    return P.dtype == 0 ? launch_m2l_t<float>(P, M, Lout, s) : launch_m2l_t<double>(P, M, Lout, s);
}

}  // namespace bfm
