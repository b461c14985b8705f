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
// registers. The reduced multipole rows of a round's 32 sources are copied
// into shared memory with 16-byte asynchronous copies one round ahead of the
// round that uses them (double buffer, one copy group per round), coalesced:
// a group of NV lanes streams one row (NV 16-byte pieces), so one copy
// instruction reads whole rows instead of 32 scattered 16-byte pieces (those
// kept the L1 at ~90 % of its request throughput). Each lane then reads its
// own source's row back with 16-byte loads; rows sit an odd number of 16-byte
// units apart, so these reads are free of bank conflicts. A fixed reduction
// sums the lanes, so the result is reproducible.
#include "expansions_gen.cuh"
#include "plan.h"

#include <type_traits>
#include "rotation_gen.cuh"

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

// The two M2L operators on rows of (p+1)^2 coefficients: `prep` turns a node's
// moments into its row, `pair` adds one source row's translation to a
// receiver's accumulators, `finish` turns the accumulators into the complete
// Cartesian local. The results are the same (the total-degree truncation);
// the per-pair work differs.
//   OpReduced:  the reduced (trace-free) Cartesian contraction, D^n(R) built
//               by recurrence (the default);
//   OpRotation: real solid harmonics, each pair rotated so that R lies on z,
//               translated along z and rotated back (jaccpot issue 152, item
//               1: the rotations built on chip from the separation).
template <int P> struct OpReduced {
    template <class T> static __device__ __forceinline__ void prep(const T *M, T *r) { Exp<P>::template reduce_m<T>(M, r); }
    template <class T> static __device__ __forceinline__ void pair(const T *r, T rx, T ry, T rz, T *L)
    {
        Exp<P>::template m2l_r<T>(r, rx, ry, rz, L);
    }
    template <class T> static __device__ __forceinline__ void finish(const T *l, T *L) { Exp<P>::template expand_l<T>(l, L); }
};
template <int P> struct OpRotation {
    template <class T> static __device__ __forceinline__ void prep(const T *M, T *r) { Rot<P>::template to_sph<T>(M, r); }
    template <class T> static __device__ __forceinline__ void pair(const T *r, T rx, T ry, T rz, T *L)
    {
        Rot<P>::template m2l<T>(r, rx, ry, rz, L);
    }
    template <class T> static __device__ __forceinline__ void finish(const T *l, T *L) { Rot<P>::template from_sph<T>(l, L); }
};

// Rows of every node: Mr[b] = prep(M[b]), padding zeroed.
template <class T, int P, class Op>
__global__ __launch_bounds__(256) void k_moments_r(const DevCounters *__restrict__ nctr, const T *__restrict__ M, T *__restrict__ Mr)
{
    const int n_nodes = phase2_nodes(nctr);
    using S = M2LShape<T, P>;
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < n_nodes; b += gridDim.x * blockDim.x) {
        T r[S::NRP];
#pragma unroll
        for (int i = S::NRC; i < S::NRP; ++i) r[i] = T(0);
        Op::template prep<T>(M + (size_t)b * S::NCP, r);
#pragma unroll
        for (int i = 0; i < S::NRP; ++i) Mr[(size_t)b * S::NRP + i] = r[i];
    }
}

// One source of the current round: its reduced row (in this lane's shared
// slot) translated to the receiver's centre ca and added to L.
template <class T, int P, class Op>
__device__ __forceinline__ void m2l_apply_row(const T *row, const vec4<T> &ca, const vec4<T> &cb,
                                              T (&L)[M2LShape<T, P>::NR])
{
    using S = M2LShape<T, P>;
    using V16 = typename Vec16<T>::type;
    if constexpr (S::REG) {
        T m[S::NRP];
#pragma unroll
        for (int c = 0; c < S::NV; ++c) *reinterpret_cast<V16 *>(m + c * S::V) = reinterpret_cast<const V16 *>(row)[c];
        Op::template pair<T>(m, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L);
    } else {
        Op::template pair<T>(row, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L);
    }
}

// Blocks per SM the fp32 reduced-operator kernel is compiled for: more resident
// warps hide the row loads' latency (measured: 0.229 ms at 4 blocks, 0.221 at
// 5, 0.218 at 6 for p = 4); beyond these the registers spill.
template <class T, int P, class Op> struct M2LMinBlocks { static constexpr int value = 1; };
template <int P> struct M2LMinBlocks<float, P, OpReduced<P>> {
    static constexpr int value = P <= 3 ? 8 : (P == 4 ? 6 : 1);
};

template <class T, int P, class Op>
__global__ __launch_bounds__(M2L_WARPS * 32, M2LMinBlocks<T, P, Op>::value) void k_m2l(const DevCounters *__restrict__ nctr, const int *__restrict__ order,
                                                        const int *__restrict__ off,
                                                        const int *__restrict__ src, const vec4<T> *__restrict__ nc,
                                                        const T *__restrict__ Mr, T *__restrict__ Lout,
                                                        DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    using S = M2LShape<T, P>;
    extern __shared__ __align__(16) unsigned char m2l_smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T *const rows0 = reinterpret_cast<T *>(m2l_smem) + (size_t)w * 2 * 32 * S::STR;  // buffer 0
    T *const rows1 = rows0 + 32 * S::STR;                                               // buffer 1
    T *const slot = rows0 + lane * S::STR, *const slot1 = rows1 + lane * S::STR;        // this lane's row
    T *lred = reinterpret_cast<T *>(m2l_smem) + (size_t)M2L_WARPS * 2 * 32 * S::STR + (size_t)w * S::NRC;
    // the copy layout: G rows per copy instruction, row r = r0 + g streamed by lanes g NV .. g NV + NV - 1
    // (rows longer than 32 pieces take CPR passes of all 32 lanes)
    constexpr int G = S::NV <= 32 ? 32 / S::NV : 1;
    constexpr int CPR = S::NV <= 32 ? 1 : (S::NV + 31) / 32;
    const int g = S::NV <= 32 ? lane / S::NV : 0;
    const int c0 = S::NV <= 32 ? lane - g * S::NV : lane;
    // copy the rows of sources q0 .. q0 + 31 (those in the list) into the buffer at rows0;
    // returns this lane's source centre
    auto stage = [&](int q0, int end, T *rows0, bool &valid) {
        const int q = q0 + lane;
        valid = q < end;
        const int b = valid ? src[q] : -1;
        const vec4<T> cb = valid ? nc[b] : make4<T>(T(0), T(0), T(0), T(0));
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += G) {
            const int r = r0 + g;
            const int br = __shfl_sync(kFull, b, r & 31);
            if (g < G && r < 32 && br >= 0)
#pragma unroll
                for (int cc = 0; cc < CPR; ++cc) {
                    const int c = c0 + cc * 32;
                    if (c < S::NV) cp_async16(rows0 + r * S::STR + c * S::V, Mr + (size_t)br * S::NRP + c * S::V);
                }
        }
        cp_async_commit();
        return cb;
    };
    // the next receiver's ticket and node are taken while the current one computes
    auto ticket = [&]() {
        int tk = 0;
        if (lane == 0) tk = atomicAdd(&ctr->work_ctr[1], 1);
        return __shfl_sync(kFull, tk, 0);
    };
    int t = ticket();
    int a_n = t < n_nodes ? order[t] : 0;
    for (;;) {
        if (t >= n_nodes) break;
        const int a = a_n;
        const int beg = off[a], end = off[a + 1];
        const vec4<T> ca = nc[a];
        t = ticket();
        a_n = t < n_nodes ? order[t] : 0;
        T L[S::NR];
#pragma unroll
        for (int k = 0; k < S::NR; ++k) L[k] = T(0);
        bool valid;
        vec4<T> cb = stage(beg, end, rows0, valid);
        int cur = 0;
        for (int q0 = beg; q0 < end; q0 += 32) {
            bool valid_n;
            __syncwarp();  // every lane is done with the buffer the next round's rows go to
            const vec4<T> cb_n = stage(q0 + 32, end, cur ? rows0 : rows1, valid_n);
            cp_async_wait_group<1>();  // this lane's copies of the current round have landed,
            __syncwarp();              // and so have every other lane's
            if (valid) m2l_apply_row<T, P, Op>(cur ? slot1 : slot, ca, cb, L);
            valid = valid_n;
            cb = cb_n;
            cur ^= 1;
        }
        cp_async_wait_all();
        reduce_apply<T, S::NR, S::NRC>(L, lane, [&](int k, const T &x) { lred[k] = x; });
        __syncwarp();
        if (lane == 0) Op::template finish<T>(lred, Lout + (size_t)a * S::NCP);
        __syncwarp();
    }
}

// ---- mutual M2L (the scheme is described in k_mutual.cu) ----------------------
// Pass 1: a warp per receiver a (the M2L work order), a lane per entry of a's
// upper part (sources b > a), with the rows staged as in k_m2l (coalesced
// asynchronous copies one round ahead). Exp<P>::m2l_r_pair gives both
// directions from one derivative tensor: a's share stays in the lane's
// accumulators, b's share (reduced coefficients) goes through the lane's
// shared slot to the row of the mirrored entry, written by groups of lanes that
// stream whole rows. The lanes' sums are added by the fixed reduction into a's
// own reduced share.
template <class T, int P>
struct MutShape {
    using S = M2LShape<T, P>;
    static constexpr size_t per_warp = sizeof(T) * (3 * 32 * S::STR + S::NRP);
    static constexpr int W = 4 * per_warp <= 200 * 1024 ? 4 : (2 * per_warp <= 200 * 1024 ? 2 : 1);  // warps per block
    static constexpr size_t smem = W * per_warp;
};

template <class T, int P>
__global__ __launch_bounds__(MutShape<T, P>::W * 32) void k_m2l_mut1(const DevCounters *__restrict__ nctr,
                                                             const int *__restrict__ order, const int *__restrict__ off,
                                                             const int *__restrict__ src, const int *__restrict__ lo,
                                                             const int *__restrict__ mir, const vec4<T> *__restrict__ nc,
                                                             const T *__restrict__ Mr, T *__restrict__ rbuf,
                                                             long long rows, T *__restrict__ lpart, DevCounters *ctr)
{
    using S = M2LShape<T, P>;
    using V16 = typename Vec16<T>::type;
    extern __shared__ __align__(16) unsigned char m2l_smem[];
    const int n_nodes = phase2_nodes(nctr);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    T *const rows0 = reinterpret_cast<T *>(m2l_smem) + (size_t)w * 3 * 32 * S::STR;
    T *const rows1 = rows0 + 32 * S::STR;
    T *const outb = rows1 + 32 * S::STR;                        // partner shares of the round, a row per lane
    T *const s_ma = reinterpret_cast<T *>(m2l_smem) + (size_t)MutShape<T, P>::W * 3 * 32 * S::STR + (size_t)w * S::NRP;
    T *const slot = rows0 + lane * S::STR, *const slot1 = rows1 + lane * S::STR, *const oslot = outb + lane * S::STR;
    constexpr int G = S::NV <= 32 ? 32 / S::NV : 1;
    constexpr int CPR = S::NV <= 32 ? 1 : (S::NV + 31) / 32;
    const int g = S::NV <= 32 ? lane / S::NV : 0;
    const int c0 = S::NV <= 32 ? lane - g * S::NV : lane;
    auto stage = [&](int q0, int end, T *rbase, bool &valid) {
        const int q = q0 + lane;
        valid = q < end;
        const int b = valid ? src[q] : -1;
        const vec4<T> cb = valid ? nc[b] : make4<T>(T(0), T(0), T(0), T(0));
#pragma unroll
        for (int r0 = 0; r0 < 32; r0 += G) {
            const int r = r0 + g;
            const int br = __shfl_sync(kFull, b, r & 31);
            if (g < G && r < 32 && br >= 0)
#pragma unroll
                for (int cc = 0; cc < CPR; ++cc) {
                    const int c = c0 + cc * 32;
                    if (c < S::NV) cp_async16(rbase + r * S::STR + c * S::V, Mr + (size_t)br * S::NRP + c * S::V);
                }
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
        const int u0 = off[a] + lo[a], end = off[a + 1];
        const vec4<T> ca = nc[a];
        __syncwarp();
        for (int k = lane; k < S::NRP; k += 32) s_ma[k] = Mr[(size_t)a * S::NRP + k];
        T L[S::NR];
#pragma unroll
        for (int k = 0; k < S::NR; ++k) L[k] = T(0);
        bool valid;
        vec4<T> cb = stage(u0, end, rows0, valid);
        int cur = 0;
        for (int q0 = u0; q0 < end; q0 += 32) {
            bool valid_n;
            __syncwarp();
            const vec4<T> cb_n = stage(q0 + 32, end, cur ? rows0 : rows1, valid_n);
            cp_async_wait_group<1>();
            __syncwarp();
            const int q = q0 + lane;
            const int m = valid && q < rows ? mir[q] : -1;
            if (valid) {
                T lb[S::NRP];
#pragma unroll
                for (int k = 0; k < S::NRP; ++k) lb[k] = T(0);
                const T *row = cur ? slot1 : slot;
                if constexpr (S::REG) {
                    T mb[S::NRP];
#pragma unroll
                    for (int c = 0; c < S::NV; ++c)
                        *reinterpret_cast<V16 *>(mb + c * S::V) = reinterpret_cast<const V16 *>(row)[c];
                    Exp<P>::template m2l_r_pair<T>(s_ma, mb, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L, lb);
                } else {
                    Exp<P>::template m2l_r_pair<T>(s_ma, row, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, L, lb);
                }
#pragma unroll
                for (int c = 0; c < S::NV; ++c)
                    reinterpret_cast<V16 *>(oslot)[c] = *reinterpret_cast<const V16 *>(lb + c * S::V);
            }
            if (valid && !(m >= 0 && m < rows)) set_error(ctr, ERR_BOUNDS);
            __syncwarp();
            // the round's partner shares to their rows, whole rows per group of lanes
#pragma unroll
            for (int r0 = 0; r0 < 32; r0 += G) {
                const int r = r0 + g;
                const int mr = __shfl_sync(kFull, (m >= 0 && m < rows) ? m : -1, r & 31);
                if (g < G && r < 32 && mr >= 0)
#pragma unroll
                    for (int cc = 0; cc < CPR; ++cc) {
                        const int c = c0 + cc * 32;
                        if (c < S::NV)
                            reinterpret_cast<V16 *>(rbuf + (size_t)mr * S::NRP)[c] =
                                reinterpret_cast<const V16 *>(outb + r * S::STR)[c];
                    }
            }
            valid = valid_n;
            cb = cb_n;
            cur ^= 1;
        }
        cp_async_wait_all();
        reduce_apply<T, S::NR, S::NRC>(L, lane, [&](int k, const T &x) { lpart[(size_t)a * S::NRP + k] = x; });
    }
}

// Pass 2: a warp per node: the rows of its lower part (written by the partners'
// pass 1) summed over the lanes in a fixed order, added to its own share and
// expanded to the complete Cartesian local.
template <class T, int P>
__global__ __launch_bounds__(256) void k_m2l_mut2(const DevCounters *__restrict__ nctr, const int *__restrict__ off,
                                                  const int *__restrict__ lo, const T *__restrict__ rbuf, long long rows,
                                                  const T *__restrict__ lpart, T *__restrict__ Lout, DevCounters *ctr)
{
    using S = M2LShape<T, P>;
    using V16 = typename Vec16<T>::type;
    __shared__ T s_l[8][S::NRP];
    const int n_nodes = phase2_nodes(nctr);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        const int beg = off[a], stop = beg + lo[a];
        T L[S::NR];
#pragma unroll
        for (int k = 0; k < S::NR; ++k) L[k] = T(0);
        for (int q = beg + lane; q < stop; q += 32) {
            if (q >= rows) {
                set_error(ctr, ERR_BOUNDS);
                break;
            }
            const V16 *row = reinterpret_cast<const V16 *>(rbuf + (size_t)q * S::NRP);
#pragma unroll
            for (int c = 0; c < S::NV; ++c) {
                T v[S::V];
                *reinterpret_cast<V16 *>(v) = row[c];
#pragma unroll
                for (int e = 0; e < S::V; ++e)
                    if (c * S::V + e < S::NRC) L[c * S::V + e] += v[e];
            }
        }
        reduce_apply<T, S::NR, S::NRC>(L, lane, [&](int k, const T &x) { s_l[w][k] = x; });
        __syncwarp();
        if (lane == 0) {
            T l[S::NRP];
#pragma unroll
            for (int k = 0; k < S::NRC; ++k) l[k] = lpart[(size_t)a * S::NRP + k] + s_l[w][k];
            OpReduced<P>::template finish<T>(l, Lout + (size_t)a * S::NCP);
        }
        __syncwarp();
    }
}

template <class T, int P>
int launch_m2l_mutual_tp(Plan &P_, cudaStream_t s)
{
    const int launches = launch_mutual_index(P_, s);
    const long long rows = P_.mut_cap_em;
    const bool fresh = P_.mr_fresh;
    if (!fresh) k_moments_r<T, P, OpReduced<P>><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, (const T *)P_.M, (T *)P_.Mr);
    using MS = MutShape<T, P>;
    static_assert(MS::smem <= 227 * 1024, "mutual M2L staging exceeds shared memory");
    cudaFuncSetAttribute(k_m2l_mut1<T, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)MS::smem);
    k_m2l_mut1<T, P><<<P_.num_sms * 16 * (4 / MS::W), MS::W * 32, MS::smem, s>>>(
        P_.ctr, P_.order + P_.cap_nodes, P_.m2l_off, P_.m2l_src, P_.mut_lo, P_.mut_mir_m2l,
        (const vec4<T> *)P_.node_c, (const T *)P_.Mr, (T *)P_.mut_rm2l, rows, (T *)P_.mut_lpart, P_.ctr);
    k_m2l_mut2<T, P><<<P_.num_sms * 8, 256, 0, s>>>(P_.ctr, P_.m2l_off, P_.mut_lo, (const T *)P_.mut_rm2l, rows,
                                                    (const T *)P_.mut_lpart, (T *)P_.Lm2l, P_.ctr);
    return launches + (fresh ? 2 : 3);
}

template <class T>
int launch_m2l_mutual_t(Plan &P, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_m2l_mutual_tp<T, 0>(P, s);
    case 1: return launch_m2l_mutual_tp<T, 1>(P, s);
    case 2: return launch_m2l_mutual_tp<T, 2>(P, s);
    case 3: return launch_m2l_mutual_tp<T, 3>(P, s);
    case 4: return launch_m2l_mutual_tp<T, 4>(P, s);
    case 5: return launch_m2l_mutual_tp<T, 5>(P, s);
    case 6: return launch_m2l_mutual_tp<T, 6>(P, s);
    case 7: return launch_m2l_mutual_tp<T, 7>(P, s);
    default: return launch_m2l_mutual_tp<T, 8>(P, s);
    }
}

template <class T, int P, class Op>
int launch_m2l_op(Plan &P_, const void *M, void *Lout, cudaStream_t s)
{
    using S = M2LShape<T, P>;
    static_assert(S::NRP % S::V == 0, "row stride must be a whole number of 16-byte loads");
    static_assert(S::smem <= 227 * 1024, "M2L staging exceeds shared memory");
    // the forward moments' reduced rows come from the upward pass when it wrote them
    const bool fresh = std::is_same_v<Op, OpReduced<P>> && M == P_.M && P_.mr_fresh;
    if (!fresh) k_moments_r<T, P, Op><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, (const T *)M, (T *)P_.Mr);
    cudaFuncSetAttribute(k_m2l<T, P, Op>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::smem);
    k_m2l<T, P, Op><<<P_.num_sms * 16, M2L_WARPS * 32, S::smem, s>>>(
        P_.ctr, P_.order + P_.cap_nodes, P_.m2l_off, P_.m2l_src, (const vec4<T> *)P_.node_c,
        (const T *)P_.Mr, (T *)Lout, P_.ctr);
    return fresh ? 1 : 2;
}

template <class T, int P>
int launch_m2l_tp(Plan &P_, const void *M, void *Lout, cudaStream_t s)
{
    return P_.m2l_rotation ? launch_m2l_op<T, P, OpRotation<P>>(P_, M, Lout, s)
                           : launch_m2l_op<T, P, OpReduced<P>>(P_, M, Lout, s);
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
    // mutual plans: both directions per unordered pair, plain arithmetic in the plan's dtype
    if (P.mutual) return P.dtype == 0 ? launch_m2l_mutual_t<float>(P, s) : launch_m2l_mutual_t<double>(P, s);
    if (P.dtype == 0) return launch_m2l_t<float>(P, P.M, P.Lm2l, s);
    return P.p <= kMaxPDf && !P.f64_ieee && !P.m2l_rotation ? launch_m2l_df(P, s)
                                                            : launch_m2l_t<double>(P, P.M, P.Lm2l, s);
}

int launch_m2l_plain(Plan &P, const void *M, void *Lout, cudaStream_t s)
{
    return P.dtype == 0 ? launch_m2l_t<float>(P, M, Lout, s) : launch_m2l_t<double>(P, M, Lout, s);
}

}  // namespace bfm
