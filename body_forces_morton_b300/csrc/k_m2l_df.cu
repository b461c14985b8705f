// M2L of fp64 plans in double-float arithmetic on the FP32 pipe (orders <= 4;
// higher orders keep the fp64 kernel, their double-word accumulators would not
// fit in registers).
//
// The translation of JZ-FMM page, "Calculating a node-node interaction",
//     L_k(A) += -sum_{|n| <= p - |k|} (-1)^{|n|} M_n(B) D^{n+k}(R),  R = c_A - c_B,
// evaluated as in k_m2l (one warp per receiver, a lane per source, fixed-order
// lane reduction), but in double words (dfloat.cuh): the FP64 rate of this GPU
// is a small fraction of its FP32 rate.
//
// Units. fp32's exponent range cannot hold a node's moments and derivative
// tensor across the tree's depth in absolute units, so every node carries its
// level's cell half-size bound h = 2^(ex - level) (df_units) and masses are in
// 2^em. With the homogeneity D^m(R) = h^-(|m|+1) D^m(R / h):
//     M~_n(B) = M_n(B) / (2^em h_B^|n|)              (stored once per node),
//     L~_k(A) = sum_n (-1)^{|n|} [M~_n(B) (h_B / h_A)^|n|] D^{n+k}(R / h_A),
//     L_k(A)  = 2^em h_A^-(|k|+1) L~_k(A),
// every factor an exact power of two. The contraction runs on reduced
// (trace-free) coefficients as in k_m2l (Exp<P>::reduce_m / expand_l; the
// powers of two depend only on the degree, which the reduction keeps). A pair
// outside the ranges these units are
// made for (level gap above kMaxDl, |R / h_A|^2 outside [kR2Lo, kR2Hi]) skips the
// double-word pass and is evaluated in a second, fp64 pass over the receiver's
// list, added after the first; typical trees never take it.
#include "expansions_df_gen.cuh"
#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

constexpr int MD_WARPS = 4;
constexpr int kMaxDl = 8;
constexpr float kR2Lo = 0x1p-30f, kR2Hi = 0x1p30f;

// total degree of reduced coefficient r (degree d holds 2d + 1 of them, from d^2 on)
__device__ __forceinline__ int rdegree_of(int r)
{
    return (r >= 1) + (r >= 4) + (r >= 9) + (r >= 16);
}

template <int P> struct MDShape {
    static constexpr int NC = ExpDF<P>::NC;
    static constexpr int NCP = (NC + 3) / 4 * 4;  // row stride of M and L in global memory
    static constexpr int NRC = ExpDF<P>::NRC;     // reduced coefficients
    static constexpr int NRP = (NRC + 3) / 4 * 4; // row stride of the reduced moments (double words)
    static constexpr int STR = NRP + 1;           // odd row stride (8-byte words) in shared memory
    static constexpr int NV = NRP / 2;            // 16-byte loads per row (two double words each)
    static constexpr int NR = (NRC + 7) / 8 * 8;  // accumulators, padded for the halving reduction
    static constexpr int NRF = (NC + 7) / 8 * 8;  // full accumulators of the fp64 second pass
    static constexpr size_t smem = sizeof(df) * MD_WARPS * 32 * STR + sizeof(double) * MD_WARPS * NRC;
};

// Reduced moments in their node's units: Mr[b][r] = reduce_m(M[b])_r 2^-(em + (ex - level_b) |r|).
template <int P>
__global__ __launch_bounds__(256) void k_moments_df(const DevCounters *__restrict__ nctr, const int *__restrict__ level,
                                                    const dbl4 *__restrict__ node_l, const double *__restrict__ M,
                                                    df *__restrict__ Mr)
{
    const int n_nodes = phase2_nodes(nctr);
    using S = MDShape<P>;
    if (n_nodes <= 0) return;
    int ex, em;
    df_units(node_l, M, ex, em);
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < n_nodes; b += gridDim.x * blockDim.x) {
        double r[S::NRC];
        Exp<P>::template reduce_m<double>(M + (size_t)b * S::NCP, r);
        const int eb = ex - level[b];
#pragma unroll
        for (int i = 0; i < S::NRP; ++i)
            Mr[(size_t)b * S::NRP + i] = df_from(i < S::NRC ? ldexp(r[i], -em - eb * rdegree_of(i)) : 0.0);
    }
}

// Separation in the receiver's units and whether the double-word pass takes the pair.
struct PairGeom {
    df rx, ry, rz;
    int dl;
    bool ok;
};

__device__ __forceinline__ PairGeom pair_geom(const dbl4 &ca, int la, int ea, const dbl4 &cb, int lb)
{
    PairGeom g;
    g.rx = df_from(ldexp(ca.x - cb.x, -ea));
    g.ry = df_from(ldexp(ca.y - cb.y, -ea));
    g.rz = df_from(ldexp(ca.z - cb.z, -ea));
    g.dl = la - lb;
    const float r2 = g.rx.h * g.rx.h + g.ry.h * g.ry.h + g.rz.h * g.rz.h;
    g.ok = g.dl <= kMaxDl && g.dl >= -kMaxDl && r2 >= kR2Lo && r2 <= kR2Hi;
    return g;
}

// Six blocks (24 warps) per SM: the unrolled double-float body needs more warps
// than its full register set allows to hide instruction fetch, and measured
// faster at 80 registers with some spilling (0.50 ms) than at 253 (0.72 ms).
template <int P>
__global__ __launch_bounds__(MD_WARPS * 32, 6) void k_m2l_df(const DevCounters *__restrict__ nctr, const int *__restrict__ order,
                                                          const int *__restrict__ off, const int *__restrict__ src,
                                                          const dbl4 *__restrict__ nc, const int *__restrict__ level,
                                                          const dbl4 *__restrict__ node_l,
                                                          const double *__restrict__ M, const df *__restrict__ Mr,
                                                          double *__restrict__ Lout, DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    using S = MDShape<P>;
    extern __shared__ __align__(16) unsigned char m2l_df_smem[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    df *rows = reinterpret_cast<df *>(m2l_df_smem) + (size_t)w * 32 * S::STR;
    double *lred = reinterpret_cast<double *>(reinterpret_cast<df *>(m2l_df_smem) + (size_t)MD_WARPS * 32 * S::STR) +
                   (size_t)w * S::NRC;
    int ex = 0, em = 0;
    if (n_nodes > 0) df_units(node_l, M, ex, em);
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[1], 1);
        t = __shfl_sync(kFull, t, 0);
        if (t >= n_nodes) break;
        const int a = order[t];
        const int beg = off[a], end = off[a + 1];
        const dbl4 ca = nc[a];
        const int la = level[a], ea = ex - la;
        dacc L[S::NR];
#pragma unroll
        for (int k = 0; k < S::NR; ++k) L[k] = dacc{0.0f, 0.0f};
        bool wide = false;
        for (int q0 = beg; q0 < end; q0 += 32) {
            const int q = q0 + lane;
            const bool valid = q < end;
            const int b = valid ? src[q] : 0;
            PairGeom g{};
            if (valid) g = pair_geom(ca, la, ea, nc[b], level[b]);
            wide |= valid && !g.ok;
            const int nsrc = min(32, end - q0);
            const int dls = max(-kMaxDl, min(kMaxDl, g.dl));
            __syncwarp();
            // stage this round's reduced source rows, each scaled by (h_B / h_A)^|n| = 2^(dl |n|)
            for (int t0 = 0; t0 < nsrc * S::NV; t0 += 32) {
                const int tt = t0 + lane;
                const int row = tt / S::NV, col = tt - row * S::NV;
                const int bb = __shfl_sync(kFull, b, row & 31);
                const int d = __shfl_sync(kFull, dls, row & 31);
                if (tt < nsrc * S::NV) {
                    const float4 x = __ldg(reinterpret_cast<const float4 *>(Mr + (size_t)bb * S::NRP) + col);
                    const int n0 = 2 * col;
                    rows[row * S::STR + n0] = df_scale(df_make(x.x, x.y), pow2f(d * rdegree_of(n0)));
                    rows[row * S::STR + n0 + 1] = df_scale(df_make(x.z, x.w), pow2f(d * rdegree_of(n0 + 1)));
                }
            }
            __syncwarp();
            if (valid && g.ok) ExpDF<P>::m2l_r(rows + lane * S::STR, g.rx, g.ry, g.rz, L);
        }
        df v[S::NR];
#pragma unroll
        for (int k = 0; k < S::NR; ++k) v[k] = dacc_value(L[k]);
        double *dst = Lout + (size_t)a * S::NCP;
        reduce_apply<df, S::NR, S::NRC>(v, lane, [&](int k, const df &x) {
            lred[k] = ldexp(df_to(x), em - ea * (rdegree_of(k) + 1));
        });
        __syncwarp();
        if (lane == 0) Exp<P>::template expand_l<double>(lred, dst);
        if (__any_sync(kFull, wide)) {
            // fp64 pass over the pairs the double-word units do not cover
            __syncwarp();
            double Lw[S::NRF];
#pragma unroll
            for (int k = 0; k < S::NRF; ++k) Lw[k] = 0.0;
            for (int q = beg + lane; q < end; q += 32) {
                const int b = src[q];
                const dbl4 cb = nc[b];
                if (!pair_geom(ca, la, ea, cb, level[b]).ok)
                    Exp<P>::template m2l<double>(M + (size_t)b * S::NCP, ca.x - cb.x, ca.y - cb.y, ca.z - cb.z, Lw);
            }
            reduce_apply<double, S::NRF, S::NC>(Lw, lane, [&](int k, double x) { dst[k] += x; });
        }
    }
}

template <int P>
int launch_m2l_df_p(Plan &P_, cudaStream_t s)
{
    using S = MDShape<P>;
    static_assert(S::NRP % 2 == 0, "rows must be whole 16-byte loads");
    k_moments_df<P><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, P_.node_level, (const dbl4 *)P_.node_l,
                                                   (const double *)P_.M, (df *)P_.Mr);
    cudaFuncSetAttribute(k_m2l_df<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::smem);
    k_m2l_df<P><<<P_.num_sms * 16, MD_WARPS * 32, S::smem, s>>>(
        P_.ctr, P_.order + P_.cap_nodes, P_.m2l_off, P_.m2l_src, (const dbl4 *)P_.node_c, P_.node_level,
        (const dbl4 *)P_.node_l, (const double *)P_.M, (const df *)P_.Mr, (double *)P_.Lm2l, P_.ctr);
    return 2;
}

}  // namespace

int launch_m2l_df(Plan &P, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_m2l_df_p<0>(P, s);
    case 1: return launch_m2l_df_p<1>(P, s);
    case 2: return launch_m2l_df_p<2>(P, s);
    case 3: return launch_m2l_df_p<3>(P, s);
    default: return launch_m2l_df_p<4>(P, s);
    }
}

}  // namespace bfm
