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
//   k_vjp_up        one launch, deepest level first, eight lanes per node: a
//                   leaf's moments from its particles (Exp<P>::p2m_dip), an
//                   internal node's from its children (m2m) once their flags
//                   are set, summed in a fixed order;
//   M2L and L2L     the forward kernels on the source moments (plain
//                   arithmetic in the plan's dtype);
//   k_vjp_far       a thread per particle: Phi_s and its gradient from the
//                   source locals, the forward Hessian from L
//                   (Exp<P>::l2p_hess), combined with the particle's own
//                   cotangents into (Phi_s, xbar) of the far field;
//   k_vjp_near      the P2P lists, with the work items, lane layout, staging and
//                   chunk order of the forward near field: per pair the direct
//                   terms of Phi_s, of m_i grad Phi_s and of -Hess Phi abar_i,
//                   added to the far field and written in the caller's order.
#include <type_traits>

#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

constexpr int VJP_WARPS = 4;                                                // warps per block of k_vjp_near
template <class T> struct VjpChunk { static constexpr int value = 128; };  // staged sources per warp
template <> struct VjpChunk<double> { static constexpr int value = 64; };
// receivers per lane of k_vjp_near, in both paths: four (the packed fp32 path also fills the lanes of
// partly filled leaves better than with two)
template <class T> struct VjpK { static constexpr int value = 4; };

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

// Source moments of every node in one launch, ordered like the forward upward
// pass of fp32 plans (without the boxes, which the forward evaluation left):
// warps take chunks of four nodes of one level from a shared counter, deepest
// level first, eight lanes per node. A leaf's lanes expand its particles'
// sources (Exp<P>::p2m_dip); an internal node's lanes wait, bounded, until each
// child's flag holds this pass's number and add its M2M translation. A fixed
// 8-lane reduction sums the lanes; the node's flag is then stored with release
// semantics. A chunk never spans two levels and every child lies in an earlier
// chunk, taken by a running warp, so the earliest unfinished chunk can always
// finish.
template <class T, int P>
__global__ __launch_bounds__(256) void k_vjp_up(DevCounters *ctr, const int *__restrict__ first,
                                                const int *__restrict__ count, const int *__restrict__ child0,
                                                const int *__restrict__ nchild, const vec4<T> *__restrict__ nc,
                                                const vec4<T> *__restrict__ xyzm, const vec4<T> *__restrict__ src,
                                                T *Ms, int ncp, unsigned *flag, unsigned seq)
{
    constexpr int NC = Exp<P>::NC;
    constexpr int NR = (NC + 7) / 8 * 8;
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
        const bool has = j < nch;
        const vec4<T> c = valid ? nc[a] : make4<T>(T(0), T(0), T(0), T(0));
        T m[NR];
#pragma unroll
        for (int k = 0; k < NR; ++k) m[k] = T(0);
        if (leaf) {
            const int f = first[a], e = f + count[a];
            for (int i = f + j; i < e; i += 8) {
                const vec4<T> x = xyzm[i], sv = src[i];
                Exp<P>::template p2m_dip<T>(x.x - c.x, x.y - c.y, x.z - c.z, sv.x, sv.y, sv.z, sv.w, m);
            }
        } else if (has) {
            const int ch = child0[a] + j;
            cuda::atomic_ref<unsigned, cuda::thread_scope_device> fl(flag[ch]);
            unsigned spins = 0;
            while (fl.load(cuda::memory_order_acquire) != seq) {
                if (++spins > kSpinLimit) {
                    set_error(ctr, ERR_SPIN);
                    break;
                }
                __nanosleep(32);
            }
            T mc[NC];
#pragma unroll
            for (int k = 0; k < NC; ++k) mc[k] = ld_cg(Ms + (size_t)ch * ncp + k);
            const vec4<T> cc = nc[ch];
            Exp<P>::template m2m<T>(mc, cc.x - c.x, cc.y - c.y, cc.z - c.z, m);
        }
        T *dst = Ms + (size_t)a * ncp;
        reduce_apply8<T, NR, NC>(m, j, [&](int k, const T &x) {
            if (valid) dst[k] = x;
        });
        __threadfence();
        __syncwarp();
        if (valid && j == 0)
            cuda::atomic_ref<unsigned, cuda::thread_scope_device>(flag[a]).store(seq, cuda::memory_order_release);
    }
}

// Far field of the VJP at the leaves' particles, in the sorted order (a warp
// per leaf, a lane per particle): far = (Phi_s, m_i grad Phi_s - H abar_i -
// pbar_i a_i) with Phi_s and its gradient from the source locals Ls and the
// forward Hessian H from the forward locals L.
template <class T, int P>
__global__ __launch_bounds__(256) void k_vjp_far(const DevCounters *__restrict__ ctr, const int *__restrict__ first,
                                                 const int *__restrict__ count, const int *__restrict__ nchild,
                                                 const vec4<T> *__restrict__ nc, const vec4<T> *__restrict__ xyzm,
                                                 const vec4<T> *__restrict__ src, const uint32_t *__restrict__ perm,
                                                 const T *__restrict__ L, const T *__restrict__ Ls, int ncp,
                                                 const T *__restrict__ acc_fwd, vec4<T> *__restrict__ far)
{
    const int n_nodes = phase2_nodes(ctr);
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a];
        const vec4<T> ca = nc[a];
        for (int i = f + lane; i < f + c; i += 32) {
            const vec4<T> xi = xyzm[i], si = src[i];
            const T dx = xi.x - ca.x, dy = xi.y - ca.y, dz = xi.z - ca.z;
            T phis = T(0), ngx = T(0), ngy = T(0), ngz = T(0);
            Exp<P>::template l2p<T>(Ls + (size_t)a * ncp, dx, dy, dz, phis, ngx, ngy, ngz);
            T H[6] = {T(0), T(0), T(0), T(0), T(0), T(0)};
            Exp<P>::template l2p_hess<T>(L + (size_t)a * ncp, dx, dy, dz, H);
            const T bx = -si.y, by = -si.z, bz = -si.w;  // the particle's own cotangent abar
            const T hx = H[0] * bx + H[1] * by + H[2] * bz;
            const T hy = H[1] * bx + H[3] * by + H[4] * bz;
            const T hz = H[2] * bx + H[4] * by + H[5] * bz;
            const T *ai = acc_fwd + 3 * (size_t)perm[i];
            far[i] = make4<T>(phis, -xi.w * ngx - hx - si.x * ai[0], -xi.w * ngy - hy - si.x * ai[1],
                              -xi.w * ngz - hz - si.x * ai[2]);
        }
    }
}

// One source j (position and mass xj; monopole q and dipole d in sj = (q, d))
// acting on one receiver i (position and mass p, cotangent b = abar_i), with
// u = x_i - x_j:
//   A[0] += -q / r - d.u / r^3                                  (Phi_s)
//   A[1..3] += u (m_i q / r^3 + 3 (m_i d.u + m_j b.u) / r^5) - m_i d / r^3
//   A[4] += m_j / r^3
// so that m_i grad Phi_s - Hess Phi b of the pair is A[1..3] - A[4] b (the
// Hessian of -m_j / r is m_j (r^2 I - 3 u u^T) / r^5). The own leaf holds the
// receiver itself (zero separation), which MASKED skips.
template <class T, bool MASKED>
__device__ __forceinline__ void vjp_pair(const vec4<T> &xj, const vec4<T> &sj, const vec4<T> &p, const vec4<T> &b,
                                         T (&A)[5])
{
    const T ux = p.x - xj.x, uy = p.y - xj.y, uz = p.z - xj.z;
    const T r2 = ux * ux + uy * uy + uz * uz;
    T ri = rsqrt_t(r2);
    if (MASKED) ri = r2 > T(0) ? ri : T(0);
    const T ir2 = ri * ri, ir3 = ir2 * ri, ir5 = T(3) * ir3 * ir2;
    const T wd = sj.y * ux + sj.z * uy + sj.w * uz;
    const T wb = b.x * ux + b.y * uy + b.z * uz;
    A[0] -= sj.x * ri + wd * ir3;
    const T cu = p.w * sj.x * ir3 + (p.w * wd + xj.w * wb) * ir5;
    const T mi3 = p.w * ir3;
    A[1] += cu * ux - mi3 * sj.y;
    A[2] += cu * uy - mi3 * sj.z;
    A[3] += cu * uz - mi3 * sj.w;
    A[4] += xj.w * ir3;
}

// Interactions of the staged sources q, q + S, ... with K receivers.
template <class T, bool MASKED, int K>
__device__ __forceinline__ void vjp_span(const vec4<T> *bx, const vec4<T> *bs, int n_here, int q, int S,
                                         const vec4<T> (&p)[K], const vec4<T> (&b)[K], T (&A)[K][5])
{
    for (int j = q; j < n_here; j += S) {
        const vec4<T> xj = bx[j], sj = bs[j];
#pragma unroll
        for (int k = 0; k < K; ++k) vjp_pair<T, MASKED>(xj, sj, p[k], b[k], A[k]);
    }
}

// Copy one particle's position-mass and source records into shared memory.
template <class T>
__device__ __forceinline__ void vjp_copy(vec4<T> *dx, vec4<T> *ds, const vec4<T> *sx, const vec4<T> *ss)
{
#pragma unroll
    for (int h = 0; h < (int)sizeof(vec4<T>); h += 16) {
        cp_async16(reinterpret_cast<char *>(dx) + h, reinterpret_cast<const char *>(sx) + h);
        cp_async16(reinterpret_cast<char *>(ds) + h, reinterpret_cast<const char *>(ss) + h);
    }
}

// Stage sources [g0, g0 + CH) of the concatenation of the current group's
// source leaves. Lane i holds the group's i-th leaf: first particle fb and
// exclusive prefix ex of the counts (ascending over the lanes).
template <class T, int CH>
__device__ __forceinline__ int vjp_stage(vec4<T> *bx, vec4<T> *bs, const vec4<T> *__restrict__ xyzm,
                                         const vec4<T> *__restrict__ src, int fb, int ex, int tot, int g0, int lane)
{
    const int n_here = min(CH, tot - g0);
    for (int k0 = 0; k0 < n_here; k0 += 32) {  // warp-uniform: every lane takes part in the shuffles
        const int k = k0 + lane;
        const int g = g0 + k;
        int lo = 0;  // last lane whose leaf starts at or before g
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const int exm = __shfl_sync(kFull, ex, lo + step);
            lo = exm <= g ? lo + step : lo;
        }
        const int f = __shfl_sync(kFull, fb, lo);
        const int e = __shfl_sync(kFull, ex, lo);
        if (k < n_here) vjp_copy<T>(bx + k, bs + k, xyzm + f + (g - e), src + f + (g - e));
    }
    cp_async_wait_all();
    return n_here;
}

// One round of up to 32 K receivers [r0, r0 + cr) of leaf a, laid out as in
// the forward near field: lane = q R + rp (rp < R = ceil(cr / K), q < S =
// 32 / R) holds receivers rp + k R, k < K, and walks the staged sources from
// offset q with stride S; lanes at or beyond R S only stage. The S partial
// sums of a receiver are added in order of q, and a split receiver's chunks in
// chunk order, so the result is reproducible.
template <class T, int K, bool CHUNKED>
__device__ __forceinline__ void vjp_round(int a, int f, int c, int r0, int cr, int beg, int end, int chunk, int nch,
                                          int *done, DevCounters *ctr, const int *__restrict__ first,
                                          const int *__restrict__ count, const vec4<T> *__restrict__ xyzm,
                                          const vec4<T> *__restrict__ src, const uint32_t *__restrict__ perm,
                                          const vec4<T> *far, vec4<T> *far_w, const int *__restrict__ lsrc,
                                          T *__restrict__ pos_bar, T *__restrict__ mass_bar, vec4<T> *bx,
                                          vec4<T> *bs, T (*red)[4], int lane)
{
    constexpr int CH = VjpChunk<T>::value;
    const int R = (cr + K - 1) / K, S = 32 / R;
    const int rp = lane % R, q = lane / R;
    vec4<T> p[K], b[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int rr = rp + k * R;
        const int i = f + r0 + (rr < cr ? rr : 0);
        p[k] = xyzm[i];
        const vec4<T> si = src[i];
        b[k] = make4<T>(-si.y, -si.z, -si.w, T(0));
    }
    T A[K][5];
#pragma unroll
    for (int k = 0; k < K; ++k)
#pragma unroll
        for (int v = 0; v < 5; ++v) A[k][v] = T(0);
    const int qq = q < S ? q : (1 << 30);  // idle lanes start past every chunk
    // the leaf's own particles (zero separations possible; the first chunk of a split receiver)
    for (int g0 = 0; (!CHUNKED || chunk == 0) && g0 < c; g0 += CH) {
        const int n_here = min(CH, c - g0);
        __syncwarp();
        for (int k = lane; k < n_here; k += 32) vjp_copy<T>(bx + k, bs + k, xyzm + f + g0 + k, src + f + g0 + k);
        cp_async_wait_all();
        __syncwarp();
        vjp_span<T, true, K>(bx, bs, n_here, qq, S, p, b, A);
    }
    // every other source leaf of the list, 32 entries at a time (lane i holds entry lb + i)
    for (int lb = beg; lb < end; lb += 32) {
        const int e = lb + lane;
        int fb = 0, cb = 0;
        if (e < end) {
            const int bb = lsrc[e];
            if (bb != a) {
                fb = first[bb];
                cb = count[bb];
            }
        }
        const int incl = warp_incl_scan(cb);
        const int tot = __shfl_sync(kFull, incl, 31);
        const int ex = incl - cb;
        for (int g0 = 0; g0 < tot; g0 += CH) {
            __syncwarp();
            const int n_here = vjp_stage<T, CH>(bx, bs, xyzm, src, fb, ex, tot, g0, lane);
            __syncwarp();
            vjp_span<T, false, K>(bx, bs, n_here, qq, S, p, b, A);
        }
    }
    if (CHUNKED && r0 == 0) wait_turn(done + a, chunk, ctr);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        __syncwarp();
        red[lane][0] = A[k][0];
        red[lane][1] = A[k][1] - A[k][4] * b[k].x;
        red[lane][2] = A[k][2] - A[k][4] * b[k].y;
        red[lane][3] = A[k][3] - A[k][4] * b[k].z;
        __syncwarp();
        const int rr = rp + k * R;
        if (q == 0 && rr < cr) {
            T t[4] = {red[rp][0], red[rp][1], red[rp][2], red[rp][3]};
            for (int qs = 1; qs < S; ++qs)
#pragma unroll
                for (int v = 0; v < 4; ++v) t[v] += red[qs * R + rp][v];
            const int i = f + r0 + rr;
            // the far field plus the earlier chunks' partial sums (written by other warps through far_w,
            // which aliases far: a coherent L2 load then)
            const vec4<T> fa = CHUNKED ? ld_cg(far + i) : far[i];
            if (CHUNKED && chunk < nch - 1) {
                far_w[i] = make4<T>(fa.x + t[0], fa.y + t[1], fa.z + t[2], fa.w + t[3]);
            } else {
                const uint32_t o = perm[i];
                pos_bar[3 * (size_t)o] = fa.y + t[1];
                pos_bar[3 * (size_t)o + 1] = fa.z + t[2];
                pos_bar[3 * (size_t)o + 2] = fa.w + t[3];
                mass_bar[o] = fa.x + t[0];
            }
        }
    }
}

// ---- fp32: two sources per instruction in packed f32x2 arithmetic ----------
// The staged sources are stored pair-interleaved, per pair of sources (x, y,
// z, m, q, d_x, d_y, d_z) with the two sources' values adjacent (16 floats), so
// four 16-byte shared loads give eight packed operands; an odd tail is padded
// with a massless, source-free particle far away. With u = x_j - x_i the pair
// terms become Phi_s += d.u / r^3 - q / r (accumulated as two sums, Q and P),
// X += c u - m_i d / r^3 with c = 3 (m_i d.u + m_j b.u) / r^5 - m_i q / r^3,
// and SM += m_j / r^3, the same quantities as vjp_pair with u of the opposite
// sign; the receiver's mass enters negated once per receiver, so no pair
// needs a negation.
struct VjpRecv {
    float2 nx, ny, nz, m, nm, bx, by, bz;  // -x_i (both halves), m_i, -m_i, abar_i
};

__device__ __forceinline__ float rsqrt_approx_ftz(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <bool MASKED>
__device__ __forceinline__ void vjp_two(const float4 &s0, const float4 &s1, const float4 &s2, const float4 &s3,
                                        const VjpRecv &r, float2 (&A)[6])
{
    const float2 ux = __fadd2_rn(make_float2(s0.x, s0.y), r.nx);
    const float2 uy = __fadd2_rn(make_float2(s0.z, s0.w), r.ny);
    const float2 uz = __fadd2_rn(make_float2(s1.x, s1.y), r.nz);
    const float2 mj = make_float2(s1.z, s1.w), qj = make_float2(s2.x, s2.y);
    const float2 dx = make_float2(s2.z, s2.w), dy = make_float2(s3.x, s3.y), dz = make_float2(s3.z, s3.w);
    float2 r2 = __fmul2_rn(ux, ux);
    r2 = __ffma2_rn(uy, uy, r2);
    r2 = __ffma2_rn(uz, uz, r2);
    float2 ri = make_float2(rsqrt_approx_ftz(r2.x), rsqrt_approx_ftz(r2.y));
    if (MASKED) ri = make_float2(r2.x > 0.0f ? ri.x : 0.0f, r2.y > 0.0f ? ri.y : 0.0f);
    const float2 ir2 = __fmul2_rn(ri, ri);
    const float2 ir3 = __fmul2_rn(ir2, ri);
    const float2 ir5 = __fmul2_rn(ir3, __fmul2_rn(ir2, make_float2(3.0f, 3.0f)));
    float2 wd = __fmul2_rn(dx, ux);
    wd = __ffma2_rn(dy, uy, wd);
    wd = __ffma2_rn(dz, uz, wd);
    float2 wb = __fmul2_rn(r.bx, ux);
    wb = __ffma2_rn(r.by, uy, wb);
    wb = __ffma2_rn(r.bz, uz, wb);
    A[0] = __ffma2_rn(qj, ri, A[0]);   // P = sum q / r
    A[1] = __ffma2_rn(wd, ir3, A[1]);  // Q = sum d.u / r^3
    float2 t = __fmul2_rn(r.m, wd);
    t = __ffma2_rn(mj, wb, t);
    const float2 cu = __ffma2_rn(r.nm, __fmul2_rn(qj, ir3), __fmul2_rn(t, ir5));
    const float2 nmi3 = __fmul2_rn(r.nm, ir3);
    A[2] = __ffma2_rn(nmi3, dx, __ffma2_rn(cu, ux, A[2]));
    A[3] = __ffma2_rn(nmi3, dy, __ffma2_rn(cu, uy, A[3]));
    A[4] = __ffma2_rn(nmi3, dz, __ffma2_rn(cu, uz, A[4]));
    A[5] = __ffma2_rn(mj, ir3, A[5]);  // SM = sum m_j / r^3
}

// Source k of the staging buffer into its pair-interleaved slots (asynchronous 4-byte copies).
__device__ __forceinline__ void vjp_copy_pair(float *fb, int k, const float4 *x, const float4 *sv)
{
    float *d = fb + (k >> 1) * 16 + (k & 1);
    const float *a = reinterpret_cast<const float *>(x), *b = reinterpret_cast<const float *>(sv);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        cp_async4(d + 2 * v, a + v);
        cp_async4(d + 8 + 2 * v, b + v);
    }
}

__device__ __forceinline__ void vjp_pad_pair(float *fb, int k)
{
    float *d = fb + (k >> 1) * 16 + (k & 1);
    d[0] = d[2] = d[4] = 1e18f;
    d[6] = d[8] = d[10] = d[12] = d[14] = 0.0f;
}

template <int CH>
__device__ __forceinline__ int vjp_stage_pairs(float *fb, const float4 *__restrict__ xyzm,
                                               const float4 *__restrict__ src, int lf, int ex, int tot, int g0,
                                               int lane)
{
    const int n_here = min(CH, tot - g0);
    for (int k0 = 0; k0 < n_here; k0 += 32) {  // warp-uniform: every lane takes part in the shuffles
        const int k = k0 + lane;
        const int g = g0 + k;
        int lo = 0;
#pragma unroll
        for (int step = 16; step > 0; step >>= 1) {
            const int exm = __shfl_sync(kFull, ex, lo + step);
            lo = exm <= g ? lo + step : lo;
        }
        const int f = __shfl_sync(kFull, lf, lo);
        const int e = __shfl_sync(kFull, ex, lo);
        if (k < n_here) vjp_copy_pair(fb, k, xyzm + f + (g - e), src + f + (g - e));
    }
    if ((n_here & 1) && lane == 0) vjp_pad_pair(fb, n_here);
    cp_async_wait_all();
    return (n_here + 1) >> 1;
}

template <int K, bool MASKED>
__device__ __forceinline__ void vjp_span_pairs(const float *fb, int npairs, int q, int S, const VjpRecv (&r)[K],
                                               float2 (&A)[K][6])
{
    const float4 *pb = reinterpret_cast<const float4 *>(fb);
    for (int j = q; j < npairs; j += S) {
        const float4 s0 = pb[4 * j], s1 = pb[4 * j + 1], s2 = pb[4 * j + 2], s3 = pb[4 * j + 3];
#pragma unroll
        for (int k = 0; k < K; ++k) vjp_two<MASKED>(s0, s1, s2, s3, r[k], A[k]);
    }
}

// vjp_round for fp32 plans: the same lane layout and order of sums, the pair
// terms by vjp_two on pair-interleaved sources.
template <int K, bool CHUNKED>
__device__ __forceinline__ void vjp_round_f32(int a, int f, int c, int r0, int cr, int beg, int end, int chunk,
                                              int nch, int *done, DevCounters *ctr, const int *__restrict__ first,
                                              const int *__restrict__ count, const float4 *__restrict__ xyzm,
                                              const float4 *__restrict__ src, const uint32_t *__restrict__ perm,
                                              const float4 *far, float4 *far_w, const int *__restrict__ lsrc,
                                              float *__restrict__ pos_bar, float *__restrict__ mass_bar, float *fb,
                                              float (*red)[4], int lane)
{
    constexpr int CH = VjpChunk<float>::value;
    const int R = (cr + K - 1) / K, S = 32 / R;
    const int rp = lane % R, q = lane / R;
    VjpRecv rv[K];
    float2 A[K][6];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int rr = rp + k * R;
        const int i = f + r0 + (rr < cr ? rr : 0);
        const float4 x = xyzm[i], sv = src[i];
        rv[k].nx = make_float2(-x.x, -x.x);
        rv[k].ny = make_float2(-x.y, -x.y);
        rv[k].nz = make_float2(-x.z, -x.z);
        rv[k].m = make_float2(x.w, x.w);
        rv[k].nm = make_float2(-x.w, -x.w);
        rv[k].bx = make_float2(-sv.y, -sv.y);
        rv[k].by = make_float2(-sv.z, -sv.z);
        rv[k].bz = make_float2(-sv.w, -sv.w);
#pragma unroll
        for (int v = 0; v < 6; ++v) A[k][v] = make_float2(0.0f, 0.0f);
    }
    const int qq = q < S ? q : (1 << 30);
    // the leaf's own particles (zero separations masked; the first chunk of a split receiver)
    for (int g0 = 0; (!CHUNKED || chunk == 0) && g0 < c; g0 += CH) {
        const int n_here = min(CH, c - g0);
        __syncwarp();
        for (int k = lane; k < n_here; k += 32) vjp_copy_pair(fb, k, xyzm + f + g0 + k, src + f + g0 + k);
        if ((n_here & 1) && lane == 0) vjp_pad_pair(fb, n_here);
        cp_async_wait_all();
        __syncwarp();
        vjp_span_pairs<K, true>(fb, (n_here + 1) >> 1, qq, S, rv, A);
    }
    for (int lb = beg; lb < end; lb += 32) {
        const int e = lb + lane;
        int fs = 0, cs = 0;
        if (e < end) {
            const int bb = lsrc[e];
            if (bb != a) {
                fs = first[bb];
                cs = count[bb];
            }
        }
        const int incl = warp_incl_scan(cs);
        const int tot = __shfl_sync(kFull, incl, 31);
        const int ex = incl - cs;
        for (int g0 = 0; g0 < tot; g0 += CH) {
            __syncwarp();
            const int npairs = vjp_stage_pairs<CH>(fb, xyzm, src, fs, ex, tot, g0, lane);
            __syncwarp();
            vjp_span_pairs<K, false>(fb, npairs, qq, S, rv, A);
        }
    }
    if (CHUNKED && r0 == 0) wait_turn(done + a, chunk, ctr);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const float sm = A[k][5].x + A[k][5].y;
        __syncwarp();
        red[lane][0] = (A[k][1].x + A[k][1].y) - (A[k][0].x + A[k][0].y);
        red[lane][1] = (A[k][2].x + A[k][2].y) - sm * rv[k].bx.x;
        red[lane][2] = (A[k][3].x + A[k][3].y) - sm * rv[k].by.x;
        red[lane][3] = (A[k][4].x + A[k][4].y) - sm * rv[k].bz.x;
        __syncwarp();
        const int rr = rp + k * R;
        if (q == 0 && rr < cr) {
            float t[4] = {red[rp][0], red[rp][1], red[rp][2], red[rp][3]};
            for (int qs = 1; qs < S; ++qs)
#pragma unroll
                for (int v = 0; v < 4; ++v) t[v] += red[qs * R + rp][v];
            const int i = f + r0 + rr;
            const float4 fa = CHUNKED ? ld_cg(far + i) : far[i];
            if (CHUNKED && chunk < nch - 1) {
                far_w[i] = make_float4(fa.x + t[0], fa.y + t[1], fa.z + t[2], fa.w + t[3]);
            } else {
                const uint32_t o = perm[i];
                pos_bar[3 * (size_t)o] = fa.y + t[1];
                pos_bar[3 * (size_t)o + 1] = fa.z + t[2];
                pos_bar[3 * (size_t)o + 2] = fa.w + t[3];
                mass_bar[o] = fa.x + t[0];
            }
        }
    }
}

// The near field of the VJP: the forward evaluation's P2P work items (a
// receiving leaf, or one chunk of a split one), taken from a shared counter
// in decreasing order of work, a warp each.
template <class T, int K>
__global__ __launch_bounds__(VJP_WARPS * 32) void k_vjp_near(
    const DevCounters *__restrict__ cst, const int2 *__restrict__ items, int *done, DevCounters *ctr,
    const int *__restrict__ first, const int *__restrict__ count, const vec4<T> *__restrict__ xyzm,
    const vec4<T> *__restrict__ src, const uint32_t *__restrict__ perm, const vec4<T> *far, vec4<T> *far_w,
    const int *__restrict__ off, const int *__restrict__ lsrc, T *__restrict__ pos_bar, T *__restrict__ mass_bar)
{
    constexpr int CH = VjpChunk<T>::value;
    __shared__ __align__(16) unsigned char s_buf[VJP_WARPS][2 * CH * sizeof(vec4<T>)];  // staged sources
    __shared__ T s_red[VJP_WARPS][32][4];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int n_work = 0;
    for (int bkt = 1; bkt < 64; ++bkt) n_work += cst->order_cnt[0][bkt];
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[0], 1);
        t = __shfl_sync(kFull, t, 0);
        if (t >= n_work) break;
        const int2 item = items[t];
        const int a = item.x, nch = item.y >> 8, chunk = item.y & 255;
        const int f = first[a], c = count[a];
        int beg = off[a], end = off[a + 1];
        if (nch > 1) {
            const int len = end - beg;
            end = beg + len * (chunk + 1) / nch;
            beg = beg + len * chunk / nch;
        }
        vec4<T> *const bx = reinterpret_cast<vec4<T> *>(s_buf[w]), *const bs = bx + CH;
        for (int r0 = 0; r0 < c; r0 += 32 * K) {
            const int cr = min(32 * K, c - r0);
            if constexpr (std::is_same<T, float>::value) {
                float *const fb = reinterpret_cast<float *>(s_buf[w]);  // CH sources of 8 floats
                if (nch == 1)
                    vjp_round_f32<K, false>(a, f, c, r0, cr, beg, end, 0, 1, done, ctr, first, count, xyzm, src,
                                            perm, far, far_w, lsrc, pos_bar, mass_bar, fb, s_red[w], lane);
                else
                    vjp_round_f32<K, true>(a, f, c, r0, cr, beg, end, chunk, nch, done, ctr, first, count, xyzm,
                                           src, perm, far, far_w, lsrc, pos_bar, mass_bar, fb, s_red[w], lane);
            } else {
                if (nch == 1)
                    vjp_round<T, K, false>(a, f, c, r0, cr, beg, end, 0, 1, done, ctr, first, count, xyzm, src,
                                           perm, far, far_w, lsrc, pos_bar, mass_bar, bx, bs, s_red[w], lane);
                else
                    vjp_round<T, K, true>(a, f, c, r0, cr, beg, end, chunk, nch, done, ctr, first, count, xyzm,
                                          src, perm, far, far_w, lsrc, pos_bar, mass_bar, bx, bs, s_red[w], lane);
            }
        }
        if (nch > 1 && chunk < nch - 1) pass_turn(done + a, chunk + 1);
    }
}

template <class T, int P>
int launch_vjp_tp(Plan &P_, const void *abar, const void *pbar, void *pos_bar, void *mass_bar, cudaStream_t s)
{
    const int n = (int)P_.n;
    k_vjp_sources<T><<<P_.num_sms * 4, 256, 0, s>>>(n, P_.idx[0], (const T *)abar, (const T *)pbar,
                                                     (vec4<T> *)P_.vjp_src);
    // the work counters of the forward evaluation ran to their ends: start them afresh (the source
    // moments take counter 3, M2L 1, L2L 2, the near field 0)
    cudaMemsetAsync(P_.ctr->work_ctr, 0, sizeof(P_.ctr->work_ctr), s);
    const unsigned seq = P_.next_flag_seq(s);
    k_vjp_up<T, P><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, P_.node_first, P_.node_count, P_.node_child0,
                                                  P_.node_nchild, (const vec4<T> *)P_.node_c,
                                                  (const vec4<T> *)P_.xyzm, (const vec4<T> *)P_.vjp_src, (T *)P_.Ms,
                                                  P_.ncp, P_.node_flag, seq);
    int launches = 2;
    launches += launch_m2l_plain(P_, P_.Ms, P_.Lsm, s);
    // L2L of the source locals: the forward kernel on the source buffers
    void *fwd_lm2l = P_.Lm2l, *fwd_l = P_.L;
    P_.Lm2l = P_.Lsm;
    P_.L = P_.Ls;
    launches += launch_l2l(P_, P_.depth, s);
    P_.Lm2l = fwd_lm2l;
    P_.L = fwd_l;
    k_vjp_far<T, P><<<P_.num_sms * 8, 256, 0, s>>>(P_.ctr, P_.node_first, P_.node_count, P_.node_nchild,
                                                   (const vec4<T> *)P_.node_c, (const vec4<T> *)P_.xyzm,
                                                   (const vec4<T> *)P_.vjp_src, P_.idx[0], (const T *)P_.L,
                                                   (const T *)P_.Ls, P_.ncp, (const T *)P_.vjp_acc,
                                                   (vec4<T> *)P_.far);
    // the near field takes the forward evaluation's work items afresh (work counter 0 was reset above
    // and neither M2L nor L2L uses it); its chunk flags start again from zero
    cudaMemsetAsync(P_.p2p_done, 0, (size_t)P_.cap_nodes * sizeof(int), s);
    k_vjp_near<T, VjpK<T>::value><<<P_.num_sms * 16, VJP_WARPS * 32, 0, s>>>(
        P_.ctr, P_.p2p_items, P_.p2p_done, P_.ctr, P_.node_first, P_.node_count, (const vec4<T> *)P_.xyzm,
        (const vec4<T> *)P_.vjp_src, P_.idx[0], (const vec4<T> *)P_.far, (vec4<T> *)P_.far, P_.p2p_off,
        P_.p2p_src, (T *)pos_bar, (T *)mass_bar);
    return launches + 2;
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
