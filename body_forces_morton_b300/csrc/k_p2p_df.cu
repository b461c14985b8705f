// P2P of fp64 plans in double-float arithmetic on the FP32 pipe.
//
// The near field of the direct-gravity eq. (JZ-FMM page, "From particle pairs
// to node pairs") for receiving leaf A and source leaf B, as in k_p2p, but every
// value is an unevaluated sum hi + lo of two fp32 numbers (about 48 significant
// bits). The FP64 rate of this GPU is a small fraction of its FP32 rate, so the
// ~180 fp32 operations of a double-float interaction cost several times less
// than the ~20 fp64 operations of a native one.
//
// Positions enter as offsets from their own leaf's centre, s = x - c_leaf
// (formed in fp64, then split), and the separation of a source j in B from a
// receiver i in A is (delta + s_j) - s_i with delta = c_B - c_A: every value is
// of the size of a leaf, so the separation keeps ~48 bits relative to the leaf
// size rather than to |x|. Sums run in a fixed order (reproducible).
#include "dfloat.cuh"
#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

// a staged source: position offset from the receiving leaf's centre and mass
struct SrcDF { df x, y, z, m; };

// The separation (delta + s_j) - s_i carries an absolute error of about 2^-46 E,
// E = |delta| + |s_j| + |s_i|. A pair closer than kExact E (or inside fp32's
// exponent floor, kTinyR2) is evaluated in fp64 from the sorted positions
// instead, with x_j - x_i formed directly as the direct sum forms it; every
// other pair keeps a relative separation error below ~2^-38 (6e-12).
constexpr float kExact = 0x1p-8f;
constexpr float kTinyR2 = 0x1p-84f;

// fp64 evaluation of one pair from the sorted positions (scaled units), as
// (m / r^2) (d / r) so that no intermediate leaves the fp32 range of the result.
__device__ __noinline__ void p2p_exact(const dbl4 *__restrict__ xyzm, int i, int j, int ex, int em, df (&acc)[4])
{
    const dbl4 pi = xyzm[i], pj = xyzm[j];
    const double x = ldexp(pj.x - pi.x, -ex), y = ldexp(pj.y - pi.y, -ex), z = ldexp(pj.z - pi.z, -ex);
    const double r2 = x * x + y * y + z * z;
    if (r2 == 0.0) return;  // zero separation: the particle itself (or an exact duplicate)
    const double ri = rsqrt(r2);
    const double mr = ldexp(pj.w, -em) * ri;
    const double g = mr * ri;
    acc[1] = df_add(acc[1], df_from(g * (x * ri)));
    acc[2] = df_add(acc[2], df_from(g * (y * ri)));
    acc[3] = df_add(acc[3], df_from(g * (z * ri)));
    acc[0] = df_sub(acc[0], df_from(mr));
}

struct ExactCtx {
    const dbl4 *xyzm;
    int ex, em;
};

__device__ __forceinline__ void p2p_df_one(const SrcDF &s, int j, const df &xi, const df &yi, const df &zi, int i,
                                           float thr2, const ExactCtx &cx, df (&acc)[4])
{
    const df dx = df_sub(s.x, xi), dy = df_sub(s.y, yi), dz = df_sub(s.z, zi);
    const df r2 = df_add(df_add(df_sqr(dx), df_sqr(dy)), df_sqr(dz));
    if (r2.h < thr2) {
        p2p_exact(cx.xyzm, i, j, cx.ex, cx.em, acc);
        return;
    }
    const df ri = df_rsqrt(r2);
    const df mr = df_mul(s.m, ri);
    const df mr3 = df_mul(mr, df_sqr(ri));
    acc[1] = df_add(acc[1], df_mul(mr3, dx));
    acc[2] = df_add(acc[2], df_mul(mr3, dy));
    acc[3] = df_add(acc[3], df_mul(mr3, dz));
    acc[0] = df_sub(acc[0], mr);
}

constexpr int DF_WARPS = 4;
constexpr int DF_CH = 128;  // staged source particles per warp

// Scaled offsets of every particle from its leaf's centre (units of df_units:
// scaled offsets and centre differences stay below 2 and masses at most 1, so
// fp32's exponent range holds every intermediate of a pair separated by more
// than 2^-42 of the box; acc = acc' 2^(em - 2 ex), phi = phi' 2^(em - ex)), split
// into double words: rel[i] = (sx.h, sy.h, sz.h, m.h) and rel[N + i] = (sx.l, sy.l, sz.l, m.l).
__global__ __launch_bounds__(256) void k_leaf_offsets(const DevCounters *__restrict__ nctr, int n, const int *__restrict__ first,
                                                      const int *__restrict__ count, const int *__restrict__ nchild,
                                                      const dbl4 *__restrict__ xyzm, const dbl4 *__restrict__ nc,
                                                      const dbl4 *__restrict__ nl, const double *__restrict__ M,
                                                      float4 *__restrict__ rel)
{
    const int n_nodes = phase2_nodes(nctr);
    if (n_nodes <= 0) return;
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    __shared__ int s_units[2];  // the unit exponents, found once per block
    if (threadIdx.x == 0) df_units(nl, M, s_units[0], s_units[1]);
    __syncthreads();
    const int ex = s_units[0], em = s_units[1];
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const dbl4 c = nc[a];
        for (int i = first[a] + lane; i < first[a] + count[a]; i += 32) {
            const dbl4 q = xyzm[i];
            const df x = df_from(scale2(q.x - c.x, -ex)), y = df_from(scale2(q.y - c.y, -ex));
            const df z = df_from(scale2(q.z - c.z, -ex)), m = df_from(scale2(q.w, -em));
            rel[i] = make_float4(x.h, y.h, z.h, m.h);
            rel[n + i] = make_float4(x.l, y.l, z.l, m.l);
        }
    }
}

__device__ __forceinline__ void put_src(float4 *buf, int k, const SrcDF &s)
{
    buf[2 * k] = make_float4(s.x.h, s.y.h, s.z.h, s.m.h);
    buf[2 * k + 1] = make_float4(s.x.l, s.y.l, s.z.l, s.m.l);
}

__device__ __forceinline__ SrcDF get_src(const float4 *buf, int k)
{
    const float4 h = buf[2 * k], l = buf[2 * k + 1];
    SrcDF s;
    s.x = {h.x, l.x};
    s.y = {h.y, l.y};
    s.z = {h.z, l.z};
    s.m = {h.w, l.w};
    return s;
}

// Stage particles [g0, g0 + CH) of the current group's source leaves, each as
// delta + s_j relative to the receiving leaf (lane i holds the group's i-th
// leaf: first particle lf, exclusive prefix ex, centre offset delta), with its
// sorted index for the exact branch.
__device__ __forceinline__ int stage_df(float4 *buf, int *sidx, const float4 *__restrict__ rel, int n, int lf, int ex,
                                        df dxl, df dyl, df dzl, int tot, int g0, int lane)
{
    const int n_here = min(DF_CH, tot - g0);
    for (int k0 = 0; k0 < n_here; k0 += 32) {
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
        df d[3] = {dxl, dyl, dzl};
#pragma unroll
        for (int c = 0; c < 3; ++c) {
            d[c].h = __shfl_sync(kFull, d[c].h, lo);
            d[c].l = __shfl_sync(kFull, d[c].l, lo);
        }
        if (k < n_here) {
            const int j = f + (g - e);
            const float4 h = rel[j], l = rel[n + j];
            SrcDF s;
            s.x = df_add(d[0], df_make(h.x, l.x));
            s.y = df_add(d[1], df_make(h.y, l.y));
            s.z = df_add(d[2], df_make(h.z, l.z));
            s.m = {h.w, l.w};
            put_src(buf, k, s);
            sidx[k] = j;
        }
    }
    return n_here;
}

template <int K>
__device__ __forceinline__ void span_df(const float4 *buf, const int *sidx, int n_here, int q, int S,
                                        const df (&rx)[K], const df (&ry)[K], const df (&rz)[K], const int (&ri)[K],
                                        float thr2, const ExactCtx &cx, df (&acc)[K][4])
{
    for (int j = q; j < n_here; j += S) {
        const SrcDF s = get_src(buf, j);
        const int js = sidx[j];
#pragma unroll
        for (int k = 0; k < K; ++k) p2p_df_one(s, js, rx[k], ry[k], rz[k], ri[k], thr2, cx, acc[k]);
    }
}

// |l| of a node (from the |l|^2 stored with its centre) in the scaled units
__device__ __forceinline__ float ext_scaled(const dbl4 &c, int ex) { return sqrtf((float)scale2(c.w, -2 * ex)); }

__device__ __forceinline__ float exact_thr2(float e)
{
    const float t = kExact * e;
    return fmaxf(t * t, kTinyR2);
}

template <int K, bool CHUNKED>
__device__ __forceinline__ void round_df(int a, int f, int c, int r0, int cr, int beg, int end, int chunk, int nch,
                                         int *done, DevCounters *ctr, int n, const ExactCtx &cx,
                                         const int *__restrict__ first,
                                         const int *__restrict__ count, const dbl4 *__restrict__ nc,
                                         const float4 *__restrict__ rel, const uint32_t *__restrict__ perm,
                                         dbl4 *far, const int *__restrict__ src,
                                         double *__restrict__ acc_out, double *__restrict__ pot_out, float4 *buf,
                                         int *sidx, double (*red)[4], int lane)
{
    const int R = (cr + K - 1) / K, S = 32 / R;
    const int rp = lane % R, q = lane / R;
    const int qq = q < S ? q : (1 << 30);
    df rx[K], ry[K], rz[K], acc[K][4];
    int ri[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int rr = rp + k * R;
        ri[k] = f + r0 + (rr < cr ? rr : 0);
        const float4 h = rel[ri[k]], l = rel[n + ri[k]];
        rx[k] = df_make(h.x, l.x);
        ry[k] = df_make(h.y, l.y);
        rz[k] = df_make(h.z, l.z);
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[k][v] = df_make(0.0f, 0.0f);
    }
    const dbl4 ca = nc[a];
    const float ext_a = ext_scaled(ca, cx.ex);
    // the leaf's own particles (delta = 0; zero separations go to the exact branch and are skipped there)
    const float thr_own = exact_thr2(2.0f * ext_a);
    for (int g0 = 0; (!CHUNKED || chunk == 0) && g0 < c; g0 += DF_CH) {
        const int n_here = min(DF_CH, c - g0);
        __syncwarp();
        for (int k = lane; k < n_here; k += 32) {
            const float4 h = rel[f + g0 + k], l = rel[n + f + g0 + k];
            SrcDF s;
            s.x = df_make(h.x, l.x);
            s.y = df_make(h.y, l.y);
            s.z = df_make(h.z, l.z);
            s.m = df_make(h.w, l.w);
            put_src(buf, k, s);
            sidx[k] = f + g0 + k;
        }
        __syncwarp();
        span_df<K>(buf, sidx, n_here, qq, S, rx, ry, rz, ri, thr_own, cx, acc);
    }
    for (int lb = beg; lb < end; lb += 32) {
        const int e = lb + lane;
        int lf = 0, cb = 0;
        float eb = 0.0f;  // |delta| + |l_B|: bound on |delta + s_j|
        df dxl = df_make(0.0f, 0.0f), dyl = dxl, dzl = dxl;
        if (e < end) {
            const int b = src[e];
            if (b != a) {
                lf = first[b];
                cb = count[b];
                const dbl4 cbc = nc[b];
                dxl = df_from(scale2(cbc.x - ca.x, -cx.ex));
                dyl = df_from(scale2(cbc.y - ca.y, -cx.ex));
                dzl = df_from(scale2(cbc.z - ca.z, -cx.ex));
                eb = sqrtf(dxl.h * dxl.h + dyl.h * dyl.h + dzl.h * dzl.h) + ext_scaled(cbc, cx.ex);
            }
        }
        const int incl = warp_incl_scan(cb);
        const int tot = __shfl_sync(kFull, incl, 31);
        const int xs = incl - cb;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) eb = fmaxf(eb, __shfl_xor_sync(kFull, eb, o));
        // 1.01: margin for the fp32 rounding of the bound itself
        const float thr = exact_thr2(1.01f * (eb + ext_a));
        for (int g0 = 0; g0 < tot; g0 += DF_CH) {
            __syncwarp();
            const int n_here = stage_df(buf, sidx, rel, n, lf, xs, dxl, dyl, dzl, tot, g0, lane);
            __syncwarp();
            span_df<K>(buf, sidx, n_here, qq, S, rx, ry, rz, ri, thr, cx, acc);
        }
    }
    const int eacc = cx.em - 2 * cx.ex, epot = cx.em - cx.ex;
    // a split receiver's chunks add up in chunk order: wait for the previous chunk
    if (CHUNKED && r0 == 0) wait_turn(done + a, chunk, ctr);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        __syncwarp();
#pragma unroll
        for (int v = 0; v < 4; ++v) red[lane][v] = (double)acc[k][v].h + (double)acc[k][v].l;
        __syncwarp();
        const int rr = rp + k * R;
        if (q == 0 && rr < cr) {
            double t[4] = {red[rp][0], red[rp][1], red[rp][2], red[rp][3]};
            for (int qs = 1; qs < S; ++qs)
#pragma unroll
                for (int v = 0; v < 4; ++v) t[v] += red[qs * R + rp][v];
            const int i = f + r0 + rr;
            // the far field, plus the partial sums of the earlier chunks (written by other warps)
            const dbl4 fa = CHUNKED ? ld_cg(far + i) : far[i];
            const double sx = fa.x + scale2(t[0], epot), sy = fa.y + scale2(t[1], eacc);
            const double sz = fa.z + scale2(t[2], eacc), sw = fa.w + scale2(t[3], eacc);
            if (CHUNKED && chunk < nch - 1) {
                far[i] = make4<double>(sx, sy, sz, sw);
            } else {
                const uint32_t o = perm[i];
                acc_out[3 * (size_t)o] = sy;
                acc_out[3 * (size_t)o + 1] = sz;
                acc_out[3 * (size_t)o + 2] = sw;
                if (pot_out) pot_out[o] = sx;
            }
        }
    }
}

// One work item: a receiving leaf, or one chunk of a split one (the chunk's
// share of the source list; the own leaf goes with chunk 0; chunks apply their
// sums in chunk order).
template <bool CHUNKED>
__device__ __forceinline__ void item_df(int a, int chunk, int nch, int *done, DevCounters *ctr, int n,
                                        const ExactCtx &cx, const int *__restrict__ first,
                                        const int *__restrict__ count, const dbl4 *__restrict__ nc,
                                        const float4 *__restrict__ rel, const uint32_t *__restrict__ perm, dbl4 *far,
                                        const int *__restrict__ off, const int *__restrict__ src,
                                        double *__restrict__ acc_out, double *__restrict__ pot_out, float4 *buf,
                                        int *sidx, double (*red)[4], int lane)
{
    const int f = first[a], c = count[a];
    int beg = off[a], end = off[a + 1];
    if (CHUNKED) {
        const int len = end - beg;
        end = beg + len * (chunk + 1) / nch;
        beg = beg + len * chunk / nch;
    }
    for (int r0 = 0; r0 < c; r0 += 64) {
        const int cr = min(64, c - r0);
        // K = 2 receivers per lane unless K = 1 keeps more lanes busy
        const int R1 = cr, R2 = (cr + 1) / 2;
        const int num1 = R1 <= 32 ? cr * (32 / R1) * 2 : -1;
        const int num2 = cr * (32 / R2);
        if (num1 > num2)
            round_df<1, CHUNKED>(a, f, c, r0, cr, beg, end, chunk, nch, done, ctr, n, cx, first, count, nc, rel,
                                 perm, far, src, acc_out, pot_out, buf, sidx, red, lane);
        else
            round_df<2, CHUNKED>(a, f, c, r0, cr, beg, end, chunk, nch, done, ctr, n, cx, first, count, nc, rel,
                                 perm, far, src, acc_out, pot_out, buf, sidx, red, lane);
    }
    if (CHUNKED && chunk < nch - 1) pass_turn(done + a, chunk + 1);
}

__global__ __launch_bounds__(DF_WARPS * 32, 4) void k_p2p_df(const DevCounters *__restrict__ cst,
                                                          const int2 *__restrict__ items, int *done,
                                                          DevCounters *ctr, int n,
                                                          const int *__restrict__ first, const int *__restrict__ count,
                                                          const dbl4 *__restrict__ xyzm, const dbl4 *__restrict__ nc,
                                                          const float4 *__restrict__ rel,
                                                          const uint32_t *__restrict__ perm, dbl4 *far,
                                                          const int *__restrict__ off,
                                                          const int *__restrict__ src, const dbl4 *__restrict__ nl,
                                                          const double *__restrict__ M, double *__restrict__ acc_out,
                                                          double *__restrict__ pot_out)
{
    __shared__ float4 s_src[DF_WARPS][2 * DF_CH];
    __shared__ int s_idx[DF_WARPS][DF_CH];
    __shared__ double s_red[DF_WARPS][32][4];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int n_work = 0;
    for (int b = 1; b < 64; ++b) n_work += cst->order_cnt[0][b];
    ExactCtx cx{xyzm, 0, 0};
    if (n_work > 0) df_units(nl, M, cx.ex, cx.em);
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[0], 1);
        t = __shfl_sync(kFull, t, 0);
        if (t >= n_work) break;
        const int2 item = items[t];
        const int a = item.x, nch = item.y >> 8;
        if (nch == 1)
            item_df<false>(a, 0, 1, done, ctr, n, cx, first, count, nc, rel, perm, far, off, src, acc_out, pot_out,
                           s_src[w], s_idx[w], s_red[w], lane);
        else
            item_df<true>(a, item.y & 255, nch, done, ctr, n, cx, first, count, nc, rel, perm, far, off, src, acc_out,
                          pot_out, s_src[w], s_idx[w], s_red[w], lane);
    }
}

// L2P of fp64 plans in double-float: every leaf's complete local expansion
// evaluated at its particles (Taylor eq.), into `far` (phi, a). In exact
// power-of-two units: lengths in the leaf level's cell bound h = 2^(ex - l),
// masses in 2^em (df_units), so u = (x - c) / h stays below 2 and the
// coefficients L~_k = L_k 2^(-em) h^|k| 2^(ex) are of one scale; then
// phi = 2^(em - ex) sum L~_k u^k / k!, a = -2^(em - ex) / h sum L~_(k+e) u^k / k!.
// The offsets come from the leaf-relative double words of k_leaf_offsets (box
// units, scaled exactly to u), so the FP64 pipe only converts the
// coefficients (once per leaf) and the four results.
template <int P>
__global__ __launch_bounds__(256) void k_l2p_df(const DevCounters *__restrict__ nctr, const int *__restrict__ first,
                                                const int *__restrict__ count, const int *__restrict__ nchild,
                                                const int *__restrict__ level, const float4 *__restrict__ rel, int n,
                                                const dbl4 *__restrict__ nl, const double *__restrict__ M,
                                                const double *__restrict__ L, int ncp, dbl4 *__restrict__ far)
{
    constexpr int NC = Exp<P>::NC;
    __shared__ df s_L[8][NC];
    const int n_nodes = phase2_nodes(nctr);
    if (n_nodes == 0) return;
    int ex, em;
    df_units(nl, M, ex, em);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a], lv = level[a];
        __syncwarp();
        for (int k = lane; k < NC; k += 32)
            s_L[w][k] = df_from(scale2(L[(size_t)a * ncp + k], ex - em + (ex - lv) * coef_degree(k)));
        __syncwarp();
        const float su = pow2f(lv);  // box units -> leaf units
        const int ephi = em - ex, eacc = em - ex - (ex - lv);
        for (int i = f + lane; i < f + c; i += 32) {
            const float4 h = rel[i], l = rel[n + i];
            const df ux = df_scale(df(h.x, l.x), su), uy = df_scale(df(h.y, l.y), su), uz = df_scale(df(h.z, l.z), su);
            df phi(0.0f, 0.0f), ax(0.0f, 0.0f), ay(0.0f, 0.0f), az(0.0f, 0.0f);
            Exp<P>::template l2p<df>(s_L[w], ux, uy, uz, phi, ax, ay, az);
            far[i] = make4<double>(scale2(df_to(phi), ephi), scale2(df_to(ax), eacc), scale2(df_to(ay), eacc),
                                   scale2(df_to(az), eacc));
        }
    }
}

template <int P>
int launch_l2p_df_p(Plan &P_, cudaStream_t s)
{
    // leaf-relative offsets first (they serve this kernel and the near field)
    k_leaf_offsets<<<P_.num_sms * 2, 256, 0, s>>>(P_.ctr, (int)P_.n, P_.node_first, P_.node_count, P_.node_nchild,
                                                  (const dbl4 *)P_.xyzm, (const dbl4 *)P_.node_c,
                                                  (const dbl4 *)P_.node_l, (const double *)P_.M, (float4 *)P_.rel);
    k_l2p_df<P><<<P_.num_sms * 8, 256, 0, s>>>(P_.ctr, P_.node_first, P_.node_count, P_.node_nchild, P_.node_level,
                                               (const float4 *)P_.rel, (int)P_.n, (const dbl4 *)P_.node_l,
                                               (const double *)P_.M, (const double *)P_.L, P_.ncp, (dbl4 *)P_.far);
    return 2;
}

}  // namespace

int launch_l2p_df(Plan &P, cudaStream_t s)
{
    switch (P.p) {
    case 0: return launch_l2p_df_p<0>(P, s);
    case 1: return launch_l2p_df_p<1>(P, s);
    case 2: return launch_l2p_df_p<2>(P, s);
    case 3: return launch_l2p_df_p<3>(P, s);
    case 4: return launch_l2p_df_p<4>(P, s);
    case 5: return launch_l2p_df_p<5>(P, s);
    default: return launch_l2p_df_p<6>(P, s);
    }
}

int launch_p2p_df(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    int launches = 1;
    if (P.p > kMaxPL2pDf) {  // the double-float L2P, which computes the offsets, did not run
        ++launches;
        k_leaf_offsets<<<P.num_sms * 8, 256, 0, s>>>(P.ctr, (int)P.n, P.node_first, P.node_count, P.node_nchild,
                                                    (const dbl4 *)P.xyzm, (const dbl4 *)P.node_c,
                                                    (const dbl4 *)P.node_l, (const double *)P.M, (float4 *)P.rel);
    }
    k_p2p_df<<<P.num_sms * 16, DF_WARPS * 32, 0, s>>>(P.ctr, P.p2p_items, P.p2p_done, P.ctr, (int)P.n, P.node_first,
                                                      P.node_count, (const dbl4 *)P.xyzm, (const dbl4 *)P.node_c,
                                                      (const float4 *)P.rel, P.idx[0], (dbl4 *)P.far, P.p2p_off,
                                                      P.p2p_src, (const dbl4 *)P.node_l, (const double *)P.M,
                                                      (double *)acc, (double *)pot);
    return launches;
}

}  // namespace bfm
