// Downward pass: L2L from the root down (one launch, ordered by level), then
// L2P + P2P at the leaves.
//
// JZ-FMM page, "Combining near and far interactions", stage 3: translate each
// parent's local Taylor expansion to its children, evaluate the expansions at
// the particle positions (Taylor eq.: Phi(c + dx) = sum_k L_k dx^k / k!,
// a = -grad Phi) and calculate the remaining nearby interactions directly
// (direct gravity eq.: Phi_i += -G m_j / r, a_i += G m_j (x_j - x_i) / r^3,
// skipping zero separations, i.e. the particle itself).
//
// Leaves: a small L2P kernel evaluates the local expansions at the particles;
// the P2P kernel (one warp per receiving leaf) stages the particles of the
// source leaves through shared memory (32 list entries and up to a chunk of
// particles at a time), reads them back as broadcasts, keeps all lanes busy for
// small leaves by splitting the sources, adds the far field and writes straight
// to the caller's particle order.
#include <type_traits>

#include "expansions_gen.cuh"
#include "plan.h"

#include <algorithm>

namespace bfm {

namespace {

// One source particle s acting on a receiver at (x, y, z). The self leaf may
// hold the receiver itself (zero separation), which MASKED skips; between two
// different leaves the separation is never zero (equal positions share a key
// and so a leaf), so the main loop runs unmasked.
template <class T, bool MASKED>
__device__ __forceinline__ void p2p_one(const vec4<T> &s, T x, T y, T z, T &phi, T &ax, T &ay, T &az)
{
    const T dx = s.x - x, dy = s.y - y, dz = s.z - z;
    const T r2 = dx * dx + dy * dy + dz * dz;
    T rinv = rsqrt_t(r2);
    if (MASKED) rinv = r2 > T(0) ? rinv : T(0);
    const T mr = s.w * rinv;
    const T mr3 = mr * rinv * rinv;
    ax += mr3 * dx;
    ay += mr3 * dy;
    az += mr3 * dz;
    phi -= mr;
}

// L2P: the complete local expansion of every leaf at its particles, into `far`
// (sorted order, (phi, ax, ay, az)); the P2P kernel adds the near field.
template <class T, int P>
__global__ __launch_bounds__(256) void k_l2p(const DevCounters *__restrict__ nctr, const int *__restrict__ first, const int *__restrict__ count,
                                             const int *__restrict__ nchild, const vec4<T> *__restrict__ xyzm,
                                             const vec4<T> *__restrict__ nc, const T *__restrict__ L, int ncp,
                                             vec4<T> *__restrict__ far)
{
    const int n_nodes = phase2_nodes(nctr);
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a];
        const vec4<T> ca = nc[a];
        const T *La = L + (size_t)a * ncp;
        for (int i = f + lane; i < f + c; i += 32) {
            const vec4<T> q = xyzm[i];
            T phi = T(0), ax = T(0), ay = T(0), az = T(0);
            Exp<P>::template l2p<T>(La, q.x - ca.x, q.y - ca.y, q.z - ca.z, phi, ax, ay, az);
            far[i] = make4<T>(phi, ax, ay, az);
        }
    }
}

constexpr int LF_WARPS = 4;                            // warps per block of the P2P kernel
template <class T> struct LeafChunk { static constexpr int value = 256; };   // staged source particles per warp
template <> struct LeafChunk<double> { static constexpr int value = 128; };

// Stage particles [g0, g0 + CH) of the concatenation of the current group's
// source leaves into shared memory. Lane i holds the group's i-th leaf: first
// particle fb and exclusive prefix ex of the counts (ascending over the lanes).
template <class T, int CH>
__device__ __forceinline__ int stage_sources(vec4<T> *buf, const vec4<T> *__restrict__ xyzm, int fb, int ex,
                                             int tot, int g0, int lane)
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
        if (k < n_here) buf[k] = xyzm[f + (g - e)];
    }
    return n_here;
}

// Interactions of the staged sources buf[q], buf[q+S], ... with K receivers.
template <class T, bool MASKED, int K>
__device__ __forceinline__ void p2p_span(const vec4<T> *buf, int n_here, int q, int S, const vec4<T> (&p)[K],
                                         T (&acc)[K][4])
{
    int j = q;
    for (; j + S < n_here; j += 2 * S) {
        const vec4<T> s0 = buf[j], s1 = buf[j + S];
#pragma unroll
        for (int k = 0; k < K; ++k) p2p_one<T, MASKED>(s0, p[k].x, p[k].y, p[k].z, acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
#pragma unroll
        for (int k = 0; k < K; ++k) p2p_one<T, MASKED>(s1, p[k].x, p[k].y, p[k].z, acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
    }
    if (j < n_here) {
        const vec4<T> s0 = buf[j];
#pragma unroll
        for (int k = 0; k < K; ++k) p2p_one<T, MASKED>(s0, p[k].x, p[k].y, p[k].z, acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
    }
}

// ---- fp32: two sources per instruction with the packed f32x2 arithmetic of
// sm_100-family GPUs (one instruction issues the operation for both halves;
// the compiler's float2 builtins let it keep the halves in register pairs).
// Staged sources are stored pair-interleaved, (x_j, x_j+1, y_j, y_j+1, z_j,
// z_j+1, m_j, m_j+1) per pair, so two 16-byte shared loads give four packed
// operands; an odd tail is padded with a massless particle far away.
__device__ __forceinline__ void put_pair_layout(float *fb, int k, float x, float y, float z, float m)
{
    const int base = (k >> 1) * 8 + (k & 1);
    fb[base] = x;
    fb[base + 2] = y;
    fb[base + 4] = z;
    fb[base + 6] = m;
}

// Reciprocal square root with subnormal inputs flushed to zero: the bare
// special-function instruction. r^2 of two distinct fp32 particles is subnormal
// only for separations below 1.1e-19, which fp32 inputs of this code never
// reach (such a pair would get an infinite force).
__device__ __forceinline__ float rsqrt_ftz(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Two sources (packed SX, SY, SZ, SM) acting on one receiver given as the
// negated broadcast position (NX, NY, NZ); A = (sum m/r, ax, ay, az), each the
// even-source and odd-source halves (the potential is minus the first sum).
__device__ __forceinline__ void p2p_two(float2 SX, float2 SY, float2 SZ, float2 SM, float2 NX, float2 NY, float2 NZ,
                                        float2 (&A)[4])
{
    const float2 dx = __fadd2_rn(SX, NX), dy = __fadd2_rn(SY, NY), dz = __fadd2_rn(SZ, NZ);
    float2 r2 = __fmul2_rn(dx, dx);
    r2 = __ffma2_rn(dy, dy, r2);
    r2 = __ffma2_rn(dz, dz, r2);
    const float2 ri = make_float2(rsqrt_ftz(r2.x), rsqrt_ftz(r2.y));
    const float2 mr = __fmul2_rn(SM, ri);
    const float2 mr3 = __fmul2_rn(mr, __fmul2_rn(ri, ri));
    A[1] = __ffma2_rn(mr3, dx, A[1]);
    A[2] = __ffma2_rn(mr3, dy, A[2]);
    A[3] = __ffma2_rn(mr3, dz, A[3]);
    A[0] = __fadd2_rn(A[0], mr);
}

template <int CH>
__device__ __forceinline__ int stage_sources_pairs(float *fb, const float4 *__restrict__ xyzm, int lf, int ex,
                                                   int tot, int g0, int lane)
{
    const int n_here = min(CH, tot - g0);
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
        if (k < n_here) {
            const float *v = reinterpret_cast<const float *>(xyzm + f + (g - e));
            float *d = fb + (k >> 1) * 8 + (k & 1);  // the pair-interleaved slots of put_pair_layout
            cp_async4(d, v);
            cp_async4(d + 2, v + 1);
            cp_async4(d + 4, v + 2);
            cp_async4(d + 6, v + 3);
        }
    }
    if ((n_here & 1) && lane == 0) put_pair_layout(fb, n_here, 1e18f, 1e18f, 1e18f, 0.0f);
    cp_async_wait_all();
    return (n_here + 1) >> 1;
}

template <int K>
__device__ __forceinline__ void p2p_span_pairs(const float *fb, int npairs, int q, int S, const float2 (&X)[K],
                                               const float2 (&Y)[K], const float2 (&Z)[K], float2 (&A)[K][4])
{
    const float4 *pb = reinterpret_cast<const float4 *>(fb);
    int j = q;
    for (; j + S < npairs; j += 2 * S) {
        const float4 a0 = pb[2 * j], b0 = pb[2 * j + 1];
        const float4 a1 = pb[2 * (j + S)], b1 = pb[2 * (j + S) + 1];
#pragma unroll
        for (int k = 0; k < K; ++k)
            p2p_two(make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(b0.x, b0.y),
                    make_float2(b0.z, b0.w), X[k], Y[k], Z[k], A[k]);
#pragma unroll
        for (int k = 0; k < K; ++k)
            p2p_two(make_float2(a1.x, a1.y), make_float2(a1.z, a1.w), make_float2(b1.x, b1.y),
                    make_float2(b1.z, b1.w), X[k], Y[k], Z[k], A[k]);
    }
    if (j < npairs) {
        const float4 a0 = pb[2 * j], b0 = pb[2 * j + 1];
#pragma unroll
        for (int k = 0; k < K; ++k)
            p2p_two(make_float2(a0.x, a0.y), make_float2(a0.z, a0.w), make_float2(b0.x, b0.y),
                    make_float2(b0.z, b0.w), X[k], Y[k], Z[k], A[k]);
    }
}

// One round of up to 32 K receivers [r0, r0 + cr) of leaf a. Lane = q R + rp
// (rp < R = ceil(cr / K), q < S = 32 / R) holds receivers rp + k R, k < K, and
// walks the staged sources from offset q with stride S. Lanes at or beyond
// R S only stage. The S partial sums of a receiver are added in order of q
// through shared memory, so the result is reproducible.
template <class T, int K, bool CHUNKED>
__device__ __forceinline__ void p2p_round(int a, int f, int c, int r0, int cr, int beg, int end, int chunk, int nch,
                                          int *done, DevCounters *ctr,
                                          const int *__restrict__ first, const int *__restrict__ count,
                                          const vec4<T> *__restrict__ xyzm, const uint32_t *__restrict__ perm,
                                          const vec4<T> *far, vec4<T> *far_w,
                                          const int *__restrict__ src,
                                          T *__restrict__ acc_out, T *__restrict__ pot_out, vec4<T> *buf,
                                          T (*red)[4], int lane)
{
    constexpr int CH = LeafChunk<T>::value;
    const int R = (cr + K - 1) / K, S = 32 / R;
    const int rp = lane % R, q = lane / R;
    const bool worker = q < S;
    vec4<T> p[K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int rr = rp + k * R;
        p[k] = xyzm[f + r0 + (rr < cr ? rr : 0)];
    }
    T acc[K][4];
#pragma unroll
    for (int k = 0; k < K; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = T(0);
    const int qq = worker ? q : (1 << 30);  // idle lanes start past every chunk
    // source leaves of the list, 32 entries at a time: lane i holds entry lb + i (first particle, count;
    // the receiving leaf itself counts as empty). The next group's entries load while this one computes.
    auto fetch = [&](int lb, int &fb, int &cb) {
        const int e = lb + lane;
        fb = 0;
        cb = 0;
        if (e < end) {
            const int b = src[e];
            if (b != a) {
                fb = first[b];
                cb = count[b];
            }
        }
    };
    int fb_next = 0, cb_next = 0;
    if (beg < end) fetch(beg, fb_next, cb_next);
    // the leaf's own particles (zero separations possible; the first chunk of a split receiver)
    for (int g0 = 0; (!CHUNKED || chunk == 0) && g0 < c; g0 += CH) {
        const int n_here = min(CH, c - g0);
        __syncwarp();
        for (int k = lane; k < n_here; k += 32)
#pragma unroll
            for (int h = 0; h < (int)sizeof(vec4<T>); h += 16)
                cp_async16(reinterpret_cast<char *>(buf + k) + h, reinterpret_cast<const char *>(xyzm + f + g0 + k) + h);
        cp_async_wait_all();
        __syncwarp();
        p2p_span<T, true, K>(buf, n_here, qq, S, p, acc);
    }
    // every other source leaf
    if constexpr (std::is_same<T, float>::value) {
        // packed accumulators start from the own-leaf sums (A[0] collects +m/r, the potential is its negative)
        float2 X[K], Y[K], Z[K], A[K][4];
#pragma unroll
        for (int k = 0; k < K; ++k) {
            X[k] = make_float2(-p[k].x, -p[k].x);
            Y[k] = make_float2(-p[k].y, -p[k].y);
            Z[k] = make_float2(-p[k].z, -p[k].z);
            A[k][0] = make_float2(-acc[k][0], 0.0f);
#pragma unroll
            for (int v = 1; v < 4; ++v) A[k][v] = make_float2(acc[k][v], 0.0f);
        }
        float *fbuf = reinterpret_cast<float *>(buf);
        for (int lb = beg; lb < end; lb += 32) {
            const int fb = fb_next, cb = cb_next;
            if (lb + 32 < end) fetch(lb + 32, fb_next, cb_next);
            const int incl = warp_incl_scan(cb);
            const int tot = __shfl_sync(kFull, incl, 31);
            const int ex = incl - cb;
            for (int g0 = 0; g0 < tot; g0 += CH) {
                __syncwarp();
                const int npairs = stage_sources_pairs<CH>(fbuf, xyzm, fb, ex, tot, g0, lane);
                __syncwarp();
                p2p_span_pairs<K>(fbuf, npairs, qq, S, X, Y, Z, A);
            }
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
            acc[k][0] = -(A[k][0].x + A[k][0].y);
#pragma unroll
            for (int v = 1; v < 4; ++v) acc[k][v] = A[k][v].x + A[k][v].y;
        }
    } else {
        for (int lb = beg; lb < end; lb += 32) {
            const int fb = fb_next, cb = cb_next;
            if (lb + 32 < end) fetch(lb + 32, fb_next, cb_next);
            const int incl = warp_incl_scan(cb);
            const int tot = __shfl_sync(kFull, incl, 31);
            const int ex = incl - cb;
            for (int g0 = 0; g0 < tot; g0 += CH) {
                __syncwarp();
                const int n_here = stage_sources<T, CH>(buf, xyzm, fb, ex, tot, g0, lane);
                __syncwarp();
                p2p_span<T, false, K>(buf, n_here, qq, S, p, acc);
            }
        }
    }
    // a split receiver's chunks add up in chunk order: wait for the previous chunk
    if (CHUNKED && r0 == 0) wait_turn(done + a, chunk, ctr);
    // sum the S strides of each receiver in order of q
#pragma unroll
    for (int k = 0; k < K; ++k) {
        __syncwarp();
        red[lane][0] = acc[k][0];
        red[lane][1] = acc[k][1];
        red[lane][2] = acc[k][2];
        red[lane][3] = acc[k][3];
        __syncwarp();
        const int rr = rp + k * R;
        if (q == 0 && rr < cr) {
            T t[4] = {red[rp][0], red[rp][1], red[rp][2], red[rp][3]};
            for (int qs = 1; qs < S; ++qs)
#pragma unroll
                for (int v = 0; v < 4; ++v) t[v] += red[qs * R + rp][v];
            const int i = f + r0 + rr;
            // the far field, plus the partial sums of the earlier chunks (written by other warps through
            // far_w, which aliases far: hence no __restrict__ on either, and a coherent L2 load here, never
            // the non-coherent read-only path)
            const vec4<T> fa = CHUNKED ? ld_cg(far + i) : far[i];
            if (CHUNKED && chunk < nch - 1) {
                far_w[i] = make4<T>(fa.x + t[0], fa.y + t[1], fa.z + t[2], fa.w + t[3]);
            } else {
                const uint32_t o = perm[i];
                acc_out[3 * (size_t)o] = fa.y + t[1];
                acc_out[3 * (size_t)o + 1] = fa.z + t[2];
                acc_out[3 * (size_t)o + 2] = fa.w + t[3];
                if (pot_out) pot_out[o] = fa.x + t[0];
            }
        }
    }
}

// One work item: a receiving leaf, or one chunk of a split one (the chunk's
// share of the source list; the own leaf goes with chunk 0; chunks apply their
// sums in chunk order).
template <class T, bool CHUNKED>
__device__ __forceinline__ void p2p_item(int a, int chunk, int nch, int *done, DevCounters *ctr,
                                         const int *__restrict__ first, const int *__restrict__ count,
                                         const vec4<T> *__restrict__ xyzm, const uint32_t *__restrict__ perm,
                                         const vec4<T> *far, vec4<T> *far_w,
                                         const int *__restrict__ off, const int *__restrict__ src,
                                         T *__restrict__ acc_out, T *__restrict__ pot_out, vec4<T> *buf,
                                         T (*red)[4], int lane)
{
    const int f = first[a], c = count[a];
    int beg = off[a], end = off[a + 1];
    if (CHUNKED) {
        const int len = end - beg;
        end = beg + len * (chunk + 1) / nch;
        beg = beg + len * chunk / nch;
    }
    for (int r0 = 0; r0 < c; r0 += 128) {
        const int cr = min(128, c - r0);
        // four receivers per lane (R = ceil(cr / 4) lanes, the sources split S = 32 / R ways), or three
        // where that leaves fewer lane slots idle (17 particles: 6 lanes x 3 = 18 slots over 5 source
        // groups, against 5 x 4 = 20): measured faster than four alone. Two receivers per lane (tried as
        // 2 or 4) was slower: each staged source then feeds too little arithmetic.
        const int R4 = (cr + 3) / 4, R3 = (cr + 2) / 3;
        const float e4 = (float)cr / (4 * R4) * (float)(R4 * (32 / R4)) / 32.0f;
        const float e3 = R3 <= 32 ? (float)cr / (3 * R3) * (float)(R3 * (32 / R3)) / 32.0f : 0.0f;
        if (e3 > e4 * 1.02f)
            p2p_round<T, 3, CHUNKED>(a, f, c, r0, cr, beg, end, chunk, nch, done, ctr, first, count, xyzm, perm, far,
                                     far_w, src, acc_out, pot_out, buf, red, lane);
        else
            p2p_round<T, 4, CHUNKED>(a, f, c, r0, cr, beg, end, chunk, nch, done, ctr, first, count, xyzm, perm, far,
                                     far_w, src, acc_out, pot_out, buf, red, lane);
    }
    if (CHUNKED && chunk < nch - 1) pass_turn(done + a, chunk + 1);
}

// P2P for one receiving leaf per warp (leaves taken from a shared counter in
// decreasing order of work), plus the far field from `far`, scattered to the
// caller's order. Each lane takes up to four receivers of the leaf; the
// leaf's own particles are a separate masked pass, the rest runs unmasked.
template <class T>
__global__ __launch_bounds__(LF_WARPS * 32) void k_p2p(const DevCounters *__restrict__ cst,
                                                       const int2 *__restrict__ items, int *done,
                                                       DevCounters *ctr, const int *__restrict__ first,
                                                       const int *__restrict__ count,
                                                       const int *__restrict__ nchild,
                                                       const vec4<T> *__restrict__ xyzm,
                                                       const uint32_t *__restrict__ perm,
                                                       const vec4<T> *far, vec4<T> *far_w,
                                                       const int *__restrict__ off,
                                                       const int *__restrict__ src, T *__restrict__ acc_out,
                                                       T *__restrict__ pot_out)
{
    constexpr int CH = LeafChunk<T>::value;
    __shared__ vec4<T> s_src[LF_WARPS][CH];
    __shared__ T s_red[LF_WARPS][32][4];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int n_work = 0;
    for (int b = 1; b < 64; ++b) n_work += cst->order_cnt[0][b];
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[0], 1);
        t = __shfl_sync(kFull, t, 0);
        if (t >= n_work) break;
        const int2 item = items[t];
        const int a = item.x, nch = item.y >> 8;
        if (nch == 1)
            p2p_item<T, false>(a, 0, 1, done, ctr, first, count, xyzm, perm, far, far_w, off, src, acc_out, pot_out,
                               s_src[w], s_red[w], lane);
        else
            p2p_item<T, true>(a, item.y & 255, nch, done, ctr, first, count, xyzm, perm, far, far_w, off, src,
                              acc_out, pot_out, s_src[w], s_red[w], lane);
    }
}

// A node's row of NC coefficients moved in 16-byte pieces (rows are padded to
// a multiple of 4 elements, so every piece lies inside the row): loads plain
// or through L2 (CG, for rows other blocks of the launch wrote), stores with
// the padding zeroed.
template <class T, int NC, bool CG>
__device__ __forceinline__ void row_load16(const T *row, T (&r)[NC])
{
    if constexpr (sizeof(T) == 4) {
        const float4 *v = reinterpret_cast<const float4 *>(row);
#pragma unroll
        for (int q = 0; q < (NC + 3) / 4; ++q) {
            const float4 x = CG ? __ldcg(v + q) : v[q];
            const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (4 * q + h < NC) r[4 * q + h] = e[h];
        }
    } else {
        const double2 *v = reinterpret_cast<const double2 *>(row);
#pragma unroll
        for (int q = 0; q < (NC + 1) / 2; ++q) {
            const double2 x = CG ? __ldcg(v + q) : v[q];
            r[2 * q] = x.x;
            if (2 * q + 1 < NC) r[2 * q + 1] = x.y;
        }
    }
}

template <class T, int NC>
__device__ __forceinline__ void row_store16(T *row, const T (&r)[NC])
{
    if constexpr (sizeof(T) == 4) {
        float4 *v = reinterpret_cast<float4 *>(row);
#pragma unroll
        for (int q = 0; q < (NC + 3) / 4; ++q) {
            float e[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) e[h] = 4 * q + h < NC ? r[4 * q + h] : 0.0f;
            v[q] = make_float4(e[0], e[1], e[2], e[3]);
        }
    } else {
        double2 *v = reinterpret_cast<double2 *>(row);
#pragma unroll
        for (int q = 0; q < (NC + 1) / 2; ++q) v[q] = make_double2(r[2 * q], 2 * q + 1 < NC ? r[2 * q + 1] : 0.0);
    }
}

// L2L in one launch, without grid barriers: warps take chunks of up to 32
// nodes of one level from a shared counter, in level order (root first). A
// node's thread waits, bounded, until its parent's flag holds this pass's
// number (`want`, equal to `seq` unless a test injects an expired wait), which
// the parent's thread stores with release
// semantics after writing the parent's complete local; then it reads that
// local from L2 and adds its translation to its own M2L local. A chunk never
// spans two levels, so no lane waits for a lane of its own warp; every parent
// lies in an earlier chunk, taken by a warp already running, so the earliest
// unfinished chunk can always finish. Levels beyond the tree's depth cost
// nothing and there is no barrier per level.
template <class T, int P>
__global__ __launch_bounds__(256) void k_l2l_flags(DevCounters *ctr, const int *__restrict__ parent,
                                                   const vec4<T> *__restrict__ nc, const T *__restrict__ Lm2l,
                                                   T *L, int ncp, unsigned *flag, unsigned seq, unsigned want)
{
    constexpr int NC = Exp<P>::NC;
    __shared__ int s_off[kMaxLevel + 2];
    const int n = phase2_nodes(ctr);
    if (n == 0) return;
    const int depth = ctr->depth;
    for (int l = threadIdx.x; l <= depth + 1; l += blockDim.x) s_off[l] = min(ctr->level_off[l], n);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    for (;;) {
        int t = 0;
        if (lane == 0) t = atomicAdd(&ctr->work_ctr[2], 1);
        t = __shfl_sync(kFull, t, 0);
        int level = -1, lo = 0, hi = 0;
        for (int l = 0; l <= depth; ++l) {  // chunk t -> (level, node range)
            const int nch = (s_off[l + 1] - s_off[l] + 31) >> 5;
            if (t < nch) {
                level = l;
                lo = s_off[l] + 32 * t;
                hi = min(s_off[l + 1], lo + 32);
                break;
            }
            t -= nch;
        }
        if (level < 0) break;
        const int a = lo + lane;
        if (a >= hi) continue;
        T out[NC];
        row_load16<T, NC, false>(Lm2l + (size_t)a * ncp, out);
        if (level > 0) {
            const int par = parent[a];
            cuda::atomic_ref<unsigned, cuda::thread_scope_device> f(flag[par]);
            unsigned spins = 0;
            while (f.load(cuda::memory_order_acquire) != want) {
                if (++spins > kSpinLimit) {
                    set_error(ctr, ERR_SPIN);
                    break;
                }
                __nanosleep(32);
            }
            T lp[NC];
            row_load16<T, NC, true>(L + (size_t)par * ncp, lp);
            const vec4<T> c = nc[a], cp = nc[par];
            Exp<P>::template l2l<T>(lp, c.x - cp.x, c.y - cp.y, c.z - cp.z, out);
        }
        row_store16<T, NC>(L + (size_t)a * ncp, out);
        cuda::atomic_ref<unsigned, cuda::thread_scope_device>(flag[a]).store(seq, cuda::memory_order_release);
    }
}

// fp32 plans, p <= 4: every node's complete local at once, its own M2L local
// plus each ancestor's M2L local translated straight to the node's centre
// (nearest ancestor first). A degree-p local shifts exactly, so this is the
// level-by-level translation through the intermediate centres up to rounding,
// and no node waits for another: a thread per node walks its parent chain.
template <class T, int P>
__global__ __launch_bounds__(256) void k_l2l_direct(const DevCounters *__restrict__ ctr,
                                                    const int *__restrict__ parent, const vec4<T> *__restrict__ nc,
                                                    const T *__restrict__ Lm2l, T *__restrict__ L, int ncp,
                                                    const int *__restrict__ nchild, const int *__restrict__ first,
                                                    const int *__restrict__ count, int *__restrict__ leaf_of)
{
    constexpr int NC = Exp<P>::NC;
    static_assert(sizeof(T) == 4, "rows move as float4: fp32 plans only");
    constexpr int NV = (NC + 3) / 4;  // 16-byte pieces of a row (rows are padded to a multiple of 4)
    // a row into registers in 16-byte loads (one thread per node touches its own rows, so scalar loads
    // would each be a separate request)
    auto load_row = [](const T *row, T (&r)[NC]) {
        const float4 *v = reinterpret_cast<const float4 *>(row);
#pragma unroll
        for (int q = 0; q < NV; ++q) {
            const float4 x = v[q];
            const float e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                if (4 * q + h < NC) r[4 * q + h] = e[h];
        }
    };
    const int n = phase2_nodes(ctr);
    for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < n; a += gridDim.x * blockDim.x) {
        T out[NC];
        load_row(Lm2l + (size_t)a * ncp, out);
        const vec4<T> c = nc[a];
        int b = parent[a];
        for (int up = 0; b >= 0 && up <= kMaxLevel; ++up) {
            T lb[NC];
            load_row(Lm2l + (size_t)b * ncp, lb);
            const vec4<T> cb = nc[b];
            Exp<P>::template l2l<T>(lb, c.x - cb.x, c.y - cb.y, c.z - cb.z, out);
            b = parent[b];
        }
        float4 *dst = reinterpret_cast<float4 *>(L + (size_t)a * ncp);
#pragma unroll
        for (int q = 0; q < NV; ++q) {
            float e[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) e[h] = 4 * q + h < NC ? out[4 * q + h] : 0.0f;
            dst[q] = make_float4(e[0], e[1], e[2], e[3]);
        }
        if (nchild[a] == 0) {  // a leaf: its particles' leaf, for the L2P by particle
            const int f = first[a], c = count[a];
            for (int i = f; i < f + c; ++i) leaf_of[i] = a;
        }
    }
}

// L2P by particle, after k_l2l_direct: thread i evaluates its leaf's complete
// local (the same arithmetic as k_l2p, so the same bits) at particle i.
template <class T, int P>
__global__ __launch_bounds__(256) void k_l2p_part(const DevCounters *__restrict__ nctr, int n,
                                                  const int *__restrict__ leaf_of, const vec4<T> *__restrict__ xyzm,
                                                  const vec4<T> *__restrict__ nc, const T *__restrict__ L, int ncp,
                                                  vec4<T> *__restrict__ far, DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    if (n_nodes == 0) return;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int a = leaf_of[i];
        if (a < 0 || a >= n_nodes) {
            set_error(ctr, ERR_BOUNDS);
            continue;
        }
        const vec4<T> ca = nc[a], q = xyzm[i];
        T phi = T(0), ax = T(0), ay = T(0), az = T(0);
        T la[Exp<P>::NC];
        row_load16<T, Exp<P>::NC, false>(L + (size_t)a * ncp, la);  // the leaf's local in 16-byte pieces
        Exp<P>::template l2p<T>(la, q.x - ca.x, q.y - ca.y, q.z - ca.z, phi, ax, ay, az);
        far[i] = make4<T>(phi, ax, ay, az);
    }
}

template <class T, int P>
int launch_l2l_tp(Plan &P_, int depth, cudaStream_t s)
{
    (void)depth;  // read on the device
    if constexpr (sizeof(T) == 4 && P <= 4) {
        // (under the injected spin fault the level-ordered kernel below runs, whose waits it exercises)
        if (!P_.fault_spin) {
            k_l2l_direct<T, P><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, P_.node_parent, (const vec4<T> *)P_.node_c,
                                                              (const T *)P_.Lm2l, (T *)P_.L, P_.ncp, P_.node_nchild,
                                                              P_.node_first, P_.node_count, P_.leaf_of);
            return 1;
        }
    }
    const unsigned seq = P_.next_flag_seq(s);
    // a parent is complete when its flag holds seq; the injected fault waits for a value no pass stores
    // (pass numbers stay below 2^31)
    const unsigned want = P_.fault_spin ? (seq | 0x80000000u) : seq;
    k_l2l_flags<T, P><<<P_.num_sms * 4, 256, 0, s>>>(P_.ctr, P_.node_parent, (const vec4<T> *)P_.node_c,
                                                     (const T *)P_.Lm2l, (T *)P_.L, P_.ncp, P_.node_flag, seq,
                                                     want);
    return 1;
}

template <class T, int P>
int launch_l2p_tp(Plan &P_, cudaStream_t s)
{
    if constexpr (sizeof(T) == 4 && P <= 4) {
        if (!P_.fault_spin) {  // the direct L2L ran and recorded each particle's leaf
            k_l2p_part<T, P><<<P_.num_sms * 8, 256, 0, s>>>(P_.ctr, (int)P_.n, P_.leaf_of, (const vec4<T> *)P_.xyzm,
                                                            (const vec4<T> *)P_.node_c, (const T *)P_.L, P_.ncp,
                                                            (vec4<T> *)P_.far, P_.ctr);
            return 1;
        }
    }
    k_l2p<T, P><<<P_.num_sms * 8, 256, 0, s>>>(P_.ctr, P_.node_first, P_.node_count, P_.node_nchild,
                                               (const vec4<T> *)P_.xyzm, (const vec4<T> *)P_.node_c,
                                               (const T *)P_.L, P_.ncp, (vec4<T> *)P_.far);
    return 1;
}

#define BFM_DISPATCH_P(fn, T, ...)                        \
    switch (P.p) {                                        \
    case 0: return fn<T, 0>(P, __VA_ARGS__);              \
    case 1: return fn<T, 1>(P, __VA_ARGS__);              \
    case 2: return fn<T, 2>(P, __VA_ARGS__);              \
    case 3: return fn<T, 3>(P, __VA_ARGS__);              \
    case 4: return fn<T, 4>(P, __VA_ARGS__);              \
    case 5: return fn<T, 5>(P, __VA_ARGS__);              \
    case 6: return fn<T, 6>(P, __VA_ARGS__);              \
    case 7: return fn<T, 7>(P, __VA_ARGS__);              \
    default: return fn<T, 8>(P, __VA_ARGS__);             \
    }

template <class T> int launch_l2l_t(Plan &P, int depth, cudaStream_t s) { BFM_DISPATCH_P(launch_l2l_tp, T, depth, s) }
template <class T> int launch_l2p_t(Plan &P, cudaStream_t s) { BFM_DISPATCH_P(launch_l2p_tp, T, s) }

}  // namespace

int launch_l2l(Plan &P, int depth, cudaStream_t s)
{
    return P.dtype == 0 ? launch_l2l_t<float>(P, depth, s) : launch_l2l_t<double>(P, depth, s);
}

int launch_l2p(Plan &P, cudaStream_t s)
{
    if (P.dtype == 0) return launch_l2p_t<float>(P, s);
    return P.p <= kMaxPL2pDf && !P.f64_ieee ? launch_l2p_df(P, s) : launch_l2p_t<double>(P, s);
}

// fp32 plans: k_p2p<float>; fp64 plans: the double-float near field (k_p2p_df.cu), or k_p2p<double> in
// IEEE fp64 when the plan asks for it
template <class T>
int launch_p2p_t(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    k_p2p<T><<<P.num_sms * 16, LF_WARPS * 32, 0, s>>>(P.ctr, P.p2p_items, P.p2p_done, P.ctr, P.node_first,
                                                      P.node_count, P.node_nchild, (const vec4<T> *)P.xyzm, P.idx[0],
                                                      (const vec4<T> *)P.far, (vec4<T> *)P.far, P.p2p_off, P.p2p_src,
                                                      (T *)acc, (T *)pot);
    return 1;
}

int launch_p2p(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    if (P.mutual) return launch_p2p_mutual(P, acc, pot, s);
    if (P.dtype == 0) return launch_p2p_t<float>(P, acc, pot, s);
    return P.f64_ieee ? launch_p2p_t<double>(P, acc, pot, s) : launch_p2p_df(P, acc, pot, s);
}

}  // namespace bfm
