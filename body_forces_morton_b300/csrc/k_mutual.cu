// Mutual (symmetric) evaluation of the interaction lists.
//
// jaccpot issue 152, "Mutual FMM": every accepted pair of nodes is evaluated
// once and serves both receivers, which makes each level's forces equal and
// opposite by construction. For M2L that is one derivative tensor per
// unordered pair, D^m(-R) = (-1)^{|m|} D^m(R) giving the second direction
// (Exp<P>::m2l_r_pair, in k_m2l.cu); for P2P one separation, r^2 and
// reciprocal square root per unordered particle pair, whose opposite forces
// go to both particles (this file).
//
// Sums stay deterministic without floating-point atomics. The lists hold every
// unordered pair twice, once under each receiver, each segment sorted by
// source, so receiver a's segment is a lower part (sources < a), the self
// entry (P2P only) and an upper part (sources > a). A receiver evaluates the
// pairs of its upper part: its own share goes to its accumulators, the
// partner's share to the buffer slot of the mirrored entry (the entry for a in
// the partner's lower part). A second pass adds, for every receiver, its own
// sums and then the buffered shares of its lower part in list order.
//
//   k_mut_index  a warp per node: lower-part lengths of both lists, where the
//                P2P upper part starts, and the mirrored entry of every upper
//                entry (binary search in the partner's sorted segment);
//   k_mut_scan   a chained scan: each receiving leaf b gets count[b] x lower(b)
//                particle slots of the P2P buffer; if that buffer or the
//                per-entry ones are short, the evaluation grows them and runs
//                again;
//   k_p2p_mut1   a warp per receiving leaf: the self pair directed, as in the
//                forward near field; each upper partner leaf as a tile of
//                particle pairs walked in diagonal order, so that in one step
//                no two lanes touch the same partner particle, whose sums sit
//                in shared memory;
//   k_p2p_mut2   a warp per leaf, a lane per particle: own sums, the lower
//                part's buffered sums in list order and the far field, written
//                in the caller's order.
#include <climits>
#include <type_traits>

#include "expansions_gen.cuh"
#include "plan.h"

namespace bfm {

namespace {

constexpr int MUT_WARPS = 4;    // warps per block of k_p2p_mut1
constexpr int MUT_SLOTS = 128;  // staged partner particles per warp, shared by its lane groups

__global__ __launch_bounds__(256) void k_mut_index(const DevCounters *__restrict__ nctr,
                                                   const int *__restrict__ m2l_off, const int *__restrict__ m2l_src,
                                                   const int *__restrict__ p2p_off, const int *__restrict__ p2p_src,
                                                   int *__restrict__ lo_m2l, int *__restrict__ lo_p2p,
                                                   int *__restrict__ up_p2p, int *__restrict__ mir_m2l,
                                                   int *__restrict__ mir_p2p, long long cap_em, long long cap_ep,
                                                   DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
#pragma unroll 1
        for (int list = 0; list < 2; ++list) {
            const int *off = list ? p2p_off : m2l_off;
            const int *src = list ? p2p_src : m2l_src;
            int *mir = list ? mir_p2p : mir_m2l;
            const long long cap = list ? cap_ep : cap_em;  // entries beyond it: k_mut_scan reports the need
            const int beg = off[a], end = off[a + 1];
            int lo = 0, up = 0;
            for (int q0 = beg; q0 < end; q0 += 32) {
                const int q = q0 + lane;
                const int b = q < end ? src[q] : INT_MAX;
                lo += __popc(__ballot_sync(kFull, b < a));
                up += __popc(__ballot_sync(kFull, b <= a));
                if (q < end && b > a && q < cap) {
                    // first entry of b's segment whose source is not below a: the mirrored entry
                    int l = off[b], h = off[b + 1];
                    const int hb = h;
                    while (l < h) {
                        const int m = (l + h) >> 1;
                        if (src[m] < a) l = m + 1;
                        else h = m;
                    }
                    if (l < hb && src[l] == a) {
                        mir[q] = l;
                    } else {
                        mir[q] = -1;
                        set_error(ctr, ERR_BOUNDS);
                    }
                }
            }
            if (lane == 0) {
                if (list) {
                    lo_p2p[a] = lo;
                    up_p2p[a] = up;
                } else {
                    lo_m2l[a] = lo;
                }
            }
        }
    }
}

// Exclusive prefix of count[b] x lo_p2p[b] over the nodes (internal nodes have
// no P2P list, so they add nothing) into base[], base[n_nodes] the total: tiles
// of 1024 nodes taken from a ticket counter, chained by a decoupled look-back.
// The last tile also checks the three sized buffers: P2P share slots, M2L and
// P2P list entries (mirrored entries and M2L rows).
constexpr int MS_THREADS = 256, MS_ITEMS = 4, MS_TILE = MS_THREADS * MS_ITEMS;

__global__ __launch_bounds__(MS_THREADS) void k_mut_scan(const DevCounters *__restrict__ nctr,
                                                         const int *__restrict__ count, const int *__restrict__ lo_p2p,
                                                         const int *__restrict__ m2l_off,
                                                         const int *__restrict__ p2p_off, long long *__restrict__ base,
                                                         long long cap_rp, long long cap_em, long long cap_ep,
                                                         unsigned long long *flags, unsigned epoch, int slot,
                                                         DevCounters *ctr)
{
    __shared__ int s_tile;
    __shared__ long long s_w[MS_THREADS / 32];
    __shared__ long long s_ex;
    const int n = phase2_nodes(nctr);
    const int tid = (int)threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntiles = (n + MS_TILE - 1) / MS_TILE;
    for (;;) {
        if (tid == 0) s_tile = (int)atomicAdd(&ctr->tile_ctr[slot], 1u);
        __syncthreads();
        const int tile = s_tile;
        if (tile >= ntiles) break;
        const int i0 = tile * MS_TILE + tid * MS_ITEMS;
        long long v[MS_ITEMS], sum = 0;
#pragma unroll
        for (int k = 0; k < MS_ITEMS; ++k) {
            const int i = i0 + k;
            v[k] = i < n ? (long long)count[i] * lo_p2p[i] : 0;
            sum += v[k];
        }
        long long incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long t = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) s_w[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            long long tot = 0;
            for (int w = 0; w < MS_THREADS / 32; ++w) tot += s_w[w];
            const long long ex =
                (long long)chained_exclusive_warp(flags, 1, tile, (unsigned long long)tot, epoch, ctr);
            if (lane == 0) {
                s_ex = ex;
                if (tile == ntiles - 1) {
                    base[n] = ex + tot;
                    const long long need[3] = {ex + tot, (long long)m2l_off[n], (long long)p2p_off[n]};
                    const long long cap[3] = {cap_rp, cap_em, cap_ep};
                    for (int k = 0; k < 3; ++k)
                        if (need[k] > cap[k]) {
                            atomicMax(&ctr->mut_need[k], need[k]);
                            set_error(ctr, ERR_MUT_CAP);
                        }
                }
            }
        }
        __syncthreads();
        long long run = s_ex + incl - sum;
        for (int w = 0; w < warp; ++w) run += s_w[w];
#pragma unroll
        for (int k = 0; k < MS_ITEMS; ++k) {
            const int i = i0 + k;
            if (i < n) base[i] = run;
            run += v[k];
        }
        __syncthreads();
    }
}

// Source s on receiver p, one direction; MASKED skips a zero separation (the
// receiver itself in its own leaf).
template <class T>
__device__ __forceinline__ void pair_directed_masked(const vec4<T> &s, const vec4<T> &p, T (&A)[4])
{
    const T dx = s.x - p.x, dy = s.y - p.y, dz = s.z - p.z;
    const T r2 = dx * dx + dy * dy + dz * dz;
    T ri = rsqrt_t(r2);
    ri = r2 > T(0) ? ri : T(0);
    const T mr = s.w * ri;
    const T mr3 = mr * ri * ri;
    A[0] -= mr;
    A[1] += mr3 * dx;
    A[2] += mr3 * dy;
    A[3] += mr3 * dz;
}

// Particles i (in pi, sums A) and j (in pj, sums B) of two different leaves,
// so r > 0: one separation and reciprocal square root, opposite forces.
template <class T>
__device__ __forceinline__ void pair_mutual(const vec4<T> &pi, const vec4<T> &pj, T (&A)[4], vec4<T> &B)
{
    const T dx = pj.x - pi.x, dy = pj.y - pi.y, dz = pj.z - pi.z;
    const T r2 = dx * dx + dy * dy + dz * dz;
    const T ri = rsqrt_t(r2);
    const T ri3 = ri * ri * ri;
    const T mj3 = pj.w * ri3, mi3 = pi.w * ri3;
    A[0] -= pj.w * ri;
    A[1] += mj3 * dx;
    A[2] += mj3 * dy;
    A[3] += mj3 * dz;
    B.x -= pi.w * ri;
    B.y -= mi3 * dx;
    B.z -= mi3 * dy;
    B.w -= mi3 * dz;
}

template <class T> __device__ __forceinline__ vec4<T> add4(const vec4<T> &a, const vec4<T> &b)
{
    return make4<T>(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

// Pass 1 of the mutual near field, on the forward near field's work items (a
// receiving leaf, or one chunk of a split one: that chunk's share of the upper
// part; the self pair goes with chunk 0). The leaf's c particles take lanes in
// groups of G = min(32, next power of two >= c): lane = g G + il holds receiver
// il (blocks of 32 when c > 32) and group g takes the upper entries g, g +
// 32 / G, ... A group stages up to SG = MUT_SLOTS / (32 / G) particles of its
// partner leaf at a time, with zeroed sums, and walks m = max(rows, staged)
// steps: in step s lane il pairs its receiver with staged particle (il + s) mod
// m, distinct for distinct lanes, so every staged particle has at most one
// writer per step and its sum is added in step order, while every receiver row
// is busy in every step. The partner sums go to their buffer slots (added to
// those of the earlier receiver blocks, which the same lane wrote); the groups'
// sums of a receiver are added in a fixed butterfly, and the chunks of a split
// receiver add theirs to its own sums in chunk order (each waits, bounded, for
// the one before).
template <class T>
__global__ __launch_bounds__(MUT_WARPS * 32) void k_p2p_mut1(
    const DevCounters *__restrict__ cst, const int2 *__restrict__ items, int *done, DevCounters *ctr,
    const int *__restrict__ first, const int *__restrict__ count, const vec4<T> *__restrict__ xyzm,
    const int *__restrict__ off, const int *__restrict__ src, const int *__restrict__ up_p2p,
    const int *__restrict__ mir, long long cap_ep, const long long *__restrict__ base, long long cap_rp,
    vec4<T> *rbuf, vec4<T> *own)
{
    __shared__ vec4<T> s_x[MUT_WARPS][MUT_SLOTS];
    __shared__ vec4<T> s_b[MUT_WARPS][MUT_SLOTS];
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
        const int u0 = off[a] + up_p2p[a], ulen = off[a + 1] - u0;
        const int ub = u0 + (int)((long long)ulen * chunk / nch), ue = u0 + (int)((long long)ulen * (chunk + 1) / nch);
        int G = 1;
        while (G < c && G < 32) G <<= 1;
        const int ng = 32 / G, g = lane / G, il = lane - g * G;
        const int SG = MUT_SLOTS / ng;
        vec4<T> *const gx = s_x[w] + g * SG, *const gb = s_b[w] + g * SG;
        for (int i0 = 0; i0 < c; i0 += 32) {
            const int ci = min(c - i0, G);  // receiver rows of this block
            const int i = i0 + il;
            const bool iv = il < ci;
            const vec4<T> pi = xyzm[f + (iv ? i : 0)];
            T A[4] = {T(0), T(0), T(0), T(0)};
            // the leaf itself, directed (sources j = g, g + ng, ...)
            if (chunk == 0 && iv)
                for (int j = g; j < c; j += ng) pair_directed_masked<T>(xyzm[f + j], pi, A);
            // this item's upper partners
            for (int q0 = ub; q0 < ue; q0 += ng) {
                const int q = q0 + g;
                const bool qv = q < ue;
                int fb = 0, cb = 0;
                long long slot = 0;
                if (qv) {
                    const int b = src[q];
                    const int m = q < cap_ep ? mir[q] : -1;
                    fb = first[b];
                    cb = count[b];
                    slot = m >= 0 ? base[b] + (long long)(m - off[b]) * cb : LLONG_MAX / 2;
                }
                int cmax = cb;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) cmax = max(cmax, __shfl_xor_sync(kFull, cmax, o));
                for (int j0 = 0; j0 < cmax; j0 += SG) {
                    const int nb = qv ? max(0, min(SG, cb - j0)) : 0;
                    __syncwarp();
                    for (int k = il; k < nb; k += G) {
                        gx[k] = xyzm[fb + j0 + k];
                        gb[k] = make4<T>(T(0), T(0), T(0), T(0));
                    }
                    __syncwarp();
                    const int m = nb > 0 ? max(ci, nb) : 0;
                    int msteps = m;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) msteps = max(msteps, __shfl_xor_sync(kFull, msteps, o));
                    for (int st = 0; st < msteps; ++st) {
                        int jj = il + st;
                        jj = jj >= m ? jj - m : jj;
                        if (st < m && iv && jj < nb) {
                            vec4<T> B = gb[jj];
                            pair_mutual<T>(pi, gx[jj], A, B);
                            gb[jj] = B;
                        }
                        __syncwarp();
                    }
                    for (int k = il; k < nb; k += G) {
                        const long long kk = slot + j0 + k;
                        if (kk >= 0 && kk < cap_rp) {
                            vec4<T> v = gb[k];
                            if (i0 > 0) v = add4<T>(v, rbuf[kk]);
                            rbuf[kk] = v;
                        } else {
                            set_error(ctr, ERR_BOUNDS);
                        }
                    }
                }
            }
            // the groups' sums of receiver il, added in a fixed butterfly
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                if (o >= G)
#pragma unroll
                    for (int v = 0; v < 4; ++v) A[v] += __shfl_xor_sync(kFull, A[v], o);
            // a split receiver's chunks add their sums in chunk order
            if (nch > 1 && i0 == 0) wait_turn(done + a, chunk, ctr);
            if (g == 0 && iv) {
                vec4<T> v = make4<T>(A[0], A[1], A[2], A[3]);
                if (chunk > 0) v = add4<T>(ld_cg(own + f + i), v);  // written by another warp: through L2
                own[f + i] = v;
            }
        }
        if (nch > 1 && chunk < nch - 1) pass_turn(done + a, chunk + 1);
    }
}

// Pass 2: a warp per leaf, a lane per particle.
template <class T>
__global__ __launch_bounds__(256) void k_p2p_mut2(const DevCounters *__restrict__ nctr, const int *__restrict__ first,
                                                  const int *__restrict__ count, const int *__restrict__ nchild,
                                                  const int *__restrict__ lo_p2p, const long long *__restrict__ base,
                                                  long long cap_rp, const vec4<T> *__restrict__ rbuf,
                                                  const vec4<T> *__restrict__ own, const vec4<T> *__restrict__ far,
                                                  const uint32_t *__restrict__ perm, T *__restrict__ acc_out,
                                                  T *__restrict__ pot_out, DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int a = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; a < n_nodes; a += nwarps) {
        if (nchild[a] != 0) continue;
        const int f = first[a], c = count[a], nlo = lo_p2p[a];
        const long long b0 = base[a];
        if (b0 + (long long)nlo * c > cap_rp) {
            if (lane == 0) set_error(ctr, ERR_BOUNDS);
            continue;
        }
        for (int i = lane; i < c; i += 32) {
            vec4<T> t = own[f + i];
            for (int k = 0; k < nlo; ++k) t = add4<T>(t, rbuf[b0 + (long long)k * c + i]);
            const vec4<T> fa = far[f + i];
            const uint32_t o = perm[f + i];
            acc_out[3 * (size_t)o] = fa.y + t.y;
            acc_out[3 * (size_t)o + 1] = fa.z + t.z;
            acc_out[3 * (size_t)o + 2] = fa.w + t.w;
            if (pot_out) pot_out[o] = fa.x + t.x;
        }
    }
}

// ---- fp32: the mutual near field on the forward near field's lane layout ----
// k_p2p_mutf replaces k_p2p_mut1 for fp32 plans. A round holds up to 32 K
// receivers of leaf a: lane = q R + rp (rp < R = ceil(cr / K), q < S = 32 / R)
// holds receivers rp + k R, k < K; the lanes of group q walk the staged
// partner particles in pairs q, q + S, ..., two sources per f32x2
// instruction. For each source pair a lane sums the reaction of its K
// receivers in registers; every MF_FLUSH steps the group's R partial reactions
// of each pair go through shared memory and are added in order of rp by one lane
// of the group (a transpose: lane rp of the group finishes the flush's rp-th
// pair), which adds them to the pair's buffer slots. Receivers beyond the leaf
// (the last round's padding) carry zero mass, so they react with nothing.
constexpr int MF_WARPS = 4;
constexpr int MF_CH = 256;    // staged partner particles per chunk
constexpr int MF_K = 4;       // receivers per lane
constexpr int MF_FLUSH = 6;   // source-pair steps per flush of the partial reactions (shared memory: 4 blocks per SM)

struct MfWarp {
    float pos[MF_CH * 4];              // pair-interleaved (x0, x1, y0, y1, z0, z1, m0, m1) per source pair
    long long dst[MF_CH];              // share slot of each staged particle (-1: a padding particle)
    float4 part[MF_FLUSH][65];         // a flush's partial reactions: step, then lane x two float4 of packed
                                       // halves, rows padded to an odd number of 16-byte units (the finishing
                                       // lanes read down a column)
    float red[32][4];                  // the receivers' sums over the S groups
};

__device__ __forceinline__ float rsqrt_fast(float x)
{
    float y;
    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Sources (SX, SY, SZ, SM: two particles) and one receiver (negated position
// NX, NY, NZ and mass MI, both halves equal): the receiver's sums A (sum m_j /
// r, then the acceleration) and the sources' reaction B (their potential, then
// their acceleration), in packed halves.
__device__ __forceinline__ void mf_pair(float2 SX, float2 SY, float2 SZ, float2 SM, float2 NX, float2 NY, float2 NZ,
                                        float2 NMI, float2 (&A)[4], float2 (&B)[4])
{
    const float2 dx = __fadd2_rn(SX, NX), dy = __fadd2_rn(SY, NY), dz = __fadd2_rn(SZ, NZ);
    float2 r2 = __fmul2_rn(dx, dx);
    r2 = __ffma2_rn(dy, dy, r2);
    r2 = __ffma2_rn(dz, dz, r2);
    const float2 ri = make_float2(rsqrt_fast(r2.x), rsqrt_fast(r2.y));
    const float2 ri2 = __fmul2_rn(ri, ri);
    const float2 mr = __fmul2_rn(SM, ri);
    const float2 mr3 = __fmul2_rn(mr, ri2);
    A[0] = __fadd2_rn(A[0], mr);
    A[1] = __ffma2_rn(mr3, dx, A[1]);
    A[2] = __ffma2_rn(mr3, dy, A[2]);
    A[3] = __ffma2_rn(mr3, dz, A[3]);
    const float2 nmr = __fmul2_rn(NMI, ri);  // -m_i / r
    const float2 nmr3 = __fmul2_rn(nmr, ri2);
    B[0] = __fadd2_rn(B[0], nmr);            // the sources' potential
    B[1] = __ffma2_rn(nmr3, dx, B[1]);       // and acceleration, -m_i (x_j - x_i) / r^3
    B[2] = __ffma2_rn(nmr3, dy, B[2]);
    B[3] = __ffma2_rn(nmr3, dz, B[3]);
}

// One source of the own leaf (zero separations masked) on one receiver, scalar.
__device__ __forceinline__ void mf_own(const float4 &s, float x, float y, float z, float (&a)[4])
{
    const float dx = s.x - x, dy = s.y - y, dz = s.z - z;
    const float r2 = dx * dx + dy * dy + dz * dz;
    const float ri = r2 > 0.0f ? rsqrt_fast(r2) : 0.0f;
    const float mr = s.w * ri;
    const float mr3 = mr * ri * ri;
    a[0] += mr;
    a[1] += mr3 * dx;
    a[2] += mr3 * dy;
    a[3] += mr3 * dz;
}

__device__ __forceinline__ void mf_put_pad(float *pb, int k)
{
    float *d = pb + (k >> 1) * 8 + (k & 1);
    d[0] = d[2] = d[4] = 1e18f;
    d[6] = 0.0f;
}

// Add a finished flush: lane rp < nf of group q adds the R partials of source
// pair (pair0 + (t0 + rp) S) in order of rp' and adds the two sources' sums to
// their slots (round 0 stores, later rounds of the same receiver add).
__device__ __forceinline__ void mf_flush(MfWarp &W, int nf, int t0, int q, int rp, int R, int S, bool worker,
                                         int npairs, bool first_round, float4 *rbuf, long long cap_rp,
                                         DevCounters *ctr)
{
    __syncwarp();
    if (worker && rp < nf) {
        const int j = q + (t0 + rp) * S;  // the pair this lane finishes
        if (j < npairs) {
            float4 u = W.part[rp][2 * (q * R)], v = W.part[rp][2 * (q * R) + 1];
            float2 u0 = make_float2(u.x, u.y), u1 = make_float2(u.z, u.w);
            float2 v0 = make_float2(v.x, v.y), v1 = make_float2(v.z, v.w);
            for (int r = 1; r < R; ++r) {  // packed adds, in order of r
                const float4 u2 = W.part[rp][2 * (q * R + r)], v2 = W.part[rp][2 * (q * R + r) + 1];
                u0 = __fadd2_rn(u0, make_float2(u2.x, u2.y));
                u1 = __fadd2_rn(u1, make_float2(u2.z, u2.w));
                v0 = __fadd2_rn(v0, make_float2(v2.x, v2.y));
                v1 = __fadd2_rn(v1, make_float2(v2.z, v2.w));
            }
            u = make_float4(u0.x, u0.y, u1.x, u1.y);
            v = make_float4(v0.x, v0.y, v1.x, v1.y);
            // u = (pot0, pot1, ax0, ax1), v = (ay0, ay1, az0, az1)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const long long d = W.dst[2 * j + h];
                if (d < 0) continue;
                if (d >= cap_rp) {
                    set_error(ctr, ERR_BOUNDS);
                    continue;
                }
                float4 val = h == 0 ? make_float4(u.x, u.z, v.x, v.z) : make_float4(u.y, u.w, v.y, v.w);
                if (!first_round) {
                    const float4 old = rbuf[d];
                    val = make_float4(old.x + val.x, old.y + val.y, old.z + val.z, old.w + val.w);
                }
                rbuf[d] = val;
            }
        }
    }
    __syncwarp();
}

// One round of up to 32 K receivers [r0, r0 + cr) of leaf a against the upper
// entries [ub, ue) of its list (and, for the first chunk, its own leaf).
template <bool CHUNKED>
__device__ __forceinline__ void mf_round(int a, int f, int c, int r0, int cr, int ub, int ue, int chunk, int *done,
                                         DevCounters *ctr, const int *__restrict__ first,
                                         const int *__restrict__ count, const float4 *__restrict__ xyzm,
                                         const int *__restrict__ off, const int *__restrict__ src,
                                         const int *__restrict__ mir, long long cap_ep,
                                         const long long *__restrict__ base, long long cap_rp, float4 *rbuf,
                                         float4 *own, MfWarp &W, int lane)
{
    constexpr int K = MF_K;
    const int R = (cr + K - 1) / K, S = 32 / R;
    const int rp = lane % R, q = lane / R;
    const bool worker = q < S;
    const int F = R < MF_FLUSH ? R : MF_FLUSH;  // steps per flush: a group's lanes finish one pair each
    float2 NX[K], NY[K], NZ[K], NMI[K];
    float2 A[K][4];
#pragma unroll
    for (int k = 0; k < K; ++k) {
        const int rr = rp + k * R;
        const bool valid = rr < cr;
        const float4 x = xyzm[f + r0 + (valid ? rr : 0)];
        NX[k] = make_float2(-x.x, -x.x);
        NY[k] = make_float2(-x.y, -x.y);
        NZ[k] = make_float2(-x.z, -x.z);
        NMI[k] = valid ? make_float2(-x.w, -x.w) : make_float2(0.0f, 0.0f);  // padding receivers: no reaction
#pragma unroll
        for (int v = 0; v < 4; ++v) A[k][v] = make_float2(0.0f, 0.0f);
    }
    // the leaf's own particles, directed (zero separations masked), with the first chunk
    if (!CHUNKED || chunk == 0) {
        float o[K][4];
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int v = 0; v < 4; ++v) o[k][v] = 0.0f;
        float4 *buf = reinterpret_cast<float4 *>(W.pos);
        for (int g0 = 0; g0 < c; g0 += MF_CH) {
            const int n_here = min(MF_CH, c - g0);
            __syncwarp();
            for (int k = lane; k < n_here; k += 32) buf[k] = xyzm[f + g0 + k];
            __syncwarp();
            if (worker)
                for (int j = q; j < n_here; j += S) {
                    const float4 s4 = buf[j];
#pragma unroll
                    for (int k = 0; k < K; ++k) mf_own(s4, -NX[k].x, -NY[k].x, -NZ[k].x, o[k]);
                }
        }
#pragma unroll
        for (int k = 0; k < K; ++k)
#pragma unroll
            for (int v = 0; v < 4; ++v) A[k][v].x += o[k][v];
    }
    const float4 *pb = reinterpret_cast<const float4 *>(W.pos);
    // the upper partners, 32 list entries at a time (lane i holds entry lb + i and its share slot); the
    // next group's entries load while this one computes
    auto fetch = [&](int lb, int &fb, int &cb, long long &sl) {
        const int e = lb + lane;
        fb = 0;
        cb = 0;
        sl = -1;
        if (e < ue) {
            const int b = src[e];
            const int m = e < cap_ep ? mir[e] : -1;
            fb = first[b];
            cb = count[b];
            sl = m >= 0 ? base[b] + (long long)(m - off[b]) * cb : -1;
        }
    };
    int fb_n = 0, cb_n = 0;
    long long sl_n = -1;
    if (ub < ue) fetch(ub, fb_n, cb_n, sl_n);
    for (int lb = ub; lb < ue; lb += 32) {
        const int fb = fb_n, cb = cb_n;
        const long long sl = sl_n;
        if (lb + 32 < ue) fetch(lb + 32, fb_n, cb_n, sl_n);
        const int incl = warp_incl_scan(cb);
        const int tot = __shfl_sync(kFull, incl, 31);
        const int ex = incl - cb;
        for (int g0 = 0; g0 < tot; g0 += MF_CH) {
            const int n_here = min(MF_CH, tot - g0);
            __syncwarp();
            for (int k0 = 0; k0 < n_here; k0 += 32) {  // warp-uniform: every lane takes part in the shuffles
                const int k = k0 + lane;
                const int g = g0 + k;
                int lo = 0;  // last lane whose leaf starts at or before g
#pragma unroll
                for (int step = 16; step > 0; step >>= 1) {
                    const int exm = __shfl_sync(kFull, ex, lo + step);
                    lo = exm <= g ? lo + step : lo;
                }
                const int fs = __shfl_sync(kFull, fb, lo);
                const int es = __shfl_sync(kFull, ex, lo);
                const long long ss = __shfl_sync(kFull, sl, lo);
                if (k < n_here) {
                    const float *v = reinterpret_cast<const float *>(xyzm + fs + (g - es));
                    float *d = W.pos + (k >> 1) * 8 + (k & 1);
                    cp_async4(d, v);
                    cp_async4(d + 2, v + 1);
                    cp_async4(d + 4, v + 2);
                    cp_async4(d + 6, v + 3);
                    W.dst[k] = ss >= 0 ? ss + (g - es) : -1;
                }
            }
            if ((n_here & 1) && lane == 0) {
                mf_put_pad(W.pos, n_here);
                W.dst[n_here] = -1;
            }
            cp_async_wait_all();
            __syncwarp();
            const int npairs = (n_here + 1) >> 1;
            const int T = (npairs + S - 1) / S;  // steps: pair q + t S of group q at step t
            for (int t0 = 0; t0 < T; t0 += F) {
                const int nf = min(F, T - t0);
                for (int tt = 0; tt < nf; ++tt) {
                    const int j = q + (t0 + tt) * S;
                    float2 B[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                                   make_float2(0.0f, 0.0f)};
                    if (worker && j < npairs) {
                        const float4 p0 = pb[2 * j], p1 = pb[2 * j + 1];
                        const float2 SX = make_float2(p0.x, p0.y), SY = make_float2(p0.z, p0.w);
                        const float2 SZ = make_float2(p1.x, p1.y), SM = make_float2(p1.z, p1.w);
#pragma unroll
                        for (int k = 0; k < K; ++k) mf_pair(SX, SY, SZ, SM, NX[k], NY[k], NZ[k], NMI[k], A[k], B);
                    }
                    W.part[tt][2 * lane] = make_float4(B[0].x, B[0].y, B[1].x, B[1].y);
                    W.part[tt][2 * lane + 1] = make_float4(B[2].x, B[2].y, B[3].x, B[3].y);
                }
                mf_flush(W, nf, t0, q, rp, R, S, worker, npairs, r0 == 0, rbuf, cap_rp, ctr);
            }
        }
    }
    // the receivers' sums over the S groups, then the chunks of a split receiver in chunk order
    if (CHUNKED && r0 == 0) wait_turn(done + a, chunk, ctr);
#pragma unroll
    for (int k = 0; k < K; ++k) {
        __syncwarp();
        W.red[lane][0] = A[k][0].x + A[k][0].y;
        W.red[lane][1] = A[k][1].x + A[k][1].y;
        W.red[lane][2] = A[k][2].x + A[k][2].y;
        W.red[lane][3] = A[k][3].x + A[k][3].y;
        __syncwarp();
        const int rr = rp + k * R;
        if (q == 0 && rr < cr) {
            float t[4] = {W.red[rp][0], W.red[rp][1], W.red[rp][2], W.red[rp][3]};
            for (int qs = 1; qs < S; ++qs)
#pragma unroll
                for (int v = 0; v < 4; ++v) t[v] += W.red[qs * R + rp][v];
            const int i = f + r0 + rr;
            float4 v = make_float4(-t[0], t[1], t[2], t[3]);
            if (CHUNKED && chunk > 0) {
                const float4 prev = ld_cg(own + i);  // the earlier chunks' sums, written by other warps
                v = make_float4(prev.x + v.x, prev.y + v.y, prev.z + v.z, prev.w + v.w);
            }
            own[i] = v;
        }
    }
}

__global__ __launch_bounds__(MF_WARPS * 32) void k_p2p_mutf(
    const DevCounters *__restrict__ cst, const int2 *__restrict__ items, int *done, DevCounters *ctr,
    const int *__restrict__ first, const int *__restrict__ count, const float4 *__restrict__ xyzm,
    const int *__restrict__ off, const int *__restrict__ src, const int *__restrict__ up_p2p,
    const int *__restrict__ mir, long long cap_ep, const long long *__restrict__ base, long long cap_rp,
    float4 *rbuf, float4 *own)
{
    extern __shared__ __align__(16) unsigned char mf_smem[];
    MfWarp &W = reinterpret_cast<MfWarp *>(mf_smem)[threadIdx.x >> 5];
    const int lane = threadIdx.x & 31;
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
        const int u0 = off[a] + up_p2p[a], ulen = off[a + 1] - u0;
        const int ub = u0 + (int)((long long)ulen * chunk / nch), ue = u0 + (int)((long long)ulen * (chunk + 1) / nch);
        for (int r0 = 0; r0 < c; r0 += 32 * MF_K) {
            const int cr = min(32 * MF_K, c - r0);
            if (nch == 1)
                mf_round<false>(a, f, c, r0, cr, ub, ue, 0, done, ctr, first, count, xyzm, off, src, mir, cap_ep,
                                base, cap_rp, rbuf, own, W, lane);
            else
                mf_round<true>(a, f, c, r0, cr, ub, ue, chunk, done, ctr, first, count, xyzm, off, src, mir, cap_ep,
                               base, cap_rp, rbuf, own, W, lane);
        }
        if (nch > 1 && chunk < nch - 1) pass_turn(done + a, chunk + 1);
    }
}

template <class T>
int launch_p2p_mutual_t(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    if constexpr (std::is_same<T, float>::value) {
        const int smem = MF_WARPS * (int)sizeof(MfWarp);
        cudaFuncSetAttribute(k_p2p_mutf, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        k_p2p_mutf<<<P.num_sms * 16, MF_WARPS * 32, smem, s>>>(
            P.ctr, P.p2p_items, P.p2p_done, P.ctr, P.node_first, P.node_count, (const float4 *)P.xyzm, P.p2p_off,
            P.p2p_src, P.mut_lo + 2 * P.cap_nodes, P.mut_mir_p2p, P.mut_cap_ep, P.mut_base, P.mut_cap_rp,
            (float4 *)P.mut_rp2p, (float4 *)P.mut_own);
    } else
    k_p2p_mut1<T><<<P.num_sms * 16, MUT_WARPS * 32, 0, s>>>(
        P.ctr, P.p2p_items, P.p2p_done, P.ctr, P.node_first, P.node_count, (const vec4<T> *)P.xyzm, P.p2p_off, P.p2p_src,
        P.mut_lo + 2 * P.cap_nodes, P.mut_mir_p2p, P.mut_cap_ep, P.mut_base, P.mut_cap_rp, (vec4<T> *)P.mut_rp2p,
        (vec4<T> *)P.mut_own);
    k_p2p_mut2<T><<<P.num_sms * 8, 256, 0, s>>>(P.ctr, P.node_first, P.node_count, P.node_nchild,
                                                P.mut_lo + P.cap_nodes, P.mut_base, P.mut_cap_rp,
                                                (const vec4<T> *)P.mut_rp2p, (const vec4<T> *)P.mut_own,
                                                (const vec4<T> *)P.far, P.idx[0], (T *)acc, (T *)pot, P.ctr);
    return 2;
}

}  // namespace

int launch_mutual_index(Plan &P, cudaStream_t s)
{
    const int64_t c = P.cap_nodes;
    k_mut_index<<<P.num_sms * 8, 256, 0, s>>>(P.ctr, P.m2l_off, P.m2l_src, P.p2p_off, P.p2p_src, P.mut_lo,
                                              P.mut_lo + c, P.mut_lo + 2 * c, P.mut_mir_m2l, P.mut_mir_p2p,
                                              P.mut_cap_em, P.mut_cap_ep, P.ctr);
    const int slot = P.next_slot();
    const unsigned ep = P.next_epoch();
    k_mut_scan<<<P.num_sms * 2, MS_THREADS, 0, s>>>(P.ctr, P.node_count, P.mut_lo + c, P.m2l_off, P.p2p_off,
                                                    P.mut_base, P.mut_cap_rp, P.mut_cap_em, P.mut_cap_ep, P.flags, ep,
                                                    slot, P.ctr);
    return 2;
}

int launch_p2p_mutual(Plan &P, void *acc, void *pot, cudaStream_t s)
{
    return P.dtype == 0 ? launch_p2p_mutual_t<float>(P, acc, pot, s) : launch_p2p_mutual_t<double>(P, acc, pot, s);
}

}  // namespace bfm
