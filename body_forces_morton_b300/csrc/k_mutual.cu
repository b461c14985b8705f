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

template <class T>
int launch_p2p_mutual_t(Plan &P, void *acc, void *pot, cudaStream_t s)
{
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
