// Dual-tree walk and the interaction lists.
//
// JZ-FMM page, "Combining near and far interactions", stage 2: accept
// well-separated node pairs for multipole-to-local translations and refine the
// rest; the opening-criterion eq. accepts (A, B), A != B, when
// |l_A + l_B| < theta |c_A - c_B|, here evaluated squared, operation by
// operation in the plan's precision. The traversal is the symmetric one:
//   (A, A): a leaf gives P2P(A <- A); otherwise every child pair (C_i, C_j), i <= j;
//   (A, B) accepted: M2L both ways;
//   (A, B) both leaves: P2P both ways;
//   otherwise split the node with the larger |l| (the lower index on a tie),
//   never a leaf, and visit (child, other).
// The set of pairs this produces does not depend on the visiting order, so
// the walk runs breadth first, all frontier generations in one cooperative
// launch with a grid barrier between generations, appending through
// block-aggregated atomics on sharded output lists.
//
// Lists: per-receiver counts (taken during the walk) -> exclusive scan (one
// kernel, decoupled look-back) -> atomic fill -> every receiver's segment sorted
// ascending by source, which makes the order, and with it every later sum,
// independent of the atomics.
#include "plan.h"

namespace bfm {

namespace {

constexpr int WK_THREADS = 256;
constexpr int SEG_WARP_MAX = 1024;     // segments up to this length sort in a warp
constexpr int CS_THREADS = 256, CS_ITEMS = 4, CS_TILE = CS_THREADS * CS_ITEMS;

// Integer bits in a floating-point slot of a node record (stored and loaded,
// never computed with).
__device__ __forceinline__ float int_slot(int v, float) { return __int_as_float(v); }
__device__ __forceinline__ double int_slot(int v, double) { return __longlong_as_double((long long)v); }
__device__ __forceinline__ int slot_int(float v) { return __float_as_int(v); }
__device__ __forceinline__ int slot_int(double v) { return (int)__double_as_longlong(v); }

// The walk's first frontier, and every node's record for the walk: what it
// reads of a node (centre, half-widths, child count and first child) in one
// 2 x vec4<T> record, so a node costs two loads from one sector (fp32) instead
// of four loads from four arrays.
template <class T>
__global__ void k_walk_init(int2 *f0, const DevCounters *__restrict__ nctr, const vec4<T> *__restrict__ nc,
                            const vec4<T> *__restrict__ nl, const int *__restrict__ nchild,
                            const int *__restrict__ child0, vec4<T> *__restrict__ wrec, DevCounters *ctr)
{
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        f0[0] = make_int2(0, 0);
        ctr->frontier_cnt[0][0] = 1;
        ctr->frontier_max = 1;
    }
    const int n = phase2_nodes(nctr);
    for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < n; a += gridDim.x * blockDim.x) {
        const vec4<T> c = nc[a], l = nl[a];
        wrec[2 * a] = make4<T>(c.x, c.y, c.z, int_slot(nchild[a], T(0)));
        wrec[2 * a + 1] = make4<T>(l.x, l.y, l.z, int_slot(child0[a], T(0)));
    }
}

// Prefix over the shards of a sharded list (each shard's count clamped to its
// capacity) into s_pre[0 .. kShards]; called by a whole block of >= 64 threads.
// The 64 counts are read in parallel and scanned by two warps.
__device__ __forceinline__ void shard_prefix(const int *cnt, int cap_s, int *s_pre)
{
    __shared__ int s_half;
    const int t = threadIdx.x, lane = t & 31;
    int v = 0, incl = 0;
    if (t < kShards) {
        v = min(ld_cg(cnt + t), cap_s);
        incl = warp_incl_scan(v);
        if (t == 31) s_half = incl;
    }
    __syncthreads();
    if (t < kShards) {
        const int add = t >= 32 ? s_half : 0;
        s_pre[t] = add + incl - v;
        if (t == kShards - 1) s_pre[kShards] = add + incl;
    }
    (void)lane;
    __syncthreads();
}

// Storage address of element g of a sharded list (s_pre from shard_prefix).
__device__ __forceinline__ size_t shard_addr(const int *s_pre, int g, int cap_s)
{
    int lo = 0;
#pragma unroll
    for (int step = kShards / 2; step > 0; step >>= 1)
        if (s_pre[lo + step] <= g) lo += step;
    return (size_t)lo * cap_s + (g - s_pre[lo]);
}

// The walk: generations until the frontier is empty (at most `max_iters`; a
// walk of depth D ends after 2 D + 1, so running out sets ERR_WALK). In each
// generation every frontier pair is decided and
// its outputs (an M2L pair, a P2P pair or child pairs) are appended. Each output
// list is split into kShards shards with their own counters; a block reserves
// the space of a whole 256-pair tile in the shard of its index with one atomic
// per list, so no single counter is hot. The frontier and its counts were
// written by other blocks of this launch, so they are read through L2.
template <class T>
__global__ __launch_bounds__(WK_THREADS) void k_walk_all(int max_iters, int2 *f0, int2 *f1, int capf_s,
                                                         const int *__restrict__ count,
                                                         const vec4<T> *__restrict__ wrec, T th2, int2 *m2l_pairs,
                                                         int capm_s, int2 *p2p_pairs, int capp_s, int *m2l_cnt,
                                                         int *p2p_cnt, GridBarrier *gb, DevCounters *ctr)
{
    __shared__ int s_pre[kShards + 1];
    __shared__ int s_wtot[3][WK_THREADS / 32];
    __shared__ int s_base[3];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int bshard = blockIdx.x % kShards;
    long long inter_sum = 0;
    int visited = 0, fill_max = 0;
    const int iters = phase2_nodes(ctr) > 0 ? max_iters : 0;
    for (int it = 0; it < iters; ++it) {
        const int2 *fin = (it & 1) ? f1 : f0;
        int2 *fout = (it & 1) ? f0 : f1;
        int *cnt_out = ctr->frontier_cnt[(it + 1) % 3];
        if (blockIdx.x == 0 && threadIdx.x < kShards) ctr->frontier_cnt[(it + 2) % 3][threadIdx.x] = 0;
        shard_prefix(ctr->frontier_cnt[it % 3], capf_s, s_pre);
        const int nread = s_pre[kShards];
        if (nread == 0) break;  // the walk is complete (every block reads the same counts)
        if (it == iters - 1) {
            if (blockIdx.x == 0 && threadIdx.x == 0) set_error(ctr, ERR_WALK);
            break;
        }
        // each thread's next frontier pair is loaded one tile ahead, so its latency overlaps the
        // current tile's decisions, reservations and writes
        const int stride = gridDim.x * WK_THREADS;
        int2 pr_next = make_int2(-1, -1);
        if (blockIdx.x * WK_THREADS + threadIdx.x < nread)
            pr_next = ld_cg(fin + shard_addr(s_pre, blockIdx.x * WK_THREADS + threadIdx.x, capf_s));
        for (int base = blockIdx.x * WK_THREADS; base < nread; base += stride) {
            const int i = base + threadIdx.x;
            const int2 pr = pr_next;
            if (i + stride < nread) pr_next = ld_cg(fin + shard_addr(s_pre, i + stride, capf_s));
            int A = -1, B = -1, kids = 0, other = 0, m2l = 0, p2p = 0, c0 = 0;
            if (i < nread) {
                A = pr.x;
                B = pr.y;
                ++visited;
                const vec4<T> cA = wrec[2 * A], lA = wrec[2 * A + 1];
                const int nA = slot_int(cA.w), c0A = slot_int(lA.w);
                if (A == B) {
                    if (nA == 0) {
                        p2p = 1;
                        inter_sum += (long long)count[A] * count[A];
                    } else {
                        kids = nA * (nA + 1) / 2;
                        c0 = c0A;
                        other = nA;  // a self pair: the child count
                    }
                } else {
                    const vec4<T> cB = wrec[2 * B], lB = wrec[2 * B + 1];
                    const int nB = slot_int(cB.w), c0B = slot_int(lB.w);
                    const T s2 = norm2_rn(add_rn(lA.x, lB.x), add_rn(lA.y, lB.y), add_rn(lA.z, lB.z));
                    const T r2 = norm2_rn(sub_rn(cA.x, cB.x), sub_rn(cA.y, cB.y), sub_rn(cA.z, cB.z));
                    if (s2 < mul_rn(th2, r2)) {
                        m2l = 1;
                    } else if (nA == 0 && nB == 0) {
                        p2p = 1;
                        inter_sum += 2ll * count[A] * count[B];
                    } else {
                        // |l|^2 as the upward pass computed it for the node centres' records
                        const bool splitA = (nB == 0) ? true
                                          : ((nA == 0) ? false
                                                       : (norm2_rn(lA.x, lA.y, lA.z) >= norm2_rn(lB.x, lB.y, lB.z)));
                        other = splitA ? B : A;
                        kids = splitA ? nA : nB;
                        c0 = splitA ? c0A : c0B;
                    }
                }
            }
            // warp scans, then one exchange of the warp totals and one atomic per list per tile
            const int im = warp_incl_scan(m2l), ip = warp_incl_scan(p2p), ik = warp_incl_scan(kids);
            if (lane == 31) {
                s_wtot[0][warp] = im;
                s_wtot[1][warp] = ip;
                s_wtot[2][warp] = ik;
            }
            __syncthreads();
            if (threadIdx.x < 3) {
                const int list = threadIdx.x;
                int run = 0;
                for (int w2 = 0; w2 < WK_THREADS / 32; ++w2) {
                    const int t = s_wtot[list][w2];
                    s_wtot[list][w2] = run;
                    run += t;
                }
                int *ctrp = list == 0 ? &ctr->n_m2l_pairs[bshard] : (list == 1 ? &ctr->n_p2p_pairs[bshard] : &cnt_out[bshard]);
                const int b0 = run ? atomicAdd(ctrp, run) : 0;
                s_base[list] = b0;
                if (list == 2) fill_max = max(fill_max, b0 + run);
            }
            __syncthreads();
            if (m2l) {
                const int slot = s_base[0] + s_wtot[0][warp] + im - 1;
                if (slot < capm_s) {
                    m2l_pairs[(size_t)bshard * capm_s + slot] = make_int2(A, B);
                    atomicAdd(&m2l_cnt[A], 1);
                    atomicAdd(&m2l_cnt[B], 1);
                } else {
                    set_error(ctr, ERR_M2L_CAP);
                }
            }
            if (p2p) {
                const int slot = s_base[1] + s_wtot[1][warp] + ip - 1;
                if (slot < capp_s) {
                    p2p_pairs[(size_t)bshard * capp_s + slot] = make_int2(A, B);
                    atomicAdd(&p2p_cnt[A], 1);
                    if (A != B) atomicAdd(&p2p_cnt[B], 1);
                } else {
                    set_error(ctr, ERR_P2P_CAP);
                }
            }
            if (kids) {
                int o = s_base[2] + s_wtot[2][warp] + ik - kids;
                int2 *dst = fout + (size_t)bshard * capf_s;
                if (A == B) {
                    const int nA = other;
                    for (int x = 0; x < nA; ++x)
                        for (int y = x; y < nA; ++y, ++o) {
                            if (o < capf_s) dst[o] = make_int2(c0 + x, c0 + y);
                            else set_error(ctr, ERR_FRONTIER);
                        }
                } else {
                    for (int x = 0; x < kids; ++x, ++o) {
                        const int C = c0 + x;
                        if (o < capf_s) dst[o] = C < other ? make_int2(C, other) : make_int2(other, C);
                        else set_error(ctr, ERR_FRONTIER);
                    }
                }
            }
            __syncthreads();
        }
        if (!grid_barrier(gb, (unsigned)it, ctr)) break;
    }
    // per-warp statistics, one atomic each
    for (int o = 16; o > 0; o >>= 1) {
        inter_sum += __shfl_xor_sync(kFull, inter_sum, o);
        visited += __shfl_xor_sync(kFull, visited, o);
    }
    if (lane == 0) {
        if (inter_sum) atomicAdd((unsigned long long *)&ctr->p2p_interactions, (unsigned long long)inter_sum);
        if (visited) atomicAdd((unsigned long long *)&ctr->walk_pairs, (unsigned long long)visited);
    }
    if (threadIdx.x == 2 && fill_max) atomicMax(&ctr->frontier_max, fill_max);
}

// Exclusive scan of the per-receiver counts into CSR offsets (both lists at once).
__global__ __launch_bounds__(CS_THREADS) void k_csr_scan(const DevCounters *__restrict__ nctr, const int *__restrict__ m2l_cnt,
                                                         const int *__restrict__ p2p_cnt, int *__restrict__ m2l_off,
                                                         int *__restrict__ p2p_off, unsigned long long *flags,
                                                         unsigned epoch, int slot, DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    __shared__ int s_tile;
    __shared__ int s_w[2][CS_THREADS / 32];
    __shared__ long long s_ex[2];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntiles = (n_nodes + CS_TILE - 1) / CS_TILE;
    for (;;) {
        if (tid == 0) s_tile = (int)atomicAdd(&ctr->tile_ctr[slot], 1u);
        __syncthreads();
        const int tile = s_tile;
        if (tile >= ntiles) break;
        const int i0 = tile * CS_TILE + tid * CS_ITEMS;
        int a[CS_ITEMS], b[CS_ITEMS], sa = 0, sb = 0;
#pragma unroll
        for (int k = 0; k < CS_ITEMS; ++k) {
            const int i = i0 + k;
            a[k] = i < n_nodes ? m2l_cnt[i] : 0;
            b[k] = i < n_nodes ? p2p_cnt[i] : 0;
            sa += a[k];
            sb += b[k];
        }
        const int ia = warp_incl_scan(sa), ib = warp_incl_scan(sb);
        if (lane == 31) { s_w[0][warp] = ia; s_w[1][warp] = ib; }
        __syncthreads();
        if (warp < 2) {
            int tot = 0;
            for (int w = 0; w < CS_THREADS / 32; ++w) tot += s_w[warp][w];
            const long long ex = (long long)chained_exclusive_warp(flags + warp, 2, tile, (unsigned long long)tot,
                                                                   epoch, ctr);
            if (lane == 0) {
                s_ex[warp] = ex;
                if (tile == ntiles - 1) (warp == 0 ? m2l_off : p2p_off)[n_nodes] = (int)(ex + tot);
            }
        }
        __syncthreads();
        int wa = 0, wb = 0;
        for (int w = 0; w < warp; ++w) { wa += s_w[0][w]; wb += s_w[1][w]; }
        int ra = (int)s_ex[0] + wa + ia - sa, rb = (int)s_ex[1] + wb + ib - sb;
#pragma unroll
        for (int k = 0; k < CS_ITEMS; ++k) {
            const int i = i0 + k;
            if (i < n_nodes) {
                m2l_off[i] = ra;
                p2p_off[i] = rb;
            }
            ra += a[k];
            rb += b[k];
        }
        __syncthreads();
    }
}

// One directed entry per lane (receiver r >= 0; r < 0: none) into the
// receiver's segment: the lanes of a warp with the same receiver take their
// places with one atomic, the leader's, in lane order.
__device__ __forceinline__ void fill_entry(int r, int v, int *cnt, const int *__restrict__ off, int *__restrict__ src)
{
    const unsigned peers = __match_any_sync(kFull, r);
    const int leader = __ffs(peers) - 1;
    const int lane = threadIdx.x & 31;
    int top = 0;
    if (lane == leader && r >= 0) top = atomicSub(&cnt[r], __popc(peers));
    top = __shfl_sync(kFull, top, leader);
    if (r >= 0) src[off[r] + top - 1 - __popc(peers & lanemask_lt())] = v;
}

// Scatter the unordered pairs into their receivers' segments, both directions,
// one warp-aggregated atomic per receiver and warp (pairs of one receiver come
// in runs: the children of a split against the same partner). The counts are
// used as countdown cursors and end at zero, ready for the next evaluation.
__global__ void k_csr_fill(const int2 *__restrict__ m2l_pairs, int capm_s, const int2 *__restrict__ p2p_pairs,
                           int capp_s, int *m2l_cnt, int *p2p_cnt, const int *__restrict__ m2l_off,
                           const int *__restrict__ p2p_off, int *__restrict__ m2l_src, int *__restrict__ p2p_src,
                           const DevCounters *ctr)
{
    __shared__ int pm[kShards + 1], pp[kShards + 1];
    shard_prefix(ctr->n_m2l_pairs, capm_s, pm);
    shard_prefix(ctr->n_p2p_pairs, capp_s, pp);
    const int nm = pm[kShards], np = pp[kShards];
    const int lane = threadIdx.x & 31;
    const int stride = gridDim.x * blockDim.x;
    // the M2L pairs, then the P2P pairs: a warp's lanes are all in one list, two entries each
    for (int b = blockIdx.x * blockDim.x + (threadIdx.x & ~31); b < nm; b += stride) {
        const int i = b + lane;
        const int2 pr = i < nm ? m2l_pairs[shard_addr(pm, i, capm_s)] : make_int2(-1, -1);
        fill_entry(pr.x, pr.y, m2l_cnt, m2l_off, m2l_src);
        fill_entry(pr.y, pr.x, m2l_cnt, m2l_off, m2l_src);
    }
    for (int b = blockIdx.x * blockDim.x + (threadIdx.x & ~31); b < np; b += stride) {
        const int i = b + lane;
        const int2 pr = i < np ? p2p_pairs[shard_addr(pp, i, capp_s)] : make_int2(-1, -1);
        fill_entry(pr.x, pr.y, p2p_cnt, p2p_off, p2p_src);
        fill_entry(pr.x != pr.y ? pr.y : -1, pr.x, p2p_cnt, p2p_off, p2p_src);
    }
}

// Ascending bitonic network for any length: every merge starts with the
// mirrored compare, so padding at the top (+inf) never has to move.
__device__ __forceinline__ void cmpswap(int *v, int i, int j)
{
    const int a = v[i], b = v[j];
    if (b < a) { v[i] = b; v[j] = a; }
}

// Warp-wide ascending bitonic sort of 32 NR keys in the blocked layout: key
// e = NR lane + j in v[j], so partners at distances below NR are registers of
// the same lane and only the longer distances go through shuffles (15 of the
// 36 stages at NR = 8). The network is the flip-first one of cmpswap above:
// merge level k first compares e with its mirror e ^ (k - 1), then the
// half-cleaners compare e with e ^ d, d = k/4 .. 1; the lower key of a pair
// keeps the minimum. New values are always computed from old ones.
template <int NR>
__device__ __forceinline__ void warp_sort(int (&v)[NR])
{
    constexpr int N = 32 * NR;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
        if (k <= NR) {
            // mirror inside the lane: pairs (j, j ^ (k - 1)) with bit k/2 of j clear
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                const int pj = j ^ (k - 1);
                if ((j & (k >> 1)) == 0) {
                    const int a = v[j], b = v[pj];
                    v[j] = min(a, b);
                    v[pj] = max(a, b);
                }
            }
        } else {
            // mirror across lanes: lane ^ (k/NR - 1), register NR - 1 - j
            const int m = k / NR - 1;
            const bool lower = (lane & ((k >> 1) / NR)) == 0;
#pragma unroll
            for (int j = 0; j < NR / 2; ++j) {
                const int oa = __shfl_xor_sync(kFull, v[NR - 1 - j], m);
                const int ob = __shfl_xor_sync(kFull, v[j], m);
                const int a = v[j], b = v[NR - 1 - j];
                v[j] = lower ? min(a, oa) : max(a, oa);
                v[NR - 1 - j] = lower ? min(b, ob) : max(b, ob);
            }
            if constexpr (NR == 1) {
                const int o = __shfl_xor_sync(kFull, v[0], m);
                v[0] = lower ? min(v[0], o) : max(v[0], o);
            }
        }
#pragma unroll
        for (int d = k >> 2; d >= 1; d >>= 1) {
            if (d < NR) {
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    if ((j & d) == 0) {
                        const int a = v[j], b = v[j | d];
                        v[j] = min(a, b);
                        v[j | d] = max(a, b);
                    }
                }
            } else {
                const int m = d / NR;
                const bool lower = (lane & m) == 0;
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const int o = __shfl_xor_sync(kFull, v[j], m);
                    v[j] = lower ? min(v[j], o) : max(v[j], o);
                }
            }
        }
    }
}

// A list of up to 32 NR entries sorted in registers; for NR > 1 it moves
// between global memory and the blocked layout through the warp's shared
// buffer sv (coalesced global accesses, vector shared accesses).
template <int NR>
__device__ __forceinline__ void sort_list_regs(int *src, int len, int *sv)
{
    const int lane = threadIdx.x & 31;
    int v[NR];
    if constexpr (NR == 1) {
        v[0] = lane < len ? src[lane] : 0x7fffffff;
    } else {
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int e = j * 32 + lane;
            sv[e] = e < len ? src[e] : 0x7fffffff;
        }
        __syncwarp();
        if constexpr (NR % 4 == 0) {
#pragma unroll
            for (int j = 0; j < NR; j += 4) {
                const int4 x = *reinterpret_cast<const int4 *>(sv + lane * NR + j);
                v[j] = x.x;
                v[j + 1] = x.y;
                v[j + 2] = x.z;
                v[j + 3] = x.w;
            }
        } else {
            const int2 x = *reinterpret_cast<const int2 *>(sv + lane * NR);
            v[0] = x.x;
            v[1] = x.y;
        }
    }
    warp_sort<NR>(v);
    if constexpr (NR == 1) {
        if (lane < len) src[lane] = v[0];
    } else {
        __syncwarp();
        if constexpr (NR % 4 == 0) {
#pragma unroll
            for (int j = 0; j < NR; j += 4)
                *reinterpret_cast<int4 *>(sv + lane * NR + j) = make_int4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        } else {
            *reinterpret_cast<int2 *>(sv + lane * NR) = make_int2(v[0], v[1]);
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NR; ++j) {
            const int e = j * 32 + lane;
            if (e < len) src[e] = sv[e];
        }
        __syncwarp();
    }
}

// One warp per receiver list; lists up to 512 sort in registers, up to
// SEG_WARP_MAX in shared memory, longer ones go to a second pass.
__global__ __launch_bounds__(256) void k_segsort(const DevCounters *__restrict__ nctr, int cap, long long chunk_work,
                                                 long long share_div, int max_chunks, uint8_t *nchunks,
                                                 const int *__restrict__ m2l_off, int *m2l_src,
                                                 const int *__restrict__ p2p_off, int *p2p_src, int *long_seg,
                                                 const int *__restrict__ count, uint8_t *__restrict__ key,
                                                 DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    __shared__ __align__(16) int buf[8][SEG_WARP_MAX];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int *sv = buf[w];
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int job = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; job < 2 * n_nodes; job += nwarps) {
        const int a = job >> 1;
        const bool isp = job & 1;
        const int beg = isp ? p2p_off[a] : m2l_off[a];
        const int len = (isp ? p2p_off[a + 1] : m2l_off[a + 1]) - beg;
        int *src = (isp ? p2p_src : m2l_src) + beg;
        // work bucket of this receiver (see k_order_scatter): P2P work = count * sum of the
        // source leaves' counts, split into chunks of at most max(chunk_work, total / cap, total /
        // share_div) (at most max_chunks <= 255; so the chunks of all receivers number at most 2 cap),
        // bucketed by the work of one chunk; M2L work = list length; bucket floor(log2(work)) + 1, 0 for
        // none
        {
            int k, nch = 1;
            if (isp) {
                long long s = 0;
                for (int e = lane; e < len; e += 32) s += count[src[e]];
                for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
                const long long work = s * count[a];
                const long long tot = ctr->p2p_interactions;
                const long long wmax = max(chunk_work, max(tot / cap + 1, tot / share_div + 1));
                nch = (int)min((long long)max_chunks, (work + wmax - 1) / wmax);
                nch = max(nch, 1);
                const long long wc = work / nch;
                k = work > 0 ? 64 - __clzll(max(wc, 1ll)) : 0;
            } else {
                k = len > 0 ? 32 - __clz(len) : 0;
            }
            if (lane == 0) {
                key[(isp ? 0 : cap) + a] = (uint8_t)k;
                if (isp) nchunks[a] = (uint8_t)nch;
                if (k || !isp) atomicAdd(&ctr->order_cnt[isp ? 0 : 1][k], isp ? nch : 1);
            }
        }
        if (len <= 1) continue;
        if (len <= 32) { sort_list_regs<1>(src, len, sv); continue; }
        if (len <= 64) { sort_list_regs<2>(src, len, sv); continue; }
        if (len <= 128) { sort_list_regs<4>(src, len, sv); continue; }
        if (len <= 256) { sort_list_regs<8>(src, len, sv); continue; }
        if (len <= 512) { sort_list_regs<16>(src, len, sv); continue; }
        if (len > SEG_WARP_MAX) {
            if (lane == 0) long_seg[atomicAdd(&ctr->n_long, 1)] = job;
            continue;
        }
        int S = 2;
        while (S < len) S <<= 1;
        for (int i = lane; i < S; i += 32) sv[i] = i < len ? src[i] : 0x7fffffff;
        __syncwarp();
        for (int lk = 1; (1 << lk) <= S; ++lk) {
            const int k = 1 << lk;
            for (int i = lane; i < S / 2; i += 32) {
                const int blk = i >> (lk - 1), pos = i & ((k >> 1) - 1);
                cmpswap(sv, blk * k + pos, blk * k + k - 1 - pos);
            }
            __syncwarp();
            for (int lj = lk - 2; lj >= 0; --lj) {
                const int j = 1 << lj;
                for (int i = lane; i < S / 2; i += 32) {
                    const int blk = i >> lj, pos = i & (j - 1);
                    cmpswap(sv, (blk << (lj + 1)) + pos, (blk << (lj + 1)) + pos + j);
                }
                __syncwarp();
            }
        }
        for (int i = lane; i < len; i += 32) src[i] = sv[i];
        __syncwarp();
    }
}

// Long segments: one block each, the same network on global memory (indices at
// or beyond the length stand for +inf and are never touched).
__global__ __launch_bounds__(1024) void k_segsort_long(const int *__restrict__ m2l_off, int *m2l_src,
                                                       const int *__restrict__ p2p_off, int *p2p_src,
                                                       const int *__restrict__ long_seg, const DevCounters *ctr)
{
    const int nlong = ctr->n_long;
    for (int t = blockIdx.x; t < nlong; t += gridDim.x) {
        const int job = long_seg[t];
        const int a = job >> 1;
        const bool isp = job & 1;
        const int beg = isp ? p2p_off[a] : m2l_off[a];
        const int len = (isp ? p2p_off[a + 1] : m2l_off[a + 1]) - beg;
        int *v = (isp ? p2p_src : m2l_src) + beg;
        int S = 2;
        while (S < len) S <<= 1;
        for (int lk = 1; (1 << lk) <= S; ++lk) {
            const int k = 1 << lk;
            for (int i = threadIdx.x; i < S / 2; i += blockDim.x) {
                const int blk = i >> (lk - 1), pos = i & ((k >> 1) - 1);
                const int x = blk * k + pos, y = blk * k + k - 1 - pos;
                if (y < len) cmpswap(v, x, y);
            }
            __syncthreads();
            for (int lj = lk - 2; lj >= 0; --lj) {
                const int j = 1 << lj;
                for (int i = threadIdx.x; i < S / 2; i += blockDim.x) {
                    const int blk = i >> lj, pos = i & (j - 1);
                    const int x = (blk << (lj + 1)) + pos, y = x + j;
                    if (y < len) cmpswap(v, x, y);
                }
                __syncthreads();
            }
        }
    }
}

// Work order of the receivers, heaviest first: bucket b = floor(log2(work)) + 1
// (0 for no work), buckets taken in decreasing b (keys written by k_segsort).
// The order decides only which warp takes which receiver, never a result, so
// positions inside a bucket may come in any order: a block counts its nodes
// per bucket in shared memory and reserves their places with one atomic per
// bucket. The P2P items of a receiver split into chunks take consecutive
// places, in chunk order (a chunk's warp waits for the chunk before it, which
// was taken earlier).
__global__ __launch_bounds__(256) void k_order_scatter(const DevCounters *__restrict__ nctr, int cap,
                                                       const uint8_t *__restrict__ key,
                                                       const uint8_t *__restrict__ nchunks, int2 *p2p_items,
                                                       int *order, DevCounters *ctr)
{
    const int n_nodes = phase2_nodes(nctr);
    __shared__ int base[2][64], s_cnt[2][64], s_pos[2][64];
    const int tid = (int)threadIdx.x;
    if (tid < 2) {
        const int lowest = tid == 0 ? 1 : 0;  // P2P skips bucket 0 (no work); M2L keeps it, last
        int run = 0;
        for (int b = 63; b >= lowest; --b) {
            base[tid][b] = run;
            run += ctr->order_cnt[tid][b];
        }
    }
    for (int a0 = blockIdx.x * blockDim.x; a0 < n_nodes; a0 += gridDim.x * blockDim.x) {
        if (tid < 128) (&s_cnt[0][0])[tid] = 0;
        __syncthreads();
        const int a = a0 + tid;
        int kp = 0, km = 0, rp = -1, rm = -1, nch = 1;
        if (a < n_nodes) {
            kp = key[a];
            km = key[cap + a];
            nch = nchunks[a];
            if (kp) rp = atomicAdd(&s_cnt[0][kp], nch);
            rm = atomicAdd(&s_cnt[1][km], 1);
        }
        __syncthreads();
        if (tid < 128) {
            const int list = tid >> 6, b = tid & 63;
            const int c = s_cnt[list][b];
            s_pos[list][b] = c ? base[list][b] + atomicAdd(&ctr->order_cur[list][b], c) : 0;
        }
        __syncthreads();
        if (a < n_nodes) {
            if (kp)
                for (int c = 0; c < nch; ++c) {
                    const int slot = s_pos[0][kp] + rp + c;
                    if (slot < 2 * cap) p2p_items[slot] = make_int2(a, c | (nch << 8));
                    else set_error(ctr, ERR_BOUNDS);
                }
            order[cap + s_pos[1][km] + rm] = a;
        }
        __syncthreads();
    }
}

template <class T>
int launch_walk_t(Plan &P, int depth, cudaStream_t s)
{
    T th2 = (T)(P.theta * P.theta);
    k_walk_init<T><<<P.num_sms * 4, 256, 0, s>>>(P.frontier[0], P.ctr, (const vec4<T> *)P.node_c,
                                                  (const vec4<T> *)P.node_l, P.node_nchild, P.node_child0,
                                                  (vec4<T> *)P.node_w, P.ctr);
    int iters = 2 * kMaxLevel + 2;
    (void)depth;
    int capf_s = (int)(P.cap_frontier / kShards), capm_s = (int)(P.cap_m2l / kShards);
    int capp_s = (int)(P.cap_p2p / kShards);
    const vec4<T> *wrec = (const vec4<T> *)P.node_w;
    GridBarrier *gb = P.gbar + 1;
    void *args[] = {&iters, &P.frontier[0], &P.frontier[1], &capf_s, &P.node_count, (void *)&wrec, &th2,
                    &P.m2l_pairs, &capm_s, &P.p2p_pairs, &capp_s, &P.m2l_cnt, &P.p2p_cnt, &gb, &P.ctr};
    cudaLaunchCooperativeKernel((const void *)k_walk_all<T>, dim3(P.coop_blocks_walk), dim3(WK_THREADS), args, 0, s);
    return 2;
}

}  // namespace

int walk_max_blocks_per_sm(int dtype)
{
    int b = 0;
    if (dtype == 0) cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_walk_all<float>, WK_THREADS, 0);
    else cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_walk_all<double>, WK_THREADS, 0);
    return b;
}

int launch_walk(Plan &P, int depth, cudaStream_t s)
{
    return P.dtype == 0 ? launch_walk_t<float>(P, depth, s) : launch_walk_t<double>(P, depth, s);
}

constexpr long long kChunkWorkMutual = 1ll << 14;  // interactions per chunk of a mutual plan's receiver
constexpr int kMaxChunksMutual = 255;              // (chunk numbers are stored in 8 bits)

int launch_lists(Plan &P, cudaStream_t s)
{
    const int cap = (int)P.cap_nodes;
    const int slot = P.next_slot();
    const unsigned ep = P.next_epoch();
    k_csr_scan<<<P.num_sms * 4, CS_THREADS, 0, s>>>(P.ctr, P.m2l_cnt, P.p2p_cnt, P.m2l_off, P.p2p_off, P.flags, ep, slot,
                                                    P.ctr);
    k_csr_fill<<<P.num_sms * 8, 256, 0, s>>>(P.m2l_pairs, (int)(P.cap_m2l / kShards), P.p2p_pairs,
                                             (int)(P.cap_p2p / kShards), P.m2l_cnt, P.p2p_cnt, P.m2l_off, P.p2p_off,
                                             P.m2l_src, P.p2p_src, P.ctr);
    // fp64 mutual plans split heavy receivers much finer: their near-field kernel walks each partner leaf
    // in dependent steps of one pair per lane, so one warp on a receiver with a long list would be the
    // tail (the fp32 mutual kernel has the forward near field's lane layout and its chunks)
    const bool fine = P.mutual && P.dtype != 0;
    const long long chunk_work = fine ? kChunkWorkMutual : (P.dtype == 0 ? kChunkWork : kChunkWorkF64);
    const int max_chunks = fine ? kMaxChunksMutual : kMaxChunks;
    const long long share_div = (long long)P.num_sms * kShareDiv;
    k_segsort<<<P.num_sms * 8, 256, 0, s>>>(P.ctr, cap, chunk_work, share_div, max_chunks, P.p2p_nch, P.m2l_off, P.m2l_src, P.p2p_off, P.p2p_src, P.long_seg,
                                            P.node_count, P.order_key, P.ctr);
    k_segsort_long<<<P.num_sms, 1024, 0, s>>>(P.m2l_off, P.m2l_src, P.p2p_off, P.p2p_src, P.long_seg, P.ctr);
    k_order_scatter<<<P.num_sms * 4, 256, 0, s>>>(P.ctr, cap, P.order_key, P.p2p_nch, P.p2p_items, P.order, P.ctr);
    return 5;
}

}  // namespace bfm
