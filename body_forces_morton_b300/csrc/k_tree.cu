// Octree over the sorted Morton keys.
//
// JZ-FMM page, "Why this works well on GPUs": the tree stores child nodes next
// to each other. A node of level l holding more than `leaf` particles splits
// into its non-empty octants at level l+1 (at most 21 levels). Nodes are
// numbered breadth first: level by level, within a level in key order, so the
// children of one node are contiguous and follow the children of the nodes
// before it.
//
// Every level at once (leaf <= TB_LEAF_MAX). With div[k] the first level at
// which sorted keys k-1 and k fall in different cells, the level-l cells are
// the runs of positions between the boundaries {k : div[k] <= l}. Such a run is
// a node exactly when its parent run holds more than `leaf` keys, and a run
// holds more than `leaf` keys exactly when some window of leaf + 1 consecutive
// positions lies inside it. So with
//     W(x) = min(div[x+1 .. x+leaf])        (the window starting at x),
//     V(k) = max(W(x) : x in [k-leaf, k])   (the windows holding position k),
// the level-l run through k is a node iff l = 0 or V(k) >= l, and the levels
// whose nodes start at k form the range [div[k], min(21, V(k))] (k = 0: from
// 0). A node's breadth-first index is its level's offset plus the number of
// nodes of that level starting before it. Its parent, first child and end are
// nodes and positions the same two numbers locate: the parent is the last node
// of level l - 1 starting at or before k, the first child the level-(l+1) node
// starting at k, and the node of level l through k - 1 ends at k whenever k is
// a level-l boundary; count and nchild are each the difference of one value
// added at the start and one at the end. Three launches: the windows and the
// node counts per chunk of positions; a scan of the counts per level; the
// nodes.
//
// Level by level (larger leaves): every node's child starts come from binary
// searches on the keys, one cooperative launch with a grid barrier per level.
#include "plan.h"

namespace bfm {

namespace {

constexpr int TR_THREADS = 128;

// Node count and depth for the later stages: the deepest level holding nodes,
// and the nodes up to it (at most the node capacity).
__device__ void record_tree_size(DevCounters *ctr, int cap_nodes)
{
    int depth = 0;
    for (int l = 0; l <= kMaxLevel; ++l)
        if (ld_cg(&ctr->level_off[l + 1]) > ld_cg(&ctr->level_off[l])) depth = l;
    ctr->depth = depth;
    ctr->n_nodes = min(ld_cg(&ctr->level_off[depth + 1]), cap_nodes);
}

// All levels in one cooperative launch: a tile is 32 consecutive nodes of the
// level, one per lane of a warp; tiles are taken from the level's ticket
// counter. A lane finds its node's child boundaries by seven branchless
// lower-bound searches (digit >= 1 .. 7 of the key at level + 1, which ascends
// within the node) that advance in lockstep, so their loads overlap. A warp
// scan of the child counts plus the look-back over earlier tiles numbers the
// children breadth first. A grid barrier separates the levels (the next level's
// nodes are this level's output); the loop ends at the first empty level.
// Node data of the current level was written by other blocks of this launch,
// so it is read through L2.
__global__ __launch_bounds__(TR_THREADS) void k_tree_all(int leaf, int cap_nodes, const uint64_t *__restrict__ keys,
                                                         int *first, int *count, int *child0, int *nchild,
                                                         int *parent, int *lvl, unsigned long long *flags,
                                                         unsigned epoch0, int slot0, GridBarrier *gb,
                                                         DevCounters *ctr)
{
    const int lane = threadIdx.x & 31;
    for (int level = 0; level < kMaxLevel; ++level) {
        const int lo = ld_cg(&ctr->level_off[level]);
        int hi = ld_cg(&ctr->level_off[level + 1]);
        if (hi > cap_nodes) {
            if (threadIdx.x == 0 && blockIdx.x == 0) set_error(ctr, ERR_NODES);
            hi = cap_nodes;
        }
        const int cnt = hi - lo;
        if (cnt <= 0) {
            // no deeper nodes: the remaining level offsets all equal the node count
            if (blockIdx.x == 0 && threadIdx.x == 0) {
                for (int l = level + 2; l < kMaxLevel + 3; ++l) ctr->level_off[l] = ctr->level_off[level + 1];
                record_tree_size(ctr, cap_nodes);
            }
            return;
        }
        const int ntiles = (cnt + 31) / 32;
        const int shift = 3 * (kMaxLevel - (level + 1));
        const unsigned epoch = epoch0 + (unsigned)level;
        for (;;) {
            int tile = 0;
            if (lane == 0) tile = (int)atomicAdd(&ctr->tile_ctr[slot0 + level], 1u);
            tile = __shfl_sync(kFull, tile, 0);
            if (tile >= ntiles) break;
            const int a = lo + tile * 32 + lane;
            int st[9];
            int nch = 0;
            if (a < hi) {
                const int f = ld_cg(first + a), c = ld_cg(count + a);
                if (c > leaf && level < kMaxLevel) {
                    int base[7];
#pragma unroll
                    for (int v = 0; v < 7; ++v) base[v] = f;
                    for (int n = c; n > 1;) {
                        const int half = n >> 1;
#pragma unroll
                        for (int v = 0; v < 7; ++v) {
                            const unsigned d = (unsigned)((keys[base[v] + half] >> shift) & 7u);
                            base[v] = d < (unsigned)(v + 1) ? base[v] + half : base[v];
                        }
                        n -= half;
                    }
                    int pos[9];
                    pos[0] = f;
#pragma unroll
                    for (int v = 0; v < 7; ++v) {
                        const unsigned d = (unsigned)((keys[base[v]] >> shift) & 7u);
                        pos[v + 1] = base[v] + (d < (unsigned)(v + 1) ? 1 : 0);
                    }
                    pos[8] = f + c;
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        if (pos[v] < pos[v + 1]) st[nch++] = pos[v];
                    st[nch] = f + c;
                }
            }
            const int incl = warp_incl_scan(nch);
            const int tot = __shfl_sync(kFull, incl, 31);
            const int excl = (int)chained_exclusive_warp<4>(flags, 1, tile, (unsigned long long)tot, epoch, ctr);
            if (lane == 0 && tile == ntiles - 1) ctr->level_off[level + 2] = hi + excl + tot;
            if (a < hi) {
                const int cbase = hi + excl + incl - nch;
                child0[a] = nch ? cbase : -1;
                nchild[a] = nch;
                for (int j = 0; j < nch; ++j) {
                    const int idx = cbase + j;
                    if (idx < cap_nodes) {
                        first[idx] = st[j];
                        count[idx] = st[j + 1] - st[j];
                        parent[idx] = a;
                        lvl[idx] = level + 1;
                        child0[idx] = -1;
                        nchild[idx] = 0;
                    } else {
                        set_error(ctr, ERR_NODES);
                    }
                }
            }
        }
        if (!grid_barrier(gb, (unsigned)level, ctr)) return;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) record_tree_size(ctr, cap_nodes);
}


// ---- every level at once ----
constexpr int TB_THREADS = 256;
constexpr int TB_ROWS = 4;                               // rows of 32 positions per warp
constexpr int TB_CHUNK = 32 * TB_ROWS;                   // positions per warp (one chunk)
constexpr int TB_TILE = TB_CHUNK * (TB_THREADS / 32);    // positions per block
constexpr int TB_LEAF_MAX = 4096;                        // shared memory 3 (TB_TILE + 2 leaf) bytes
constexpr int TB_LV = kMaxLevel + 1;                     // levels 0 .. 21

// Sliding extremum over a shared byte array by doubling: on return cur[i] holds
// the min (MIN) or max of the s inputs a[i .. i + s - 1], for i <= len - s, with
// s the largest power of two <= w; the result of width w at i is then
// op(cur[i], cur[i + w - s]). a and b are both overwritten.
template <bool MIN>
__device__ __forceinline__ uint8_t *slide(uint8_t *a, uint8_t *b, int len, int w, int &s)
{
    uint8_t *cur = a, *nxt = b;
    s = 1;
    while (2 * s <= w) {
        for (int i = threadIdx.x; i <= len - 2 * s; i += blockDim.x)
            nxt[i] = MIN ? min(cur[i], cur[i + s]) : max(cur[i], cur[i + s]);
        __syncthreads();
        uint8_t *t = cur;
        cur = nxt;
        nxt = t;
        s *= 2;
    }
    return cur;
}

// Per block, TB_TILE positions: V(k) for its positions (stored), and per warp
// chunk and level the number of nodes starting in the chunk. Also clears the
// count and nchild arrays, which the node kernel assembles by additions, and
// the later stages' per-node counters (list lengths, chunk turns).
__global__ __launch_bounds__(TB_THREADS) void k_tree_windows(const uint8_t *__restrict__ div, int n, int leaf,
                                                             int cap_nodes, int *count, int *nchild,
                                                             uint8_t *__restrict__ vwin, int *__restrict__ cc,
                                                             int nchunks, int *m2l_cnt, int *p2p_cnt, int *p2p_done)
{
    extern __shared__ __align__(16) uint8_t tw_smem[];
    const int span = TB_TILE + 2 * leaf;  // div[t0 - leaf .. t0 + TB_TILE + leaf)
    uint8_t *X = tw_smem, *Y = X + span, *Z = Y + span;
    const int t0 = blockIdx.x * TB_TILE;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < cap_nodes; i += gridDim.x * blockDim.x) {
        count[i] = 0;
        nchild[i] = 0;
        m2l_cnt[i] = 0;  // the walk's per-receiver list lengths and the P2P chunk turns, for this evaluation
        p2p_cnt[i] = 0;
        p2p_done[i] = 0;
    }
    for (int i = threadIdx.x; i < span; i += blockDim.x) {
        const long long g = (long long)t0 - leaf + i;
        X[i] = (g >= 1 && g < n) ? div[g] : (uint8_t)0;  // div[0] belongs to no window
    }
    __syncthreads();
    // W(x) for x = t0 - leaf + i, i < TB_TILE + leaf: min of div[x+1 .. x+leaf] = X[i+1 .. i+leaf];
    // 0 for windows that do not lie inside [0, n)
    int s;
    uint8_t *m = slide<true>(X, Y, span, leaf, s);
    const int wl = TB_TILE + leaf;
    for (int i = threadIdx.x; i < wl; i += blockDim.x) {
        const long long x = (long long)t0 - leaf + i;
        Z[i] = (x >= 0 && x + leaf <= n - 1) ? min(m[i + 1], m[i + 1 + leaf - s]) : (uint8_t)0;
    }
    __syncthreads();
    // V(t0 + q) = max of W over x in [t0 + q - leaf, t0 + q] = Z[q .. q + leaf]
    const uint8_t *v = slide<false>(Z, m == X ? Y : X, wl, leaf + 1, s);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int c = blockIdx.x * (TB_THREADS / 32) + w;
    int cnt = 0;
    for (int r = 0; r < TB_ROWS; ++r) {
        const int q = w * TB_CHUNK + r * 32 + lane;
        const int k = t0 + q;
        int lo = TB_LV, hi = -1;
        if (k < n) {
            const int vk = max(v[q], v[q + leaf + 1 - s]);
            vwin[k] = (uint8_t)vk;
            lo = k ? div[k] : 0;
            hi = min(kMaxLevel, vk);
        }
        const bool has = lo <= hi;
        if (!__any_sync(kFull, has)) continue;
        const int lmin = (int)__reduce_min_sync(kFull, (unsigned)(has ? lo : TB_LV));
        const int lmax = (int)__reduce_max_sync(kFull, (unsigned)(has ? hi : 0));
        for (int l = lmin; l <= lmax; ++l) {
            const unsigned b = __ballot_sync(kFull, l >= lo && l <= hi);
            if (lane == l) cnt += __popc(b);
        }
    }
    if (lane < TB_LV && c < nchunks) cc[lane * nchunks + c] = cnt;
}

// Per level (one block each): exclusive scan of the chunk counts in place; the
// level's node count after the last chunk.
__global__ __launch_bounds__(1024) void k_tree_scan(int *cc, int nchunks)
{
    __shared__ int s_w[32];
    __shared__ int s_tot;
    const int l = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int *row = cc + (size_t)l * nchunks;
    int carry = 0;
    for (int base = 0; base < nchunks; base += 1024) {
        const int i = base + threadIdx.x;
        const int v = i < nchunks ? row[i] : 0;
        const int incl = warp_incl_scan(v);
        if (lane == 31) s_w[w] = incl;
        __syncthreads();
        if (w == 0) {
            const int t = s_w[lane];
            const int ti = warp_incl_scan(t);
            s_w[lane] = ti - t;
            if (lane == 31) s_tot = ti;
        }
        __syncthreads();
        if (i < nchunks) row[i] = carry + s_w[w] + incl - v;
        carry += s_tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) cc[(size_t)TB_LV * nchunks + l] = carry;
}

// Per warp chunk: the breadth-first index of every node starting in it (its
// level's offset, the chunk's offset and a ballot rank), its record, and the
// start and end terms of count and nchild. Ranks are taken per row of 32
// positions over the levels the row touches, from one below the lowest to one
// above the highest, and level L is settled once the rank of L + 1 is known.
__global__ __launch_bounds__(TB_THREADS) void k_tree_nodes(const uint8_t *__restrict__ div,
                                                           const uint8_t *__restrict__ vwin,
                                                           const int *__restrict__ cc, int nchunks, int n,
                                                           int cap_nodes, int *first, int *count, int *child0,
                                                           int *nchild, int *parent, int *lvl, DevCounters *ctr)
{
    __shared__ int s_off[TB_LV + 2];  // level offsets 0 .. 23 (22 and 23: the node count)
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int l = 0; l < TB_LV; ++l) {
            s_off[l] = acc;
            acc += cc[(size_t)TB_LV * nchunks + l];
        }
        s_off[TB_LV] = acc;
        s_off[TB_LV + 1] = acc;
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        const int total = s_off[TB_LV];
        int depth = 0;
        for (int l = 0; l < TB_LV; ++l)
            if (s_off[l + 1] > s_off[l]) depth = l;
        for (int l = 0; l < kMaxLevel + 3; ++l) ctr->level_off[l] = s_off[l];
        ctr->depth = depth;
        ctr->n_nodes = min(total, cap_nodes);
        if (total > cap_nodes) set_error(ctr, ERR_NODES);
        // the last node of each level whose run reaches position n - 1 ends at n
        const int top = min(kMaxLevel, (int)vwin[n - 1]);
        for (int L = 0; L <= top; ++L) {
            const int idx = s_off[L + 1] - 1;
            if (idx >= cap_nodes) continue;
            atomicAdd(count + idx, n);
            if (L < kMaxLevel) atomicAdd(nchild + idx, s_off[L + 2]);
        }
    }
    const int lane = threadIdx.x & 31;
    const int c = blockIdx.x * (TB_THREADS / 32) + (threadIdx.x >> 5);
    if (c >= nchunks) return;
    const unsigned lt = lanemask_lt();
    // lane l < 22: index of the next node of level l (global)
    int carry = lane < TB_LV ? s_off[lane] + cc[(size_t)lane * nchunks + c] : 0;
    for (int r = 0; r < TB_ROWS; ++r) {
        const int k = c * TB_CHUNK + r * 32 + lane;
        int lo = TB_LV, hi = -1, elo = TB_LV, ehi = -1;
        if (k < n) {
            const int d = k ? div[k] : 0;
            lo = d;
            hi = min(kMaxLevel, (int)vwin[k]);
            if (k) {
                elo = d;
                ehi = min(kMaxLevel, (int)vwin[k - 1]);
            }
        }
        const bool hs = lo <= hi, he = elo <= ehi;
        if (!__any_sync(kFull, hs || he)) continue;
        const int lmin = (int)__reduce_min_sync(kFull, (unsigned)min(hs ? lo : TB_LV, he ? elo : TB_LV));
        const int lmax = (int)__reduce_max_sync(kFull, (unsigned)max(hs ? hi : 0, he ? ehi : 0));
        int ra = 0, rb = 0;  // ranks of levels l - 2 and l - 1
        for (int l = max(lmin - 1, 0); l <= lmax + 1; ++l) {
            int rc = 0;
            if (l <= kMaxLevel) {
                const unsigned b = __ballot_sync(kFull, l >= lo && l <= hi);
                rc = __shfl_sync(kFull, carry, l) + __popc(b & lt);
                if (lane == l) carry += __popc(b);
            }
            const int L = l - 1;
            if (L >= lmin) {
                if (L >= lo && L <= hi) {  // the node of level L starting at k: index rb
                    if (rb < cap_nodes) {
                        first[rb] = k;
                        lvl[rb] = L;
                        parent[rb] = L == 0 ? -1 : (L > lo ? ra : ra - 1);
                        child0[rb] = L < hi ? rc : -1;
                        atomicAdd(count + rb, -k);
                        if (L < kMaxLevel) atomicAdd(nchild + rb, -rc);
                    }
                }
                if (L >= elo && L <= ehi) {  // the node of level L before k ends at k: index rb - 1
                    const int idx = rb - 1;
                    if (idx >= 0 && idx < cap_nodes) {
                        atomicAdd(count + idx, k);
                        if (L < kMaxLevel) atomicAdd(nchild + idx, rc);
                    }
                }
            }
            ra = rb;
            rb = rc;
        }
    }
}

}  // namespace

int launch_tree(Plan &P, cudaStream_t s)
{
    int leaf = P.leaf, cap = (int)P.cap_nodes;
    if (leaf <= TB_LEAF_MAX) {
        const int n = (int)P.n;
        const int ntiles = (n + TB_TILE - 1) / TB_TILE, nchunks = (n + TB_CHUNK - 1) / TB_CHUNK;
        k_tree_windows<<<ntiles, TB_THREADS, 3 * (TB_TILE + 2 * leaf), s>>>(P.div, n, leaf, cap, P.node_count,
                                                                            P.node_nchild, P.vwin, P.tree_cc,
                                                                            nchunks, P.m2l_cnt, P.p2p_cnt,
                                                                            P.p2p_done);
        k_tree_scan<<<TB_LV, 1024, 0, s>>>(P.tree_cc, nchunks);
        k_tree_nodes<<<ntiles, TB_THREADS, 0, s>>>(P.div, P.vwin, P.tree_cc, nchunks, n, cap, P.node_first,
                                                   P.node_count, P.node_child0, P.node_nchild, P.node_parent,
                                                   P.node_level, P.ctr);
        return 3;
    }
    // one ticket counter and one look-back epoch per level
    const int slot0 = P.slot;
    P.slot += kMaxLevel;
    const unsigned epoch0 = P.next_epoch();
    for (int l = 1; l < kMaxLevel; ++l) P.next_epoch();
    const uint64_t *keys = P.keys[0];
    GridBarrier *gb = P.gbar;
    void *args[] = {&leaf, &cap, &keys, &P.node_first, &P.node_count, &P.node_child0, &P.node_nchild,
                    &P.node_parent, &P.node_level, &P.flags, (void *)&epoch0, (void *)&slot0, &gb, &P.ctr};
    cudaLaunchCooperativeKernel((const void *)k_tree_all, dim3(P.coop_blocks_tree), dim3(TR_THREADS), args, 0, s);
    // the later stages' per-node counters (the window build clears them itself)
    cudaMemsetAsync(P.m2l_cnt, 0, (size_t)P.cap_nodes * sizeof(int), s);
    cudaMemsetAsync(P.p2p_cnt, 0, (size_t)P.cap_nodes * sizeof(int), s);
    cudaMemsetAsync(P.p2p_done, 0, (size_t)P.cap_nodes * sizeof(int), s);
    return 1;
}

size_t tree_cc_ints(int64_t n) { return (size_t)TB_LV * (size_t)((n + TB_CHUNK - 1) / TB_CHUNK + 1); }

int tree_max_blocks_per_sm()
{
    int b = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_tree_all, TR_THREADS, 0);
    return b;
}

}  // namespace bfm
