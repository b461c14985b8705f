// Octree over the sorted Morton keys, one kernel per level.
//
// JZ-FMM page, "Why this works well on GPUs": the tree stores child nodes next
// to each other. A node of level l holding more than `leaf` particles splits
// into its non-empty octants at level l+1 (at most 21 levels). Nodes are
// numbered breadth first: level by level, within a level in key order, so the
// children of one node are contiguous and follow the children of the nodes
// before it.
//
// Per level: every node's child starts (the sorted positions where the key's
// digit of level l+1 changes) come from binary searches on the keys; a warp
// scan of the child counts of a tile of 32 nodes and a decoupled look-back
// over the tiles give each child its breadth-first index.
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

}  // namespace

int launch_tree(Plan &P, cudaStream_t s)
{
    // one ticket counter and one look-back epoch per level
    const int slot0 = P.slot;
    P.slot += kMaxLevel;
    const unsigned epoch0 = P.next_epoch();
    for (int l = 1; l < kMaxLevel; ++l) P.next_epoch();
    int leaf = P.leaf, cap = (int)P.cap_nodes;
    const uint64_t *keys = P.keys[0];
    GridBarrier *gb = P.gbar;
    void *args[] = {&leaf, &cap, &keys, &P.node_first, &P.node_count, &P.node_child0, &P.node_nchild,
                    &P.node_parent, &P.node_level, &P.flags, (void *)&epoch0, (void *)&slot0, &gb, &P.ctr};
    cudaLaunchCooperativeKernel((const void *)k_tree_all, dim3(P.coop_blocks_tree), dim3(TR_THREADS), args, 0, s);
    return 1;
}

int tree_max_blocks_per_sm()
{
    int b = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_tree_all, TR_THREADS, 0);
    return b;
}

}  // namespace bfm
