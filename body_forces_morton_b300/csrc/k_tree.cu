// Octree over the sorted Morton keys, one kernel per level.
//
// JZ-FMM page, "Why this works well on GPUs": the tree stores child nodes next
// to each other. A node of level l holding more than `leaf` particles splits
// into its non-empty octants at level l+1 (at most 21 levels). Nodes are
// numbered breadth first: level by level, within a level in key order, so the
// children of one node are contiguous and follow the children of the nodes
// before it.
//
// Per level: a warp finds the child starts of one node (they are the sorted
// positions where the key's digit of level l+1 changes), a block scans the
// child counts of its tile of 32 nodes, and a decoupled look-back over the
// tiles gives each tile its first child index.
#include "plan.h"

namespace bfm {

namespace {

constexpr int TR_THREADS = 256;
constexpr int TR_TILE = 32;                         // nodes per tile
constexpr int TR_PER_WARP = TR_TILE / (TR_THREADS / 32);
constexpr int TR_SCAN_LIMIT = 512;                  // nodes up to this size scan the divergence bytes

__global__ __launch_bounds__(TR_THREADS) void k_tree_level(int level, int leaf, int cap_nodes,
                                                           const uint64_t *__restrict__ keys,
                                                           const uint8_t *__restrict__ div, int *first, int *count,
                                                           int *child0, int *nchild, int *parent, int *lvl,
                                                           unsigned long long *flags, unsigned epoch, int slot,
                                                           DevCounters *ctr)
{
    __shared__ int s_tile;
    __shared__ int s_nch[TR_TILE];
    __shared__ int s_excl[TR_TILE];
    __shared__ int s_start[TR_TILE][9];
    __shared__ int s_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int lo = ctr->level_off[level];
    int hi = ctr->level_off[level + 1];
    if (hi > cap_nodes) {
        if (tid == 0 && blockIdx.x == 0) set_error(ctr, ERR_NODES);
        hi = cap_nodes;
    }
    const int cnt = hi - lo;
    if (cnt <= 0) {
        if (blockIdx.x == 0 && tid == 0) ctr->level_off[level + 2] = ctr->level_off[level + 1];
        return;
    }
    const int ntiles = (cnt + TR_TILE - 1) / TR_TILE;
    const int shift = 3 * (kMaxLevel - (level + 1));
    for (;;) {
        if (tid == 0) s_tile = (int)atomicAdd(&ctr->tile_ctr[slot], 1u);
        __syncthreads();
        const int tile = s_tile;
        if (tile >= ntiles) break;
        for (int q = 0; q < TR_PER_WARP; ++q) {
            const int ln = warp * TR_PER_WARP + q;
            const int a = lo + tile * TR_TILE + ln;
            int nch = 0;
            if (a < hi) {
                const int f = first[a], c = count[a];
                if (c > leaf && level < kMaxLevel) {
                    if (c <= TR_SCAN_LIMIT) {
                        // child starts: f and every i in (f, f+c) where the keys diverge at level+1
                        if (lane == 0) s_start[ln][0] = f;
                        int found = 1;
                        for (int base = f + 1; base < f + c; base += 32) {
                            const int i = base + lane;
                            const bool hit = i < f + c && div[i] == (uint8_t)(level + 1);
                            const unsigned m = __ballot_sync(kFull, hit);
                            if (hit) {
                                const int r = found + __popc(m & lanemask_lt());
                                if (r < 8) s_start[ln][r] = i;
                            }
                            found += __popc(m);
                        }
                        nch = found < 8 ? found : 8;
                        if (lane == 0) s_start[ln][nch] = f + c;
                    } else {
                        // lane v < 8: first position whose digit is >= v (digits ascend within the node)
                        int pos = f;
                        if (lane >= 1 && lane < 8) {
                            int l2 = f, h2 = f + c;
                            while (l2 < h2) {
                                const int mid = l2 + ((h2 - l2) >> 1);
                                if ((int)((keys[mid] >> shift) & 7u) < lane) l2 = mid + 1;
                                else h2 = mid;
                            }
                            pos = l2;
                        }
                        int nextpos = __shfl_down_sync(kFull, pos, 1);
                        if (lane == 7) nextpos = f + c;
                        const bool nonempty = lane < 8 && pos < nextpos;
                        const unsigned m = __ballot_sync(kFull, nonempty);
                        if (nonempty) s_start[ln][__popc(m & lanemask_lt())] = pos;
                        nch = __popc(m);
                        if (lane == 0) s_start[ln][nch] = f + c;
                    }
                }
            }
            if (lane == 0) s_nch[ln] = nch;
        }
        __syncthreads();
        if (warp == 0) {
            const int v = s_nch[lane];
            const int incl = warp_incl_scan(v);
            s_excl[lane] = incl - v;
            const int tot = __shfl_sync(kFull, incl, 31);
            if (lane == 0) {
                const int excl = (int)chained_exclusive(flags, 1, tile, (unsigned long long)tot, epoch, ctr);
                s_base = hi + excl;
                if (tile == ntiles - 1) ctr->level_off[level + 2] = hi + excl + tot;
            }
        }
        __syncthreads();
        {
            const int ln = tid >> 3, c = tid & 7;
            const int a = lo + tile * TR_TILE + ln;
            if (a < hi) {
                const int nch = s_nch[ln];
                const int cbase = s_base + s_excl[ln];
                if (c == 0) {
                    child0[a] = nch ? cbase : -1;
                    nchild[a] = nch;
                }
                if (c < nch) {
                    const int idx = cbase + c;
                    if (idx < cap_nodes) {
                        first[idx] = s_start[ln][c];
                        count[idx] = s_start[ln][c + 1] - s_start[ln][c];
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
        __syncthreads();
    }
}

}  // namespace

int launch_tree(Plan &P, cudaStream_t s)
{
    int launches = 0;
    for (int level = 0; level < kMaxLevel; ++level) {
        const int slot = P.next_slot();
        const unsigned ep = P.next_epoch();
        k_tree_level<<<P.num_sms * 4, TR_THREADS, 0, s>>>(level, P.leaf, (int)P.cap_nodes, P.keys[0], P.div,
                                                         P.node_first, P.node_count, P.node_child0, P.node_nchild,
                                                         P.node_parent, P.node_level, P.flags, ep, slot, P.ctr);
        ++launches;
    }
    return launches;
}

}  // namespace bfm
