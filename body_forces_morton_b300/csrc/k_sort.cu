// Root box, Morton keys and the stable LSD radix sort of (key, index) pairs.
//
// JZ-FMM page, "Why this works well on GPUs": particles are sorted so that
// neighbours sit next to each other; sorting and tree construction stay on the
// GPU. Keys interleave 21 bits per axis of the root cube (x highest within each
// 3-bit digit); the quantisation q = min(floor(((x - lo) / side) * 2^21), 2^21 - 1)
// is evaluated step by step in the plan's precision without contraction, so the
// keys are exactly those of any other implementation doing the same steps.
//
// Radix sort of (key, index) pairs: 4 passes of 8 bits over the high word
// (bits 32..63), then each run of keys with equal high words sorted by its low
// word and index (k_sort_groups, k_sort_runs): the same order
// as sorting the whole key, since the passes are stable. At 2^20 clustered
// keys the runs number about 9e4 and hold at most a dozen keys; strongly
// clustered states (collapsed halo cores) put a large share of the keys into
// long runs, and after such an evaluation the plan sorts all 8 digits instead.
// A pass ranks a 4096-key tile's keys per digit with warp match_any (stable
// within the tile), reorders the tile by digit in shared memory and writes it
// out in runs of consecutive positions (one digit's keys of a tile are
// contiguous in the output). When every tile fits on the GPU at once, the
// passes run in one cooperative launch, the offsets from a scan of the tiles'
// counts between grid barriers (k_radix_coop); otherwise each pass is one
// kernel that takes tiles from a ticket counter and finds the offsets with a
// decoupled look-back over the earlier tiles. A last kernel gathers
// (x, y, z, m) into sorted order.
#include "plan.h"

namespace bfm {

namespace {

constexpr int kBoxThreads = 256;
constexpr int RS_THREADS = 256;
constexpr int RS_WARPS = RS_THREADS / 32;
// keys per thread: 16 (4096-key tiles) from N = 2^19 on, 8 (2048-key tiles, twice the
// blocks) below, where the sort has too few tiles to fill the GPU (both measured)
constexpr int RS_ITEMS_LARGE = 16, RS_ITEMS_SMALL = 8;
// The radix passes sort by the high word (digits 4..7, bits 32..63); runs of
// keys with equal high words are then sorted by their low words: up to
// kGroupMax keys by one thread, up to kWarpRun by a warp in registers, longer
// runs by a block (in shared memory up to kBigSmem keys, else four stable
// passes over the low word). When the previous evaluation found more than
// N / kLongRunsDiv keys in runs longer than kGroupMax (strongly clustered or
// coincident particles), all 8 digits are sorted instead and the runs need no
// second step.
constexpr int kSortHighPass0 = 4;
constexpr int kGroupMax = 32;
constexpr int kWarpRun = 512;
constexpr int kBigSmem = 4096;
constexpr int kLongRunsDiv = 64;

__device__ __forceinline__ uint64_t spread3(uint32_t v)
{
    uint64_t x = v & 0x1fffffu;
    x = (x | (x << 32)) & 0x1f00000000ffffull;
    x = (x | (x << 16)) & 0x1f0000ff0000ffull;
    x = (x | (x << 8)) & 0x100f00f00f00f00full;
    x = (x | (x << 4)) & 0x10c30c30c30c30c3ull;
    x = (x | (x << 2)) & 0x1249249249249249ull;
    return x;
}

template <class T> __device__ __forceinline__ bool finite_t(T v) { return isfinite(v); }
template <class T> __device__ __forceinline__ T tmin(T a, T b) { return b < a ? b : a; }
template <class T> __device__ __forceinline__ T tmax(T a, T b) { return b > a ? b : a; }

// Root box: per-block min/max, the last block to finish reduces the partials.
template <class T>
__global__ __launch_bounds__(kBoxThreads) void k_bbox(const T *__restrict__ pos, int n, T *__restrict__ partial,
                                                      DevCounters *ctr)
{
    T lo[3], hi[3];
    for (int a = 0; a < 3; ++a) { lo[a] = pos_inf<T>(); hi[a] = -pos_inf<T>(); }
    bool bad = false;
    // four positions a stride apart per thread and loop iteration, their loads issued together
    const int stride = gridDim.x * blockDim.x;
    for (int i0 = blockIdx.x * blockDim.x + threadIdx.x; i0 < n; i0 += 4 * stride) {
        T v[4][3];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * stride;
#pragma unroll
            for (int a = 0; a < 3; ++a) v[u][a] = i < n ? pos[3 * (int64_t)i + a] : pos[a];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int a = 0; a < 3; ++a) {
                bad |= !finite_t(v[u][a]);
                lo[a] = tmin(lo[a], v[u][a]);
                hi[a] = tmax(hi[a], v[u][a]);
            }
    }
    if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0) set_error(ctr, ERR_NONFINITE);
    for (int o = 16; o > 0; o >>= 1)
        for (int a = 0; a < 3; ++a) {
            lo[a] = tmin(lo[a], __shfl_xor_sync(kFull, lo[a], o));
            hi[a] = tmax(hi[a], __shfl_xor_sync(kFull, hi[a], o));
        }
    __shared__ T s[kBoxThreads / 32][6];
    __shared__ bool s_last;
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0)
        for (int a = 0; a < 3; ++a) { s[w][a] = lo[a]; s[w][3 + a] = hi[a]; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < kBoxThreads / 32; ++k)
            for (int a = 0; a < 3; ++a) {
                s[0][a] = tmin(s[0][a], s[k][a]);
                s[0][3 + a] = tmax(s[0][3 + a], s[k][3 + a]);
            }
        for (int a = 0; a < 6; ++a) partial[6 * blockIdx.x + a] = s[0][a];
        __threadfence();
        s_last = atomicAdd(&ctr->bbox_done, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    // last block: reduce the per-block partials with all its threads
    __threadfence();
    for (int a = 0; a < 3; ++a) { lo[a] = pos_inf<T>(); hi[a] = -pos_inf<T>(); }
    for (int b = threadIdx.x; b < (int)gridDim.x; b += blockDim.x)
        for (int a = 0; a < 3; ++a) {
            lo[a] = tmin(lo[a], ld_cg(partial + 6 * b + a));
            hi[a] = tmax(hi[a], ld_cg(partial + 6 * b + 3 + a));
        }
    for (int o = 16; o > 0; o >>= 1)
        for (int a = 0; a < 3; ++a) {
            lo[a] = tmin(lo[a], __shfl_xor_sync(kFull, lo[a], o));
            hi[a] = tmax(hi[a], __shfl_xor_sync(kFull, hi[a], o));
        }
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        for (int a = 0; a < 3; ++a) { s[w][a] = lo[a]; s[w][3 + a] = hi[a]; }
    __syncthreads();
    if (threadIdx.x != 0) return;
    T r[6];
    for (int a = 0; a < 6; ++a) r[a] = s[0][a];
    for (int k = 1; k < kBoxThreads / 32; ++k)
        for (int a = 0; a < 3; ++a) {
            r[a] = tmin(r[a], s[k][a]);
            r[3 + a] = tmax(r[3 + a], s[k][3 + a]);
        }
    T side = sub_rn(r[3], r[0]);
    for (int a = 1; a < 3; ++a) {
        T e = sub_rn(r[3 + a], r[a]);
        if (e > side) side = e;
    }
    if (!(side > T(0))) side = T(1);
    for (int a = 0; a < 3; ++a) ctr->box[a] = (double)r[a];
    ctr->box[3] = (double)side;
}

template <class T> __device__ __forceinline__ uint32_t quantise(T x, T lo, T side)
{
    T u = mul_rn(div_rn(sub_rn(x, lo), side), T(2097152.0));
    T f = floor(u);
    uint32_t q = (uint32_t)f;
    return q > 2097151u ? 2097151u : q;
}

// Keys in the caller's order plus the digit histograms of the radix passes
// (the digits of the high word).
template <class T>
__global__ __launch_bounds__(1024) void k_keys(const T *__restrict__ pos, int n, uint64_t *__restrict__ keys,
                                               int p0, DevCounters *ctr)
{
    __shared__ unsigned h[8][256];
    for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) (&h[0][0])[i] = 0;
    __syncthreads();
    const T lo0 = (T)ctr->box[0], lo1 = (T)ctr->box[1], lo2 = (T)ctr->box[2], side = (T)ctr->box[3];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const T *q = pos + 3 * (int64_t)i;
        uint64_t k = (spread3(quantise(q[0], lo0, side)) << 2) | (spread3(quantise(q[1], lo1, side)) << 1) |
                     spread3(quantise(q[2], lo2, side));
        keys[i] = k;
#pragma unroll
        for (int r = 0; r < 8; ++r)
            if (r >= p0) atomicAdd(&h[r][(k >> (8 * r)) & 255u], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 8 * 256; i += blockDim.x) {
        unsigned v = (&h[0][0])[i];
        if (v) atomicAdd(&ctr->hist[0][0] + i, v);
    }
}

template <bool FIRST, int RS_ITEMS>
__global__ __launch_bounds__(RS_THREADS) void k_radix_pass(const uint64_t *__restrict__ kin,
                                                           const uint32_t *__restrict__ vin,
                                                           uint64_t *__restrict__ kout, uint32_t *__restrict__ vout,
                                                           int n, int pass, unsigned long long *flags, unsigned epoch,
                                                           int slot, DevCounters *ctr)
{
    constexpr int TILE = RS_THREADS * RS_ITEMS;
    extern __shared__ __align__(16) unsigned char rs_smem[];
    uint64_t *const s_k = reinterpret_cast<uint64_t *>(rs_smem);   // the tile in digit order
    uint32_t *const s_v = reinterpret_cast<uint32_t *>(s_k + TILE);
    __shared__ unsigned s_hist[RS_WARPS][256];
    __shared__ unsigned s_lstart[256];  // tile-local start of each digit
    __shared__ unsigned s_base[256];    // global position of the tile's first key of each digit, minus s_lstart
    __shared__ unsigned s_wsum[2][RS_WARPS];
    __shared__ int s_tile;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < RS_WARPS * 256; i += RS_THREADS) (&s_hist[0][0])[i] = 0;
    if (tid == 0) s_tile = (int)atomicAdd(&ctr->tile_ctr[slot], 1u);
    __syncthreads();
    const int tile = s_tile;
    const int shift = 8 * pass;
    const int64_t start = (int64_t)tile * TILE + warp * (32 * RS_ITEMS);
    uint64_t k[RS_ITEMS];
    uint32_t v[RS_ITEMS];
    unsigned rank[RS_ITEMS];
#pragma unroll
    for (int j = 0; j < RS_ITEMS; ++j) {
        int64_t i = start + j * 32 + lane;
        bool valid = i < n;
        k[j] = valid ? kin[i] : ~0ull;
        v[j] = valid ? (FIRST ? (uint32_t)i : vin[i]) : 0u;
    }
#pragma unroll
    for (int j = 0; j < RS_ITEMS; ++j) {
        const bool valid = start + j * 32 + lane < n;
        const unsigned d = valid ? (unsigned)((k[j] >> shift) & 255u) : 256u;
        const unsigned peers = __match_any_sync(kFull, d);
        const int leader = __ffs(peers) - 1;
        unsigned mine = (lane == leader && valid) ? s_hist[warp][d] : 0u;
        const unsigned b = __shfl_sync(kFull, mine, leader);
        rank[j] = b + __popc(peers & lanemask_lt());
        __syncwarp();
        if (lane == leader && valid) s_hist[warp][d] = b + __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // per digit: warp offsets within the tile, tile total, look-back, and two exclusive scans over the
    // digits (the pass's global histogram: where the digit starts in the output; the tile's counts:
    // where it starts in the tile)
    {
        const int d = tid;
        unsigned tot = 0;
#pragma unroll
        for (int w = 0; w < RS_WARPS; ++w) {
            unsigned c = s_hist[w][d];
            s_hist[w][d] = tot;
            tot += c;
        }
        unsigned long long excl = chained_exclusive_wide<8>(flags + d, 256, tile, tot, epoch, ctr);
        const unsigned g = ctr->hist[pass][d];
        unsigned incl = g, inct = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned t = __shfl_up_sync(kFull, incl, o);
            const unsigned u = __shfl_up_sync(kFull, inct, o);
            if (lane >= o) {
                incl += t;
                inct += u;
            }
        }
        if (lane == 31) {
            s_wsum[0][warp] = incl;
            s_wsum[1][warp] = inct;
        }
        __syncthreads();
        unsigned wbase = 0, wbase_t = 0;
        for (int w = 0; w < warp; ++w) {
            wbase += s_wsum[0][w];
            wbase_t += s_wsum[1][w];
        }
        const unsigned lstart = wbase_t + inct - tot;
        s_lstart[d] = lstart;
        s_base[d] = wbase + incl - g + (unsigned)excl - lstart;  // unsigned: the difference wraps back
    }
    __syncthreads();
    // the tile into shared memory in digit order (stable: warps, then items, then lanes in input order)
#pragma unroll
    for (int j = 0; j < RS_ITEMS; ++j) {
        if (start + j * 32 + lane < n) {
            const unsigned d = (unsigned)((k[j] >> shift) & 255u);
            const unsigned local = s_lstart[d] + s_hist[warp][d] + rank[j];
            s_k[local] = k[j];
            s_v[local] = v[j];
        }
    }
    __syncthreads();
    // and out: consecutive keys of one digit go to consecutive positions
    const int64_t left = (int64_t)n - (int64_t)tile * TILE;
    const int tile_n = left < TILE ? (int)left : TILE;
    for (int i = tid; i < tile_n; i += RS_THREADS) {
        const uint64_t key = s_k[i];
        const uint32_t val = s_v[i];
        const unsigned d = (unsigned)((key >> shift) & 255u);
        const unsigned out = s_base[d] + (unsigned)i;
        if (out < (unsigned)n) {
            kout[out] = key;
            vout[out] = val;
        } else {
            set_error(ctr, ERR_BOUNDS);
        }
    }
}

// All radix passes in one cooperative launch, one tile of RS_THREADS * ITEMS keys
// per block with every tile resident (N up to the co-resident tiles). Per
// pass: each tile ranks its keys per digit as k_radix_pass does, publishes its
// 256 digit counts and reorders itself by digit in shared memory; after a grid
// barrier the warps scan each digit's counts over the tiles (a column per
// warp, in place, into exclusive offsets); after a second barrier each tile
// writes its runs to the pass's global digit start plus its offset; a third
// barrier ends the pass. Three barriers replace the look-back chain, which
// with every tile starting at once runs through the tiles one after another.
template <int ITEMS>
__global__ __launch_bounds__(RS_THREADS) void k_radix_coop(uint64_t *k0, uint32_t *v0, uint64_t *k1, uint32_t *v1,
                                                           int n, int p0, unsigned *cnt, GridBarrier *gb,
                                                           DevCounters *ctr)
{
    constexpr int TILE = RS_THREADS * ITEMS;
    extern __shared__ __align__(16) unsigned char rs_smem[];
    uint64_t *const s_k = reinterpret_cast<uint64_t *>(rs_smem);
    uint32_t *const s_v = reinterpret_cast<uint32_t *>(s_k + TILE);
    __shared__ unsigned s_hist[RS_WARPS][256];
    __shared__ unsigned s_lstart[256];
    __shared__ unsigned s_base[256];
    __shared__ unsigned s_wsum[2][RS_WARPS];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x, ntiles = gridDim.x;
    const int64_t start = (int64_t)tile * TILE + warp * (32 * ITEMS);
    const int64_t left = (int64_t)n - (int64_t)tile * TILE;
    const int tile_n = left < TILE ? (int)left : TILE;
    unsigned bar = 0;
    for (int pass = p0; pass < 8; ++pass) {
        const uint64_t *kin = (pass & 1) ? k1 : k0;
        const uint32_t *vin = (pass & 1) ? v1 : v0;
        uint64_t *kout = (pass & 1) ? k0 : k1;
        uint32_t *vout = (pass & 1) ? v0 : v1;
        const int shift = 8 * pass;
        for (int i = tid; i < RS_WARPS * 256; i += RS_THREADS) (&s_hist[0][0])[i] = 0;
        __syncthreads();
        uint64_t k[ITEMS];
        uint32_t v[ITEMS];
        unsigned rank[ITEMS];
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const int64_t i = start + j * 32 + lane;
            const bool valid = i < n;
            k[j] = valid ? ld_cg(kin + i) : ~0ull;  // written by other blocks in the previous pass
            v[j] = valid ? (pass == p0 ? (uint32_t)i : ld_cg(vin + i)) : 0u;
        }
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            const bool valid = start + j * 32 + lane < n;
            const unsigned d = valid ? (unsigned)((k[j] >> shift) & 255u) : 256u;
            const unsigned peers = __match_any_sync(kFull, d);
            const int leader = __ffs(peers) - 1;
            unsigned mine = (lane == leader && valid) ? s_hist[warp][d] : 0u;
            const unsigned b = __shfl_sync(kFull, mine, leader);
            rank[j] = b + __popc(peers & lanemask_lt());
            __syncwarp();
            if (lane == leader && valid) s_hist[warp][d] = b + __popc(peers);
            __syncwarp();
        }
        __syncthreads();
        // per digit d: warp offsets within the tile, the tile's count (published), the tile-local start
        // and the pass's global start (from the key kernel's histogram)
        const int d = tid;
        unsigned tot = 0;
#pragma unroll
        for (int w = 0; w < RS_WARPS; ++w) {
            const unsigned c = s_hist[w][d];
            s_hist[w][d] = tot;
            tot += c;
        }
        cnt[(size_t)tile * 256 + d] = tot;
        unsigned gpart;
        {
            const unsigned g = ctr->hist[pass][d];
            unsigned incl = g, inct = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned t = __shfl_up_sync(kFull, incl, o);
                const unsigned u = __shfl_up_sync(kFull, inct, o);
                if (lane >= o) {
                    incl += t;
                    inct += u;
                }
            }
            if (lane == 31) {
                s_wsum[0][warp] = incl;
                s_wsum[1][warp] = inct;
            }
            __syncthreads();
            unsigned wbase = 0, wbase_t = 0;
            for (int w = 0; w < warp; ++w) {
                wbase += s_wsum[0][w];
                wbase_t += s_wsum[1][w];
            }
            const unsigned lstart = wbase_t + inct - tot;
            s_lstart[d] = lstart;
            gpart = wbase + incl - g - lstart;  // unsigned: wraps back once the tile offset is added
        }
        __syncthreads();
        // the tile into shared memory in digit order (stable: warps, then items, then lanes)
#pragma unroll
        for (int j = 0; j < ITEMS; ++j) {
            if (start + j * 32 + lane < n) {
                const unsigned dj = (unsigned)((k[j] >> shift) & 255u);
                const unsigned local = s_lstart[dj] + s_hist[warp][dj] + rank[j];
                s_k[local] = k[j];
                s_v[local] = v[j];
            }
        }
        if (!grid_barrier(gb, bar++, ctr)) return;
        // each digit's counts over the tiles into exclusive offsets, a column per warp (lanes over
        // tiles), so that small grids need no block barriers for it; columns go to the blocks in turn,
        // then to their warps, which spreads the column loads over the SMs
        for (int dd = blockIdx.x + ntiles * warp; dd < 256; dd += ntiles * RS_WARPS) {
            unsigned carry = 0;
            for (int t0 = 0; t0 < ntiles; t0 += 32 * 8) {
                unsigned c[8];  // eight chunks of 32 tiles loaded at once
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = t0 + 32 * u + lane;
                    c[u] = t < ntiles ? ld_cg(cnt + (size_t)t * 256 + dd) : 0u;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = t0 + 32 * u + lane;
                    const unsigned incl = (unsigned)warp_incl_scan((int)c[u]);
                    if (t < ntiles) cnt[(size_t)t * 256 + dd] = carry + incl - c[u];
                    carry += __shfl_sync(kFull, incl, 31);
                }
            }
        }
        if (!grid_barrier(gb, bar++, ctr)) return;
        s_base[d] = gpart + ld_cg(cnt + (size_t)tile * 256 + d);
        __syncthreads();
        for (int i = tid; i < tile_n; i += RS_THREADS) {
            const uint64_t key = s_k[i];
            const unsigned dk = (unsigned)((key >> shift) & 255u);
            const unsigned out = s_base[dk] + (unsigned)i;
            if (out < (unsigned)n) {
                kout[out] = key;
                vout[out] = s_v[i];
            } else {
                set_error(ctr, ERR_BOUNDS);
            }
        }
        if (pass < 7 && !grid_barrier(gb, bar++, ctr)) return;
    }
}

// After the sort: the sorted particles (x, y, z, m) gathered through the
// permutation, the divergence levels of consecutive sorted keys (the first tree
// level at which keys[i-1] and keys[i] fall in different cells, 22 when equal)
// and the root node.
template <class T>
__global__ void k_gather_diverge(const uint64_t *__restrict__ keys, const uint32_t *__restrict__ perm, int n,
                                 const T *__restrict__ pos, const T *__restrict__ mass, vec4<T> *__restrict__ xyzm,
                                 uint8_t *__restrict__ div, int *first, int *count, int *child0, int *nchild,
                                 int *parent, int *level, DevCounters *ctr)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const uint32_t o = perm[i];
        if (o < (uint32_t)n) {
            const T *q = pos + 3 * (int64_t)o;
            xyzm[i] = make4<T>(q[0], q[1], q[2], mass[o]);
        } else {
            set_error(ctr, ERR_BOUNDS);
        }
        if (i == 0) {
            div[0] = 0;
            first[0] = 0; count[0] = n; child0[0] = -1; nchild[0] = 0; parent[0] = -1; level[0] = 0;
            ctr->level_off[0] = 0;
            ctr->level_off[1] = 1;
        } else {
            const uint64_t x = keys[i - 1] ^ keys[i];
            div[i] = x ? (uint8_t)(21 - (63 - __clzll((long long)x)) / 3) : (uint8_t)22;
        }
    }
}

// Runs of equal high words after the radix passes are in index order; each is
// sorted by (key, index). The thread at a run's head sorts a run of up to
// kGroupMax keys in place (insertion sort, stable, so equal keys keep their
// index order); for a longer run it finds the run's end (galloping over the
// high words, which ascend) and lists (start, length) for the warp and block
// kernel, adding its length to the long-run key count. A run's writes permute
// keys that share one high word, so the neighbours' run tests are unaffected.
// One comparator of a sorting network on (key, index) pairs: the lower pair to a.
__device__ __forceinline__ void ce_key_idx(uint64_t &ka, uint32_t &va, uint64_t &kb, uint32_t &vb)
{
    const bool sw = kb < ka || (kb == ka && vb < va);
    const uint64_t k0 = sw ? kb : ka, k1 = sw ? ka : kb;
    const uint32_t v0 = sw ? vb : va, v1 = sw ? va : vb;
    ka = k0;
    kb = k1;
    va = v0;
    vb = v1;
}

__global__ __launch_bounds__(256) void k_sort_groups(uint64_t *keys, uint32_t *idx, int n, int2 *big, int cap_big,
                                                     DevCounters *ctr)
{
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        // the key, its neighbours, and for the head of a run the next six keys and eight indices, each
        // group loaded at once
        const uint64_t kc = keys[i];
        const uint64_t kp = i > 0 ? keys[i - 1] : 0;
        const uint64_t kn = i + 1 < n ? keys[i + 1] : 0;
        const uint32_t hi = (uint32_t)(kc >> 32);
        if (i > 0 && (uint32_t)(kp >> 32) == hi) continue;       // not the head of a run
        if (i + 1 >= n || (uint32_t)(kn >> 32) != hi) continue;  // a run of one
        {
            uint64_t k[8];
            uint32_t v[8];
            k[0] = kc;
            k[1] = kn;
#pragma unroll
            for (int j = 2; j < 8; ++j) k[j] = i + j < n ? keys[i + j] : ~0ull;
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = i + j < n ? idx[i + j] : ~0u;
            int len = 2;
#pragma unroll
            for (int j = 2; j < 8; ++j) len += (len == j && (uint32_t)(k[j] >> 32) == hi) ? 1 : 0;
            if (len < 8 || i + 8 >= n || (uint32_t)(keys[i + 8] >> 32) != hi) {
                // a run of at most 8: Batcher's odd-even merge network in registers, padded with pairs
                // above every key (keys have 63 bits); the (key, index) order is the stable order by key,
                // since the passes before left each run in index order
#pragma unroll
                for (int j = 2; j < 8; ++j)
                    if (j >= len) {
                        k[j] = ~0ull;
                        v[j] = ~0u;
                    }
                constexpr int net[19][2] = {{0, 1}, {2, 3}, {4, 5}, {6, 7}, {0, 2}, {1, 3}, {4, 6},
                                            {5, 7}, {1, 2}, {5, 6}, {0, 4}, {1, 5}, {2, 6}, {3, 7},
                                            {2, 4}, {3, 5}, {1, 2}, {3, 4}, {5, 6}};
#pragma unroll
                for (int c = 0; c < 19; ++c) ce_key_idx(k[net[c][0]], v[net[c][0]], k[net[c][1]], v[net[c][1]]);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < len) {
                        keys[i + j] = k[j];
                        idx[i + j] = v[j];
                    }
                continue;
            }
        }
        int len = 9;
        while (len <= kGroupMax && i + len < n && (uint32_t)(keys[i + len] >> 32) == hi) ++len;
        if (len > kGroupMax) {
            int a = i + kGroupMax, span = kGroupMax;  // keys[a] is in the run
            while (a + span < n && (uint32_t)(keys[a + span] >> 32) == hi) {
                a += span;
                span *= 2;
            }
            int b = min(n, a + span);  // the run ends in (a, b]
            while (b - a > 1) {
                const int m = a + (b - a) / 2;
                if ((uint32_t)(keys[m] >> 32) == hi) a = m;
                else b = m;
            }
            len = b - i;
            const int slot = atomicAdd(&ctr->n_sort_groups, 1);
            if (slot < cap_big) big[slot] = make_int2(i, len);
            else set_error(ctr, ERR_BOUNDS);
            atomicAdd(&ctr->sort_long_keys, len);
            continue;
        }
        uint64_t k[kGroupMax];
        uint32_t v[kGroupMax];
        for (int j = 0; j < len; ++j) {
            k[j] = keys[i + j];
            v[j] = idx[i + j];
        }
        for (int j = 1; j < len; ++j) {
            const uint64_t kj = k[j];
            const uint32_t vj = v[j];
            int m = j - 1;
            while (m >= 0 && k[m] > kj) {
                k[m + 1] = k[m];
                v[m + 1] = v[m];
                --m;
            }
            k[m + 1] = kj;
            v[m + 1] = vj;
        }
        for (int j = 0; j < len; ++j) {
            keys[i + j] = k[j];
            idx[i + j] = v[j];
        }
    }
}

// Warp-wide ascending bitonic sort of 32 NR unsigned 64-bit values in the
// blocked layout (value e = NR lane + j in v[j]): the network of the lists'
// warp sort, on the composites (low key word << 32 | index) of one run.
template <int NR>
__device__ __forceinline__ void warp_sort_u64(uint64_t (&v)[NR])
{
    constexpr int N = 32 * NR;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= N; k <<= 1) {
        if (k <= NR) {
#pragma unroll
            for (int j = 0; j < NR; ++j) {
                const int pj = j ^ (k - 1);
                if ((j & (k >> 1)) == 0) {
                    const uint64_t a = v[j], b = v[pj];
                    v[j] = a < b ? a : b;
                    v[pj] = a < b ? b : a;
                }
            }
        } else {
            const int m = k / NR - 1;
            const bool lower = (lane & ((k >> 1) / NR)) == 0;
#pragma unroll
            for (int j = 0; j < NR / 2; ++j) {
                const uint64_t oa = __shfl_xor_sync(kFull, v[NR - 1 - j], m);
                const uint64_t ob = __shfl_xor_sync(kFull, v[j], m);
                const uint64_t a = v[j], b = v[NR - 1 - j];
                v[j] = lower ? (a < oa ? a : oa) : (a < oa ? oa : a);
                v[NR - 1 - j] = lower ? (b < ob ? b : ob) : (b < ob ? ob : b);
            }
        }
#pragma unroll
        for (int d = k >> 2; d >= 1; d >>= 1) {
            if (d < NR) {
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    if ((j & d) == 0) {
                        const uint64_t a = v[j], b = v[j | d];
                        v[j] = a < b ? a : b;
                        v[j | d] = a < b ? b : a;
                    }
                }
            } else {
                const int m = d / NR;
                const bool lower = (lane & m) == 0;
#pragma unroll
                for (int j = 0; j < NR; ++j) {
                    const uint64_t o = __shfl_xor_sync(kFull, v[j], m);
                    v[j] = lower ? (v[j] < o ? v[j] : o) : (v[j] < o ? o : v[j]);
                }
            }
        }
    }
}

template <int NR>
__device__ __forceinline__ void sort_run_warp(uint64_t *keys, uint32_t *idx, int s, int len)
{
    const int lane = threadIdx.x & 31;
    const uint64_t hw = keys[s] & 0xffffffff00000000ull;
    uint64_t c[NR];
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int e = lane * NR + j;
        c[j] = e < len ? ((keys[s + e] & 0xffffffffull) << 32) | (uint64_t)idx[s + e] : ~0ull;
    }
    warp_sort_u64<NR>(c);
#pragma unroll
    for (int j = 0; j < NR; ++j) {
        const int e = lane * NR + j;
        if (e < len) {
            keys[s + e] = hw | (c[j] >> 32);
            idx[s + e] = (uint32_t)c[j];
        }
    }
}

// The listed runs: first those over kWarpRun keys, a block each (up to
// kBigSmem keys sorted in shared memory by (low word, index) with the bitonic
// network of cmpswap_u64 below; longer runs by four stable passes of 8 bits
// over the low word, between the run's place in buffers 0 and 1: tiles of 256
// keys in order, within a tile warp match_any ranks and per-warp digit counts
// keep the order); then the others, a warp each, the composites sorted in
// registers. The two groups of runs are disjoint, so the phases need no barrier
// between them.
__device__ __forceinline__ void cmpswap_u64(uint64_t *v, int i, int j)
{
    const uint64_t a = v[i], b = v[j];
    if (b < a) {
        v[i] = b;
        v[j] = a;
    }
}

__global__ __launch_bounds__(256) void k_sort_runs(uint64_t *k0, uint32_t *v0, uint64_t *k1, uint32_t *v1,
                                                   const int2 *__restrict__ big, int cap_big, const DevCounters *cst)
{
    __shared__ uint64_t s_c[kBigSmem];
    __shared__ unsigned s_wcnt[8][256];
    __shared__ unsigned s_base[256];
    __shared__ unsigned s_wsum[8];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = min(cst->n_sort_groups, cap_big);
    for (int b = blockIdx.x; b < nb; b += gridDim.x) {
        const int2 r = big[b];
        if (r.y <= kWarpRun) continue;  // block-uniform: the warp kernel's runs
        const int s = r.x, G = r.y, e = s + G;
        const uint32_t hw = (uint32_t)(k0[s] >> 32);
        if (G <= kBigSmem) {
            int S = 2;
            while (S < G) S <<= 1;
            for (int i = tid; i < S; i += 256)
                s_c[i] = i < G ? ((k0[s + i] & 0xffffffffull) << 32) | (uint64_t)v0[s + i] : ~0ull;
            __syncthreads();
            for (int lk = 1; (1 << lk) <= S; ++lk) {
                const int k = 1 << lk;
                for (int i = tid; i < S / 2; i += 256) {
                    const int blk = i >> (lk - 1), pos = i & ((k >> 1) - 1);
                    cmpswap_u64(s_c, blk * k + pos, blk * k + k - 1 - pos);
                }
                __syncthreads();
                for (int lj = lk - 2; lj >= 0; --lj) {
                    const int j = 1 << lj;
                    for (int i = tid; i < S / 2; i += 256) {
                        const int blk = i >> lj, pos = i & (j - 1);
                        cmpswap_u64(s_c, (blk << (lj + 1)) + pos, (blk << (lj + 1)) + pos + j);
                    }
                    __syncthreads();
                }
            }
            for (int i = tid; i < G; i += 256) {
                const uint64_t c = s_c[i];
                k0[s + i] = ((uint64_t)hw << 32) | (c >> 32);
                v0[s + i] = (uint32_t)c;
            }
            __syncthreads();
            continue;
        }
        for (int pass = 0; pass < 4; ++pass) {
            const uint64_t *ki = (pass & 1) ? k1 : k0;
            const uint32_t *vi = (pass & 1) ? v1 : v0;
            uint64_t *ko = (pass & 1) ? k0 : k1;
            uint32_t *vo = (pass & 1) ? v0 : v1;
            const int shift = 8 * pass;
            for (int i = tid; i < 8 * 256; i += 256) (&s_wcnt[0][0])[i] = 0;
            __syncthreads();
            for (int j = s + tid; j < e; j += 256) atomicAdd(&s_wcnt[0][(ki[j] >> shift) & 255u], 1u);
            __syncthreads();
            {  // exclusive scan of the run's digit counts into the digits' starts
                const unsigned c = s_wcnt[0][tid];
                const unsigned incl = (unsigned)warp_incl_scan((int)c);
                if (lane == 31) s_wsum[warp] = incl;
                __syncthreads();
                unsigned wb = 0;
                for (int w = 0; w < warp; ++w) wb += s_wsum[w];
                s_base[tid] = (unsigned)s + wb + incl - c;
                s_wcnt[0][tid] = 0;
            }
            __syncthreads();
            for (int t0 = s; t0 < e; t0 += 256) {
                const int j = t0 + tid;
                const bool valid = j < e;
                const unsigned d = valid ? (unsigned)((ki[j] >> shift) & 255u) : 256u;
                const unsigned peers = __match_any_sync(kFull, d);
                const int leader = __ffs(peers) - 1;
                if (lane == leader && valid) s_wcnt[warp][d] = __popc(peers);
                __syncthreads();
                if (valid) {
                    unsigned off = s_base[d] + __popc(peers & lanemask_lt());
                    for (int w = 0; w < warp; ++w) off += s_wcnt[w][d];
                    ko[off] = ki[j];
                    vo[off] = vi[j];
                }
                __syncthreads();
                unsigned add = 0;
                for (int w = 0; w < 8; ++w) {
                    add += s_wcnt[w][tid];
                    s_wcnt[w][tid] = 0;
                }
                s_base[tid] += add;
                __syncthreads();
            }
        }
    }
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nb; b += nwarps) {
        const int2 r = big[b];
        if (r.y <= 64) sort_run_warp<2>(k0, v0, r.x, r.y);
        else if (r.y <= 128) sort_run_warp<4>(k0, v0, r.x, r.y);
        else if (r.y <= 256) sort_run_warp<8>(k0, v0, r.x, r.y);
        else if (r.y <= kWarpRun) sort_run_warp<16>(k0, v0, r.x, r.y);
    }
}

template <class T>
int launch_keys_t(Plan &P, const void *pos, cudaStream_t s)
{
    const int nb = P.num_sms * 4;
    k_bbox<T><<<nb, kBoxThreads, 0, s>>>((const T *)pos, (int)P.n, (T *)P.scratch, P.ctr);
    // blocks of 1024 threads: each block adds its digit counts to the global histograms once, so fewer,
    // larger blocks put fewer atomics on the same counters
    k_keys<T><<<P.num_sms * 2, 1024, 0, s>>>((const T *)pos, (int)P.n, P.keys[0], P.sort_full ? 0 : kSortHighPass0,
                                             P.ctr);
    return 2;
}

template <int ITEMS>
int radix_passes(Plan &P, int p0, cudaStream_t s)
{
    const int n = (int)P.n;
    const int tiles = (n + RS_THREADS * ITEMS - 1) / (RS_THREADS * ITEMS);
    const int smem = RS_THREADS * ITEMS * (int)(sizeof(uint64_t) + sizeof(uint32_t));
    cudaFuncSetAttribute(k_radix_pass<true, ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaFuncSetAttribute(k_radix_pass<false, ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    for (int pass = p0; pass < 8; ++pass) {
        const int src = pass & 1, dst = src ^ 1;
        const int slot = P.next_slot();
        const unsigned ep = P.next_epoch();
        if (pass == p0)
            k_radix_pass<true, ITEMS><<<tiles, RS_THREADS, smem, s>>>(P.keys[src], nullptr, P.keys[dst], P.idx[dst], n,
                                                                      pass, P.flags, ep, slot, P.ctr);
        else
            k_radix_pass<false, ITEMS><<<tiles, RS_THREADS, smem, s>>>(P.keys[src], P.idx[src], P.keys[dst], P.idx[dst],
                                                                       n, pass, P.flags, ep, slot, P.ctr);
    }
    return 8 - p0;
}

template <int ITEMS>
int coop_tiles_max(int num_sms)
{
    const int smem = RS_THREADS * ITEMS * (int)(sizeof(uint64_t) + sizeof(uint32_t));
    cudaFuncSetAttribute(k_radix_coop<ITEMS>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    int b = 0;
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_radix_coop<ITEMS>, RS_THREADS, smem);
    return b * num_sms;
}

// The cooperative sort when every tile fits on the GPU at once; false otherwise.
template <int ITEMS>
bool radix_coop(Plan &P, int p0, cudaStream_t s)
{
    const int n = (int)P.n;
    const int tiles = (n + RS_THREADS * ITEMS - 1) / (RS_THREADS * ITEMS);
    // below 16 tiles the per-pass kernels win (their look-backs are short and the launches cost less than
    // the cooperative kernel's grid barriers); above the co-resident tiles they are the only choice
    if (tiles < 16 || tiles > P.coop_tiles_sort[ITEMS == RS_ITEMS_LARGE ? 1 : 0] || (size_t)tiles * 256 > P.sort_cnt_cap)
        return false;
    const int smem = RS_THREADS * ITEMS * (int)(sizeof(uint64_t) + sizeof(uint32_t));
    GridBarrier *gb = P.gbar + 2;
    void *args[] = {&P.keys[0], &P.idx[0], &P.keys[1], &P.idx[1], (void *)&n, &p0, &P.sort_cnt, &gb, &P.ctr};
    if (cudaLaunchCooperativeKernel((const void *)k_radix_coop<ITEMS>, dim3(tiles), dim3(RS_THREADS), args, smem, s) !=
        cudaSuccess) {
        cudaGetLastError();  // a refused launch (not expected: the tiles were counted against the capacity)
        return false;
    }
    return true;
}

template <class T>
int launch_sort_t(Plan &P, const void *pos, const void *mass, cudaStream_t s)
{
    const int n = (int)P.n;
    const int p0 = P.sort_full ? 0 : kSortHighPass0;  // an even number of passes: the data ends in buffer 0
    int launches;
    if (P.n >= (1 << 19) ? radix_coop<RS_ITEMS_LARGE>(P, p0, s) : radix_coop<RS_ITEMS_SMALL>(P, p0, s))
        launches = 1;
    else
        launches = P.n >= (1 << 19) ? radix_passes<RS_ITEMS_LARGE>(P, p0, s) : radix_passes<RS_ITEMS_SMALL>(P, p0, s);
    if (!P.sort_full) {
        // ordered by high word; then the runs of equal high words by low word and index
        const int cap_big = (int)P.sort_big_cap;
        // one wave of blocks: a partial second wave would wait for the first's latency-bound loads
        static int groups_per_sm = 0;
        if (!groups_per_sm) {
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&groups_per_sm, k_sort_groups, 256, 0);
            groups_per_sm = std::max(groups_per_sm, 1);
        }
        k_sort_groups<<<P.num_sms * groups_per_sm, 256, 0, s>>>(P.keys[0], P.idx[0], n, P.sort_big, cap_big, P.ctr);
        k_sort_runs<<<P.num_sms * 4, 256, 0, s>>>(P.keys[0], P.idx[0], P.keys[1], P.idx[1], P.sort_big, cap_big,
                                                  P.ctr);
        launches += 2;
    }
    if (P.mass_wait) cudaStreamWaitEvent(s, P.mass_wait, 0);  // masses still arriving on a side stream
    k_gather_diverge<T><<<P.num_sms * 4, 256, 0, s>>>(P.keys[0], P.idx[0], n, (const T *)pos, (const T *)mass,
                                                     (vec4<T> *)P.xyzm, P.div, P.node_first, P.node_count,
                                                     P.node_child0, P.node_nchild, P.node_parent, P.node_level,
                                                     P.ctr);
    return launches + 1;
}

}  // namespace

int launch_keys(Plan &P, const void *pos, cudaStream_t s)
{
    return P.dtype == 0 ? launch_keys_t<float>(P, pos, s) : launch_keys_t<double>(P, pos, s);
}

int launch_sort(Plan &P, const void *pos, const void *mass, cudaStream_t s)
{
    return P.dtype == 0 ? launch_sort_t<float>(P, pos, mass, s) : launch_sort_t<double>(P, pos, mass, s);
}

void sort_coop_capacity(int num_sms, int tiles[2])
{
    tiles[0] = coop_tiles_max<RS_ITEMS_SMALL>(num_sms);
    tiles[1] = coop_tiles_max<RS_ITEMS_LARGE>(num_sms);
}

}  // namespace bfm
