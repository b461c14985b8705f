// fmm_morton_keys_noalloc: the root box and the Morton keys of up to 2^21
// particles without any device allocation.
//
// Some callers cannot allocate device memory at the time they need keys: code
// that owns a fixed memory budget handed out by its own allocator, a library
// embedded in a host application that forbids device allocation after
// start-up, or a real-time loop that must not take the driver's allocation
// locks. This entry
// point gives them the first stage of the FMM pipeline with nothing but the
// caller's input and output buffers: the reduction's scratch (one partial box
// per block, a ticket counter, the finished box and a status word) lives in a
// fixed array of this library's device image.
//
// The arithmetic is the same as the plan path's keys: 21-bit quantisation of
// each coordinate against the root cube, every step rounded in the input
// precision, bits interleaved with x highest.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/fmm.h"

namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 8;
constexpr int kMaxBlocks = 1024;                      // partial boxes the scratch can hold
constexpr int64_t kMaxN = (int64_t)kMaxBlocks * kThreads * kPerThread;  // 2^21 particles
constexpr int kScratchDoubles = 6 * kMaxBlocks + 8;   // partials, then ticket/status words, then the box

// Shared by every call on a device and kept between calls (48 KiB per device).
static __device__ __align__(256) double g_keys_scratch[kScratchDoubles];

struct ScratchView {
    double *partial;   // [kMaxBlocks][6]: lo xyz, hi xyz
    unsigned *ticket;  // blocks finished in this call (cleared by every call)
    unsigned *status;  // bit 0: a coordinate is not finite (cleared by every call)
    double *box;       // [4]: lo xyz, side
};

__device__ __forceinline__ ScratchView view(double *s)
{
    ScratchView v;
    v.partial = s;
    v.ticket = reinterpret_cast<unsigned *>(s + 6 * kMaxBlocks);
    v.status = v.ticket + 1;
    v.box = s + 6 * kMaxBlocks + 4;
    return v;
}

template <class T> __device__ __forceinline__ T lo_of(T a, T b) { return b < a ? b : a; }
template <class T> __device__ __forceinline__ T hi_of(T a, T b) { return b > a ? b : a; }
template <class T> __device__ __forceinline__ T inf_of();
template <> __device__ __forceinline__ float inf_of<float>() { return __int_as_float(0x7f800000); }
template <> __device__ __forceinline__ double inf_of<double>() { return __longlong_as_double(0x7ff0000000000000ll); }
__device__ __forceinline__ float sub_exact(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ double sub_exact(double a, double b) { return __dsub_rn(a, b); }
__device__ __forceinline__ float div_exact(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ double div_exact(double a, double b) { return __ddiv_rn(a, b); }
__device__ __forceinline__ float mul_exact(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ double mul_exact(double a, double b) { return __dmul_rn(a, b); }

// Root box: block b covers particles [b * 2048, (b + 1) * 2048); the last block
// to finish reduces the partial boxes and stores the cube's corner and side.
template <class T>
__global__ __launch_bounds__(kThreads) void k_box_noalloc(const T *__restrict__ pos, int n, double *scratch)
{
    const ScratchView S = view(scratch);
    T lo[3], hi[3];
    for (int a = 0; a < 3; ++a) { lo[a] = inf_of<T>(); hi[a] = -inf_of<T>(); }
    bool bad = false;
    const int base = blockIdx.x * kThreads * kPerThread;
    for (int k = 0; k < kPerThread; ++k) {
        const int i = base + k * kThreads + threadIdx.x;
        if (i < n)
            for (int a = 0; a < 3; ++a) {
                const T v = pos[3 * (int64_t)i + a];
                bad |= !isfinite(v);
                lo[a] = lo_of(lo[a], v);
                hi[a] = hi_of(hi[a], v);
            }
    }
    if (__any_sync(0xffffffffu, bad) && (threadIdx.x & 31) == 0) atomicOr(S.status, 1u);
    for (int o = 16; o > 0; o >>= 1)
        for (int a = 0; a < 3; ++a) {
            lo[a] = lo_of(lo[a], __shfl_xor_sync(0xffffffffu, lo[a], o));
            hi[a] = hi_of(hi[a], __shfl_xor_sync(0xffffffffu, hi[a], o));
        }
    __shared__ T s[kThreads / 32][6];
    __shared__ bool last;
    if ((threadIdx.x & 31) == 0)
        for (int a = 0; a < 3; ++a) { s[threadIdx.x >> 5][a] = lo[a]; s[threadIdx.x >> 5][3 + a] = hi[a]; }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kThreads / 32; ++w)
            for (int a = 0; a < 3; ++a) {
                s[0][a] = lo_of(s[0][a], s[w][a]);
                s[0][3 + a] = hi_of(s[0][3 + a], s[w][3 + a]);
            }
        for (int a = 0; a < 6; ++a) S.partial[6 * blockIdx.x + a] = (double)s[0][a];
        __threadfence();
        last = atomicAdd(S.ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!last || threadIdx.x != 0) return;
    __threadfence();
    T r[6];
    for (int a = 0; a < 3; ++a) { r[a] = inf_of<T>(); r[3 + a] = -inf_of<T>(); }
    for (int b = 0; b < (int)gridDim.x; ++b)
        for (int a = 0; a < 3; ++a) {
            r[a] = lo_of(r[a], (T)__ldcg(S.partial + 6 * b + a));
            r[3 + a] = hi_of(r[3 + a], (T)__ldcg(S.partial + 6 * b + 3 + a));
        }
    T side = sub_exact(r[3], r[0]);
    for (int a = 1; a < 3; ++a) {
        const T e = sub_exact(r[3 + a], r[a]);
        if (e > side) side = e;
    }
    if (!(side > T(0))) side = T(1);
    for (int a = 0; a < 3; ++a) S.box[a] = (double)r[a];
    S.box[3] = (double)side;
}

__device__ __forceinline__ uint64_t spread_bits(uint32_t v)
{
    uint64_t x = v & 0x1fffffu;
    x = (x | (x << 32)) & 0x1f00000000ffffull;
    x = (x | (x << 16)) & 0x1f0000ff0000ffull;
    x = (x | (x << 8)) & 0x100f00f00f00f00full;
    x = (x | (x << 4)) & 0x10c30c30c30c30c3ull;
    x = (x | (x << 2)) & 0x1249249249249249ull;
    return x;
}

template <class T> __device__ __forceinline__ uint32_t cell(T x, T lo, T side)
{
    const T u = mul_exact(div_exact(sub_exact(x, lo), side), T(2097152.0));
    const uint32_t q = (uint32_t)floor(u);
    return q > 2097151u ? 2097151u : q;
}

template <class T>
__global__ __launch_bounds__(kThreads) void k_keys_noalloc(const T *__restrict__ pos, int n, const double *scratch,
                                                           uint64_t *__restrict__ keys, double *__restrict__ box_out)
{
    const double *box = scratch + 6 * kMaxBlocks + 4;
    const T lo0 = (T)box[0], lo1 = (T)box[1], lo2 = (T)box[2], side = (T)box[3];
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0 && box_out)
        for (int a = 0; a < 4; ++a) box_out[a] = box[a];
    if (i >= n) return;
    const T *q = pos + 3 * (int64_t)i;
    keys[i] = (spread_bits(cell(q[0], lo0, side)) << 2) | (spread_bits(cell(q[1], lo1, side)) << 1) |
              spread_bits(cell(q[2], lo2, side));
}

// Device address of the scratch array, looked up once per device.
std::mutex g_mu;
double *g_ptr[64] = {};

fmm_status scratch_for_current_device(double **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FMM_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_keys_scratch) != cudaSuccess || !p) return FMM_ERR_CUDA;
        g_ptr[dev] = static_cast<double *>(p);
    }
    *out = g_ptr[dev];
    return FMM_OK;
}

}  // namespace

extern "C" fmm_status fmm_morton_keys_noalloc(const void *pos, int64_t n, fmm_dtype dtype, uint64_t *keys_out,
                                              double *box_out, void *stream)
{
    if (!pos || !keys_out || n < 1 || (dtype != FMM_F32 && dtype != FMM_F64)) return FMM_ERR_INVALID_ARG;
    if (n > kMaxN) return FMM_ERR_INVALID_ARG;  // the scratch holds 1024 partial boxes of 2048 particles each
    double *scratch = nullptr;
    fmm_status st = scratch_for_current_device(&scratch);
    if (st != FMM_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const int ni = (int)n;
    const int blocks = (ni + kThreads * kPerThread - 1) / (kThreads * kPerThread);
    // the ticket and the status word start at zero in every call
    if (cudaMemsetAsync(scratch + 6 * kMaxBlocks, 0, 2 * sizeof(unsigned), s) != cudaSuccess) return FMM_ERR_CUDA;
    if (dtype == FMM_F32) {
        k_box_noalloc<float><<<blocks, kThreads, 0, s>>>((const float *)pos, ni, scratch);
        k_keys_noalloc<float><<<(ni + kThreads - 1) / kThreads, kThreads, 0, s>>>((const float *)pos, ni, scratch,
                                                                               keys_out, box_out);
    } else {
        k_box_noalloc<double><<<blocks, kThreads, 0, s>>>((const double *)pos, ni, scratch);
        k_keys_noalloc<double><<<(ni + kThreads - 1) / kThreads, kThreads, 0, s>>>((const double *)pos, ni, scratch,
                                                                                 keys_out, box_out);
    }
    if (cudaGetLastError() != cudaSuccess) return FMM_ERR_CUDA;
    unsigned status = 0;
    if (cudaMemcpyAsync(&status, reinterpret_cast<unsigned *>(scratch + 6 * kMaxBlocks) + 1, sizeof(unsigned),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return FMM_ERR_CUDA;
    return status ? FMM_ERR_NONFINITE : FMM_OK;
}
