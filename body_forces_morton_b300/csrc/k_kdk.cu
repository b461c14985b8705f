// Kick and drift of the kick-drift-kick leapfrog (Jaxion post, section
// "Implementation": half kick, full drift, half kick).
#include "plan.h"

namespace bfm {

namespace {

// y[i] += x[i] * h over m contiguous values
template <class T>
__global__ void k_axpy(T *__restrict__ y, const T *__restrict__ x, T h, int64_t m)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < m; i += (int64_t)gridDim.x * blockDim.x)
        y[i] += x[i] * h;
}

// y[i] = round_lattice(y[i]) + round_lattice(x[i] * h): lattice spacing 2^e
// (exact power-of-two scalings; rint rounds half to even, so the increment
// changes sign exactly with h). x == nullptr only rounds y onto its lattice.
template <class T>
__global__ void k_lattice_axpy(T *__restrict__ y, const T *__restrict__ x, T h, int e_y, int e_inc, int64_t m)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < m; i += (int64_t)gridDim.x * blockDim.x) {
        const T yy = ldexp(rint(ldexp(y[i], -e_y)), e_y);
        const T inc = x ? ldexp(rint(ldexp(x[i] * h, -e_inc)), e_inc) : T(0);
        y[i] = yy + inc;
    }
}

template <class T>
int lattice_t(Plan &P, void *y, const void *x, double h, int e_y, int e_inc, cudaStream_t s)
{
    k_lattice_axpy<T><<<P.num_sms * 8, 256, 0, s>>>((T *)y, (const T *)x, (T)h, e_y, e_inc, 3 * P.n);
    return 1;
}

template <class T>
int axpy_t(Plan &P, void *y, const void *x, double h, cudaStream_t s)
{
    k_axpy<T><<<P.num_sms * 8, 256, 0, s>>>((T *)y, (const T *)x, (T)h, 3 * P.n);
    return 1;
}

}  // namespace

int launch_kick(Plan &P, void *vel, const void *acc, double h, cudaStream_t s)
{
    return P.dtype == 0 ? axpy_t<float>(P, vel, acc, h, s) : axpy_t<double>(P, vel, acc, h, s);
}

int launch_lattice_axpy(Plan &P, void *y, const void *x, double h, int e_y, int e_inc, cudaStream_t s)
{
    return P.dtype == 0 ? lattice_t<float>(P, y, x, h, e_y, e_inc, s) : lattice_t<double>(P, y, x, h, e_y, e_inc, s);
}

int launch_drift(Plan &P, void *pos, const void *vel, double dt, cudaStream_t s)
{
    return P.dtype == 0 ? axpy_t<float>(P, pos, vel, dt, s) : axpy_t<double>(P, pos, vel, dt, s);
}

}  // namespace bfm
