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

int launch_drift(Plan &P, void *pos, const void *vel, double dt, cudaStream_t s)
{
    return P.dtype == 0 ? axpy_t<float>(P, pos, vel, dt, s) : axpy_t<double>(P, pos, vel, dt, s);
}

}  // namespace bfm
