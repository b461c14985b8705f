// Host build of the CUDA path's generated expansion operators, so that the
// tests can check them against the oracle without a GPU. Test-only.
#include <cmath>
#include <cstdint>
#define BFM_HOST_SHIM 1
#define __device__
#define __forceinline__ inline
namespace bfm {
inline float rsqrt_t(float x) { return 1.0f / std::sqrt(x); }
inline double rsqrt_t(double x) { return 1.0 / std::sqrt(x); }
}  // namespace bfm
#include "../../body_forces_morton_b300/csrc/expansions_gen.cuh"
#include "../../body_forces_morton_b300/csrc/rotation_gen.cuh"

using namespace bfm;

template <int P, class T>
static void run(int op, const T* a, const T* v, T* out)
{
    switch (op) {
    case 0: Exp<P>::template p2m<T>(v[0], v[1], v[2], v[3], out); break;
    case 1: Exp<P>::template m2m<T>(a, v[0], v[1], v[2], out); break;
    case 2: Exp<P>::template m2l<T>(a, v[0], v[1], v[2], out); break;
    case 3: Exp<P>::template l2l<T>(a, v[0], v[1], v[2], out); break;
    case 4: Exp<P>::template l2p<T>(a, v[0], v[1], v[2], out[0], out[1], out[2], out[3]); break;
    case 5: {  // reduced M2L: expand_l(m2l_r(reduce_m(M), R))
        T Mr[Exp<P>::NRC], Lr[Exp<P>::NRC];
        for (int i = 0; i < Exp<P>::NRC; ++i) Lr[i] = T(0);
        Exp<P>::template reduce_m<T>(a, Mr);
        Exp<P>::template m2l_r<T>(Mr, v[0], v[1], v[2], Lr);
        Exp<P>::template expand_l<T>(Lr, out);
        break;
    }
    case 7: Exp<P>::template p2m_dip<T>(v[0], v[1], v[2], v[3], v[4], v[5], v[6], out); break;  // s, q, d
    case 8: Exp<P>::template l2p_hess<T>(a, v[0], v[1], v[2], out); break;
    case 9: {  // rotation-based M2L: from_sph(m2l(to_sph(M), R))
        T Q[Rot<P>::NS], Ls[Rot<P>::NS];
        for (int i = 0; i < Rot<P>::NS; ++i) Ls[i] = T(0);
        Rot<P>::template to_sph<T>(a, Q);
        Rot<P>::template m2l<T>(Q, v[0], v[1], v[2], Ls);
        Rot<P>::template from_sph<T>(Ls, out);
        break;
    }
    case 6: {  // both directions of one pair: a = [M_A, M_B], out = [L_A, L_B]
        constexpr int NC = Exp<P>::NC, NRC = Exp<P>::NRC;
        T MA[NRC], MB[NRC], LA[NRC], LB[NRC];
        for (int i = 0; i < NRC; ++i) LA[i] = LB[i] = T(0);
        Exp<P>::template reduce_m<T>(a, MA);
        Exp<P>::template reduce_m<T>(a + NC, MB);
        Exp<P>::template m2l_r_pair<T>(MA, MB, v[0], v[1], v[2], LA, LB);
        Exp<P>::template expand_l<T>(LA, out);
        Exp<P>::template expand_l<T>(LB, out + NC);
        break;
    }
    }
}

template <class T>
static int dispatch(int p, int op, const T* a, const T* v, T* out)
{
    switch (p) {
    case 0: run<0, T>(op, a, v, out); return 0;
    case 1: run<1, T>(op, a, v, out); return 0;
    case 2: run<2, T>(op, a, v, out); return 0;
    case 3: run<3, T>(op, a, v, out); return 0;
    case 4: run<4, T>(op, a, v, out); return 0;
    case 5: run<5, T>(op, a, v, out); return 0;
    case 6: run<6, T>(op, a, v, out); return 0;
    case 7: run<7, T>(op, a, v, out); return 0;
    case 8: run<8, T>(op, a, v, out); return 0;
    }
    return 1;
}

extern "C" int shim_op_f64(int p, int op, const double* a, const double* v, double* out)
{
    return dispatch<double>(p, op, a, v, out);
}
extern "C" int shim_op_f32(int p, int op, const float* a, const float* v, float* out)
{
    return dispatch<float>(p, op, a, v, out);
}
