/*
 * fmm_oracle.c -- plain, slow CPU reference for one FMM evaluation.
 *
 * TEST INFRASTRUCTURE. This file is the oracle the CUDA path is checked
 * against. Only the test-suite, the package's smoke check and the benchmark's
 * CPU-baseline leg may load it; the library itself never does, and the two
 * share no code.
 *
 * It follows the JZ-FMM page ("How the Fast Multipole Method works"):
 *   direct gravity       -- section "From particle pairs to node pairs", first eq.
 *   multipole moments    -- section "Describing the source and the receiving region", moment eqs.
 *   local Taylor series  -- same section, Taylor eq.
 *   M2L                  -- section "Calculating a node-node interaction", Phi_B and grad Phi_B eqs.
 *   opening criterion    -- the theta eq. after the interactive demo
 *   three stages         -- section "Combining near and far interactions"
 *   GPU layout           -- section "Why this works well on GPUs" (sorted particles, contiguous children)
 * and the kick-drift-kick loop of the Jaxion post (section "Implementation", `_update`).
 *
 * Readings where the page is silent (all stated once more in the design notes):
 *   - "order p" keeps every term with |n| + |k| <= p (the demo caption: "terms through total degree p").
 *   - moments are normalised M_n = sum m s^n / n! (multi-index factorial); this only rescales coefficients.
 *   - node centre and half-width come from the tight axis-aligned box of the node's particles.
 *   - octree on 21-bit-per-axis Morton cells of the root cube; a node splits when count > leaf and depth < 21.
 *   - dual-tree walk: symmetric traversal, split the node with the larger |l| (lower index on ties),
 *     never split a leaf; accept iff |l_A + l_B|^2 < theta^2 |c_A - c_B|^2 for A != B.
 *   - pairs at zero separation (the particle itself, or a coincident one) are skipped.
 *   - geometry (centres, half-widths, criterion, split choice, Morton quantisation) is evaluated in the
 *     input precision, operation by operation, without contraction; expansion arithmetic is fp64.
 *
 * Coefficient order (an interface shared with the CUDA path's debug export, restated there):
 * graded by total degree d = 0..p; within a degree, nx from d down to 0, then ny from d-nx down to 0.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -shared -fPIC
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL 1
#define ORC_ENOMEM 2
#define ORC_ENONFINITE 3

#define ORC_MAXP 8
#define ORC_MAXP_DERIV 18  /* derivative tensors are available to this order (for tests) */
#define ORC_NCMAX 1330     /* number of monomials of degree <= ORC_MAXP_DERIV */
#define ORC_KEY_BITS 21
#define ORC_MAX_DEPTH 21
#define ORC_DTYPE_F32 0
#define ORC_DTYPE_F64 1

/* ------------------------------------------------------------------------ */
/* multi-indices                                                             */
/* ------------------------------------------------------------------------ */

int orc_ncoef(int p) { return (p + 1) * (p + 2) * (p + 3) / 6; }

/* Position of monomial x^nx y^ny z^nz in the graded order described above. */
int orc_mindex(int nx, int ny, int nz)
{
    int d = nx + ny + nz;
    int t = d - nx;
    return d * (d + 1) * (d + 2) / 6 + t * (t + 1) / 2 + (t - ny);
}

static void mi_table(int p, int (*mi)[3])
{
    for (int d = 0; d <= p; ++d)
        for (int nx = d; nx >= 0; --nx)
            for (int ny = d - nx; ny >= 0; --ny) {
                int nz = d - nx - ny;
                int i = orc_mindex(nx, ny, nz);
                mi[i][0] = nx; mi[i][1] = ny; mi[i][2] = nz;
            }
}

static double factorial(int n)
{
    double f = 1.0;
    for (int i = 2; i <= n; ++i) f *= (double)i;
    return f;
}

static double mfact(const int *n) { return factorial(n[0]) * factorial(n[1]) * factorial(n[2]); }

static double ipow(double x, int k)
{
    double r = 1.0;
    for (int i = 0; i < k; ++i) r *= x;
    return r;
}

/* x^n / n! for a 3-vector and multi-index n */
static double mono_over_fact(const double *x, const int *n)
{
    return ipow(x[0], n[0]) * ipow(x[1], n[1]) * ipow(x[2], n[2]) / mfact(n);
}

/* ------------------------------------------------------------------------ */
/* direct sum (JZ-FMM page, direct gravity eq.; acceleration a = -grad Phi)   */
/* ------------------------------------------------------------------------ */

/* Kahan-compensated accumulator */
typedef struct { double s, c; } ksum;
static void kadd(ksum *k, double v)
{
    double y = v - k->c;
    double t = k->s + y;
    k->c = (t - k->s) - y;
    k->s = t;
}

/*
 * Exact O(N^2) sum over all sources j != i with nonzero separation, for the
 * targets listed in `targets` (n_targets entries; NULL = all particles).
 * Outputs are written at the target's own index: acc[3*i..], pot[i].
 */
int orc_direct_sum(int64_t n, const double *pos, const double *mass, int64_t n_targets,
                   const int64_t *targets, double *acc, double *pot, int nthreads)
{
    if (n < 0 || !pos || !mass || !acc) return ORC_EINVAL;
    int64_t nt = targets ? n_targets : n;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t t = 0; t < nt; ++t) {
        int64_t i = targets ? targets[t] : t;
        ksum ax = {0, 0}, ay = {0, 0}, az = {0, 0}, ph = {0, 0};
        const double xi = pos[3 * i], yi = pos[3 * i + 1], zi = pos[3 * i + 2];
        for (int64_t j = 0; j < n; ++j) {
            double dx = pos[3 * j] - xi, dy = pos[3 * j + 1] - yi, dz = pos[3 * j + 2] - zi;
            double r2 = dx * dx + dy * dy + dz * dz;
            if (r2 == 0.0) continue; /* self-interaction (and exact coincidences) omitted */
            double r = sqrt(r2);
            double mr3 = mass[j] / (r2 * r);
            kadd(&ax, mr3 * dx);
            kadd(&ay, mr3 * dy);
            kadd(&az, mr3 * dz);
            kadd(&ph, -mass[j] / r);
        }
        acc[3 * i] = ax.s; acc[3 * i + 1] = ay.s; acc[3 * i + 2] = az.s;
        if (pot) pot[i] = ph.s;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* expansion operators                                                       */
/* ------------------------------------------------------------------------ */

/*
 * D^n(R) = d^n (1/r) / dR^n for all |n| <= p.
 * Recurrence from Euler's relation for the degree -(l+1) homogeneous function D^n
 * with l = |n|:
 *   l r^2 D^n = -(2l-1) sum_i n_i R_i D^{n-e_i} - (l-1) sum_i n_i (n_i-1) D^{n-2e_i}.
 */
int orc_derivs(int p, const double *R, double *D)
{
    if (p < 0 || p > ORC_MAXP_DERIV) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    double r2 = R[0] * R[0] + R[1] * R[1] + R[2] * R[2];
    D[0] = 1.0 / sqrt(r2);
    for (int a = 1; a < nc; ++a) {
        const int *n = mi[a];
        int l = n[0] + n[1] + n[2];
        double s = 0.0;
        for (int i = 0; i < 3; ++i) {
            if (n[i] >= 1) {
                int m[3] = {n[0], n[1], n[2]};
                m[i] -= 1;
                s -= (double)(2 * l - 1) * (double)n[i] * R[i] * D[orc_mindex(m[0], m[1], m[2])];
            }
            if (n[i] >= 2) {
                int m[3] = {n[0], n[1], n[2]};
                m[i] -= 2;
                s -= (double)(l - 1) * (double)(n[i] * (n[i] - 1)) * D[orc_mindex(m[0], m[1], m[2])];
            }
        }
        D[a] = s / ((double)l * r2);
    }
    return ORC_OK;
}

/* P2M: M_n += sum_j m_j s_j^n / n!, s_j = x_j - c (moment eqs.; higher moments "follow the same pattern"). */
int orc_p2m(int p, int64_t n, const double *pos, const double *mass, const double *c, double *M)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    for (int64_t j = 0; j < n; ++j) {
        double s[3] = {pos[3 * j] - c[0], pos[3 * j + 1] - c[1], pos[3 * j + 2] - c[2]};
        for (int a = 0; a < nc; ++a) M[a] += mass[j] * mono_over_fact(s, mi[a]);
    }
    return ORC_OK;
}

/* M2M: parent moments about c_P from child moments about c_C, d = c_C - c_P:
 *   M^P_n += sum_{k <= n} M^C_k d^{n-k} / (n-k)!   (stage 1: "translate and combine the children's moments") */
int orc_m2m(int p, const double *Mc, const double *d, double *Mp)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    for (int a = 0; a < nc; ++a) {
        const int *n = mi[a];
        double s = 0.0;
        for (int b = 0; b < nc; ++b) {
            const int *k = mi[b];
            if (k[0] > n[0] || k[1] > n[1] || k[2] > n[2]) continue;
            int q[3] = {n[0] - k[0], n[1] - k[1], n[2] - k[2]};
            s += Mc[b] * mono_over_fact(d, q);
        }
        Mp[a] += s;
    }
    return ORC_OK;
}

/*
 * M2L: local coefficients at c_A from source moments at c_B, R = c_A - c_B:
 *   L_k += -G sum_{|n| <= p-|k|} (-1)^{|n|} M_n D^{n+k}(R),  G = 1.
 * Obtained by Taylor-expanding 1/|R + dx - s| in both offsets; its k = 0 and
 * k = e_alpha terms through |n| <= 1 are the page's Phi_B and grad Phi_B eqs.
 * The local series is Phi(c_A + dx) = sum_k L_k dx^k / k!.
 */
int orc_m2l(int p, const double *M, const double *R, double *L)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    double D[ORC_NCMAX];
    mi_table(p, mi);
    orc_derivs(p, R, D);
    for (int a = 0; a < nc; ++a) {
        const int *k = mi[a];
        int lk = k[0] + k[1] + k[2];
        double s = 0.0;
        for (int b = 0; b < nc; ++b) {
            const int *n = mi[b];
            int ln = n[0] + n[1] + n[2];
            if (ln + lk > p) continue;
            double sign = (ln & 1) ? -1.0 : 1.0;
            s += sign * M[b] * D[orc_mindex(n[0] + k[0], n[1] + k[1], n[2] + k[2])];
        }
        L[a] += -s;
    }
    return ORC_OK;
}

/* L2L: child local about c_C = c_P + e:  L^C_k += sum_{j >= k, |j| <= p} L^P_j e^{j-k} / (j-k)!
 * (stage 3: "translate each parent's local Taylor expansion to its children") */
int orc_l2l(int p, const double *Lp, const double *e, double *Lc)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    for (int a = 0; a < nc; ++a) {
        const int *k = mi[a];
        double s = 0.0;
        for (int b = 0; b < nc; ++b) {
            const int *j = mi[b];
            if (j[0] < k[0] || j[1] < k[1] || j[2] < k[2]) continue;
            int q[3] = {j[0] - k[0], j[1] - k[1], j[2] - k[2]};
            s += Lp[b] * mono_over_fact(e, q);
        }
        Lc[a] += s;
    }
    return ORC_OK;
}

/* L2P: Phi(c + dx) = sum_k L_k dx^k/k!,  a = -grad Phi = -sum_k L_{k+e_alpha} dx^k / k! (Taylor eq.) */
int orc_l2p(int p, const double *L, const double *dx, double *pot, double *acc)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    double phi = 0.0, g[3] = {0.0, 0.0, 0.0};
    for (int a = 0; a < nc; ++a) {
        const int *k = mi[a];
        double t = mono_over_fact(dx, k);
        phi += L[a] * t;
        if (k[0] + k[1] + k[2] < p)
            for (int al = 0; al < 3; ++al) {
                int q[3] = {k[0], k[1], k[2]};
                q[al] += 1;
                g[al] += L[orc_mindex(q[0], q[1], q[2])] * t;
            }
    }
    *pot += phi;
    acc[0] -= g[0]; acc[1] -= g[1]; acc[2] -= g[2];
    return ORC_OK;
}

/*
 * Dipole P2M (used by the VJP below): a source at x_j = c + s with monopole q and dipole d has the
 * potential -G (q + d . grad_{x_j}) 1/|y - x_j|, so its moments are
 *   M_n += q s^n / n! + sum_alpha d_alpha s^{n - e_alpha} / (n - e_alpha)!,
 * the position derivative of the point-mass moments in the direction d.
 */
int orc_p2m_dipole(int p, int64_t n, const double *pos, const double *q, const double *d, const double *c,
                   double *M)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    for (int64_t j = 0; j < n; ++j) {
        double s[3] = {pos[3 * j] - c[0], pos[3 * j + 1] - c[1], pos[3 * j + 2] - c[2]};
        for (int a = 0; a < nc; ++a) {
            const int *m = mi[a];
            double v = (q ? q[j] : 0.0) * mono_over_fact(s, m);
            for (int al = 0; al < 3; ++al) {
                if (m[al] < 1) continue;
                int r[3] = {m[0], m[1], m[2]};
                r[al] -= 1;
                v += d[3 * j + al] * mono_over_fact(s, r);
            }
            M[a] += v;
        }
    }
    return ORC_OK;
}

/* Hessian of the local series (the next derivative after L2P's gradient):
 *   d_alpha d_beta Phi(c + dx) = sum_{|k| <= p-2} L_{k + e_alpha + e_beta} dx^k / k!
 * added to H = (xx, xy, xz, yy, yz, zz). */
int orc_l2p_hess(int p, const double *L, const double *dx, double *H)
{
    if (p < 0 || p > ORC_MAXP) return ORC_EINVAL;
    int nc = orc_ncoef(p);
    int mi[ORC_NCMAX][3];
    mi_table(p, mi);
    static const int pa[6] = {0, 0, 0, 1, 1, 2}, pb[6] = {0, 1, 2, 1, 2, 2};
    for (int a = 0; a < nc; ++a) {
        const int *k = mi[a];
        if (k[0] + k[1] + k[2] > p - 2) continue;
        double t = mono_over_fact(dx, k);
        for (int h = 0; h < 6; ++h) {
            int q[3] = {k[0], k[1], k[2]};
            q[pa[h]] += 1;
            q[pb[h]] += 1;
            H[h] += L[orc_mindex(q[0], q[1], q[2])] * t;
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Morton keys (21 bits per axis, x most significant within each 3-bit digit) */
/* ------------------------------------------------------------------------ */

static uint64_t interleave3(uint32_t qx, uint32_t qy, uint32_t qz)
{
    uint64_t k = 0;
    for (int b = 0; b < ORC_KEY_BITS; ++b) {
        k |= (uint64_t)((qx >> b) & 1u) << (3 * b + 2);
        k |= (uint64_t)((qy >> b) & 1u) << (3 * b + 1);
        k |= (uint64_t)((qz >> b) & 1u) << (3 * b);
    }
    return k;
}

/* Root cube: origin = min corner, side = largest extent (1 if all points coincide).
 * q = min(floor(((x - xmin) / side) * 2^21), 2^21 - 1), each step rounded in the input precision. */
static int keys_f32(int64_t n, const float *pos, uint64_t *key, double *box)
{
    float lo[3], hi[3];
    for (int a = 0; a < 3; ++a) { lo[a] = pos[a]; hi[a] = pos[a]; }
    for (int64_t i = 0; i < n; ++i)
        for (int a = 0; a < 3; ++a) {
            float v = pos[3 * i + a];
            if (!isfinite(v)) return ORC_ENONFINITE;
            if (v < lo[a]) lo[a] = v;
            if (v > hi[a]) hi[a] = v;
        }
    float side = hi[0] - lo[0];
    for (int a = 1; a < 3; ++a) { float e = hi[a] - lo[a]; if (e > side) side = e; }
    if (!(side > 0.0f)) side = 1.0f;
    const float scale = 2097152.0f; /* 2^21 */
    for (int64_t i = 0; i < n; ++i) {
        uint32_t q[3];
        for (int a = 0; a < 3; ++a) {
            volatile float t = pos[3 * i + a] - lo[a];
            volatile float u = t / side;
            volatile float w = u * scale;
            float f = floorf(w);
            uint32_t qi = (uint32_t)f;
            q[a] = qi > 2097151u ? 2097151u : qi;
        }
        key[i] = interleave3(q[0], q[1], q[2]);
    }
    for (int a = 0; a < 3; ++a) { box[a] = lo[a]; box[3 + a] = hi[a]; }
    box[6] = side;
    return ORC_OK;
}

static int keys_f64(int64_t n, const double *pos, uint64_t *key, double *box)
{
    double lo[3], hi[3];
    for (int a = 0; a < 3; ++a) { lo[a] = pos[a]; hi[a] = pos[a]; }
    for (int64_t i = 0; i < n; ++i)
        for (int a = 0; a < 3; ++a) {
            double v = pos[3 * i + a];
            if (!isfinite(v)) return ORC_ENONFINITE;
            if (v < lo[a]) lo[a] = v;
            if (v > hi[a]) hi[a] = v;
        }
    double side = hi[0] - lo[0];
    for (int a = 1; a < 3; ++a) { double e = hi[a] - lo[a]; if (e > side) side = e; }
    if (!(side > 0.0)) side = 1.0;
    const double scale = 2097152.0;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t q[3];
        for (int a = 0; a < 3; ++a) {
            volatile double t = pos[3 * i + a] - lo[a];
            volatile double u = t / side;
            volatile double w = u * scale;
            double f = floor(w);
            uint32_t qi = (uint32_t)f;
            q[a] = qi > 2097151u ? 2097151u : qi;
        }
        key[i] = interleave3(q[0], q[1], q[2]);
    }
    for (int a = 0; a < 3; ++a) { box[a] = lo[a]; box[3 + a] = hi[a]; }
    box[6] = side;
    return ORC_OK;
}

int orc_keys(int dtype, int64_t n, const void *pos, uint64_t *key, double *box7)
{
    if (n < 1 || !pos || !key || !box7) return ORC_EINVAL;
    return dtype == ORC_DTYPE_F32 ? keys_f32(n, (const float *)pos, key, box7)
                                  : keys_f64(n, (const double *)pos, key, box7);
}

/* ------------------------------------------------------------------------ */
/* full evaluation                                                           */
/* ------------------------------------------------------------------------ */

typedef struct {
    int64_t n, n_nodes, n_leaves;
    int32_t depth, nc, p, leaf, dtype, pad;
    double theta;
    double box[7];                  /* root min corner, max corner, side */
    uint64_t *keys;                 /* [n] sorted Morton keys */
    int64_t *perm;                  /* [n] sorted slot -> original particle index */
    int64_t level_off[ORC_MAX_DEPTH + 2]; /* nodes of level l are [level_off[l], level_off[l+1]) */
    int32_t *first, *count, *child0, *nchild, *parent, *level; /* [n_nodes] */
    double *lo, *hi;                /* [n_nodes*3] tight particle box (exact input values) */
    double *centre, *half;          /* [n_nodes*3] c=(lo+hi)*0.5, l=(hi-lo)*0.5 in input precision */
    double *M;                      /* [n_nodes*nc] multipoles about centre */
    double *Lm2l;                   /* [n_nodes*nc] M2L contributions only */
    double *L;                      /* [n_nodes*nc] complete local expansions (after L2L) */
    int64_t n_m2l_pairs, n_p2p_pairs; /* unordered pairs from the walk (p2p incl. self pairs) */
    int64_t n_m2l, n_p2p;           /* directed list entries */
    int64_t *m2l_off; int32_t *m2l_src; /* CSR by receiver node [n_nodes+1], [n_m2l] */
    int64_t *p2p_off; int32_t *p2p_src; /* CSR by receiver node [n_nodes+1], [n_p2p] */
    int64_t n_p2p_interactions;     /* sum over directed P2P entries of |A|*|B| */
    double *acc, *pot;              /* [n*3], [n] in original particle order (NaN where not evaluated) */
    double t_stage[8];              /* seconds: keys+sort, tree, up, walk, m2l, down(l2l), leaf(l2p+p2p), total */
} orc_result;

typedef struct { uint64_t key; int64_t idx; } kv;
static int cmp_kv(const void *a, const void *b)
{
    const kv *x = a, *y = b;
    if (x->key < y->key) return -1;
    if (x->key > y->key) return 1;
    return (x->idx > y->idx) - (x->idx < y->idx);
}

typedef struct { int32_t r, s; } pr;
static int cmp_pr(const void *a, const void *b)
{
    const pr *x = a, *y = b;
    if (x->r != y->r) return (x->r > y->r) - (x->r < y->r);
    return (x->s > y->s) - (x->s < y->s);
}

typedef struct { pr *v; int64_t n, cap; } prvec;
static int prpush(prvec *a, int32_t r, int32_t s)
{
    if (a->n == a->cap) {
        int64_t nc = a->cap ? 2 * a->cap : 1024;
        pr *nv = realloc(a->v, sizeof(pr) * (size_t)nc);
        if (!nv) return ORC_ENOMEM;
        a->v = nv; a->cap = nc;
    }
    a->v[a->n].r = r; a->v[a->n].s = s; a->n++;
    return ORC_OK;
}

static double now_s(void)
{
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

void orc_result_free(orc_result *r)
{
    if (!r) return;
    free(r->keys); free(r->perm);
    free(r->first); free(r->count); free(r->child0); free(r->nchild); free(r->parent); free(r->level);
    free(r->lo); free(r->hi); free(r->centre); free(r->half);
    free(r->M); free(r->Lm2l); free(r->L);
    free(r->m2l_off); free(r->m2l_src); free(r->p2p_off); free(r->p2p_src);
    free(r->acc); free(r->pot);
    memset(r, 0, sizeof(*r));
}

/* Opening criterion (theta eq.), evaluated in the input precision without contraction.
 * Returns 1 when the pair is accepted for M2L. */
static int accept_f32(const float *cA, const float *lA, const float *cB, const float *lB, float th2)
{
    volatile float sx = lA[0] + lB[0], sy = lA[1] + lB[1], sz = lA[2] + lB[2];
    volatile float rx = cA[0] - cB[0], ry = cA[1] - cB[1], rz = cA[2] - cB[2];
    volatile float sxx = sx * sx, syy = sy * sy, szz = sz * sz;
    volatile float rxx = rx * rx, ryy = ry * ry, rzz = rz * rz;
    volatile float s2a = sxx + syy;
    volatile float s2 = s2a + szz;
    volatile float r2a = rxx + ryy;
    volatile float r2 = r2a + rzz;
    volatile float rhs = th2 * r2;
    return s2 < rhs;
}
static int accept_f64(const double *cA, const double *lA, const double *cB, const double *lB, double th2)
{
    volatile double sx = lA[0] + lB[0], sy = lA[1] + lB[1], sz = lA[2] + lB[2];
    volatile double rx = cA[0] - cB[0], ry = cA[1] - cB[1], rz = cA[2] - cB[2];
    volatile double sxx = sx * sx, syy = sy * sy, szz = sz * sz;
    volatile double rxx = rx * rx, ryy = ry * ry, rzz = rz * rz;
    volatile double s2a = sxx + syy;
    volatile double s2 = s2a + szz;
    volatile double r2a = rxx + ryy;
    volatile double r2 = r2a + rzz;
    volatile double rhs = th2 * r2;
    return s2 < rhs;
}
static float norm2_f32(const float *l)
{
    volatile float a = l[0] * l[0], b = l[1] * l[1], c = l[2] * l[2];
    volatile float s = a + b;
    volatile float t = s + c;
    return t;
}
static double norm2_f64(const double *l)
{
    volatile double a = l[0] * l[0], b = l[1] * l[1], c = l[2] * l[2];
    volatile double s = a + b;
    volatile double t = s + c;
    return t;
}

/*
 * One FMM evaluation.
 *   dtype     ORC_DTYPE_F32 (pos/mass are float) or ORC_DTYPE_F64 (double)
 *   pos,mass  [n*3], [n] in the caller's order
 *   eval_mask NULL (evaluate every particle) or [n] bytes, nonzero = evaluate that particle;
 *             the far field is then computed only on the nodes those particles need.
 *   skip_expansions  nonzero: stop after the walk (tree and lists only)
 */
int orc_fmm(int dtype, int64_t n, const void *pos_in, const void *mass_in, int p, double theta,
            int leaf, const uint8_t *eval_mask, int skip_expansions, int nthreads, orc_result *res)
{
    if (!res) return ORC_EINVAL;
    memset(res, 0, sizeof(*res));
    if (n < 1 || !pos_in || !mass_in || p < 0 || p > ORC_MAXP || !(theta > 0.0) || theta > 1.0 ||
        leaf < 1 || (dtype != ORC_DTYPE_F32 && dtype != ORC_DTYPE_F64))
        return ORC_EINVAL;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    int st = ORC_OK;
    const int nc = orc_ncoef(p);
    res->n = n; res->p = p; res->nc = nc; res->leaf = leaf; res->dtype = dtype; res->theta = theta;
    double t0 = now_s(), t1;

    /* widened copies of the inputs (exact for fp32) */
    double *X = malloc(sizeof(double) * 3 * (size_t)n), *Mass = malloc(sizeof(double) * (size_t)n);
    if (!X || !Mass) { free(X); free(Mass); return ORC_ENOMEM; }
    for (int64_t i = 0; i < 3 * n; ++i)
        X[i] = dtype == ORC_DTYPE_F32 ? (double)((const float *)pos_in)[i] : ((const double *)pos_in)[i];
    for (int64_t i = 0; i < n; ++i)
        Mass[i] = dtype == ORC_DTYPE_F32 ? (double)((const float *)mass_in)[i] : ((const double *)mass_in)[i];

    /* ---- keys and sort: stable order by key, ties by original index ---- */
    uint64_t *key = malloc(sizeof(uint64_t) * (size_t)n);
    kv *kvs = malloc(sizeof(kv) * (size_t)n);
    res->keys = malloc(sizeof(uint64_t) * (size_t)n);
    res->perm = malloc(sizeof(int64_t) * (size_t)n);
    if (!key || !kvs || !res->keys || !res->perm) { st = ORC_ENOMEM; goto fail0; }
    st = orc_keys(dtype, n, pos_in, key, res->box);
    if (st) goto fail0;
    for (int64_t i = 0; i < n; ++i) { kvs[i].key = key[i]; kvs[i].idx = i; }
    qsort(kvs, (size_t)n, sizeof(kv), cmp_kv);
    for (int64_t i = 0; i < n; ++i) { res->keys[i] = kvs[i].key; res->perm[i] = kvs[i].idx; }
    free(kvs); kvs = NULL; free(key); key = NULL;
    /* sorted particle arrays */
    double *xs = malloc(sizeof(double) * 3 * (size_t)n), *ms = malloc(sizeof(double) * (size_t)n);
    if (!xs || !ms) { free(xs); free(ms); st = ORC_ENOMEM; goto fail0; }
    for (int64_t i = 0; i < n; ++i) {
        int64_t o = res->perm[i];
        xs[3 * i] = X[3 * o]; xs[3 * i + 1] = X[3 * o + 1]; xs[3 * i + 2] = X[3 * o + 2];
        ms[i] = Mass[o];
    }
    t1 = now_s(); res->t_stage[0] = t1 - t0; t0 = t1;

    /* ---- octree, breadth first: level by level, each level in key order ---- */
    int64_t cap = 1024, nn = 1;
    int32_t *first = malloc(sizeof(int32_t) * cap), *count = malloc(sizeof(int32_t) * cap);
    int32_t *child0 = malloc(sizeof(int32_t) * cap), *nchild = malloc(sizeof(int32_t) * cap);
    int32_t *parent = malloc(sizeof(int32_t) * cap), *level = malloc(sizeof(int32_t) * cap);
    if (!first || !count || !child0 || !nchild || !parent || !level) { st = ORC_ENOMEM; goto fail1; }
    first[0] = 0; count[0] = (int32_t)n; parent[0] = -1; level[0] = 0; child0[0] = -1; nchild[0] = 0;
    res->level_off[0] = 0;
    int64_t lb = 0, le = 1; /* current level's node range */
    int depth = 0;
    for (int l = 0; l <= ORC_MAX_DEPTH; ++l) {
        res->level_off[l + 1] = le;
        if (l == ORC_MAX_DEPTH) break;
        int64_t added = 0;
        for (int64_t a = lb; a < le; ++a) {
            child0[a] = -1; nchild[a] = 0;
            if (count[a] <= leaf) continue; /* leaf: count <= L */
            int shift = 3 * (ORC_MAX_DEPTH - (l + 1));
            int64_t i = first[a], end = (int64_t)first[a] + count[a];
            while (i < end) {
                uint64_t dig = (res->keys[i] >> shift) & 7u;
                int64_t j = i;
                while (j < end && ((res->keys[j] >> shift) & 7u) == dig) ++j;
                if (nn == cap) {
                    cap *= 2;
                    int32_t **arrs[6] = {&first, &count, &child0, &nchild, &parent, &level};
                    for (int q = 0; q < 6; ++q) {
                        int32_t *t = realloc(*arrs[q], sizeof(int32_t) * (size_t)cap);
                        if (!t) { st = ORC_ENOMEM; goto fail1; }
                        *arrs[q] = t;
                    }
                }
                if (nchild[a] == 0) child0[a] = (int32_t)nn;
                nchild[a]++;
                first[nn] = (int32_t)i; count[nn] = (int32_t)(j - i); parent[nn] = (int32_t)a;
                level[nn] = l + 1; child0[nn] = -1; nchild[nn] = 0;
                nn++; added++;
                i = j;
            }
        }
        if (added == 0) {
            for (int q = l + 2; q <= ORC_MAX_DEPTH + 1; ++q) res->level_off[q] = le;
            break;
        }
        depth = l + 1;
        lb = le; le = nn;
    }
    res->n_nodes = nn; res->depth = depth;
    res->first = first; res->count = count; res->child0 = child0; res->nchild = nchild;
    res->parent = parent; res->level = level;
    first = count = child0 = nchild = parent = level = NULL;
    int64_t nleaves = 0;
    for (int64_t a = 0; a < nn; ++a) nleaves += res->nchild[a] == 0;
    res->n_leaves = nleaves;

    /* ---- node boxes, centres and half-widths (criterion eq.: c centre, l half-width per axis) ---- */
    res->lo = malloc(sizeof(double) * 3 * (size_t)nn); res->hi = malloc(sizeof(double) * 3 * (size_t)nn);
    res->centre = malloc(sizeof(double) * 3 * (size_t)nn); res->half = malloc(sizeof(double) * 3 * (size_t)nn);
    if (!res->lo || !res->hi || !res->centre || !res->half) { st = ORC_ENOMEM; goto fail1; }
    for (int64_t a = 0; a < nn; ++a) {
        for (int d = 0; d < 3; ++d) {
            double lo = xs[3 * (int64_t)res->first[a] + d], hi = lo;
            for (int64_t i = res->first[a]; i < (int64_t)res->first[a] + res->count[a]; ++i) {
                double v = xs[3 * i + d];
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            res->lo[3 * a + d] = lo; res->hi[3 * a + d] = hi;
            if (dtype == ORC_DTYPE_F32) {
                volatile float s = (float)lo + (float)hi, w = (float)hi - (float)lo;
                volatile float c = s * 0.5f, h = w * 0.5f;
                res->centre[3 * a + d] = c; res->half[3 * a + d] = h;
            } else {
                volatile double s = lo + hi, w = hi - lo;
                volatile double c = s * 0.5, h = w * 0.5;
                res->centre[3 * a + d] = c; res->half[3 * a + d] = h;
            }
        }
    }
    t1 = now_s(); res->t_stage[1] = t1 - t0; t0 = t1;

    /* ---- stage 1 (upward): P2M at the leaves, M2M from children to parents ---- */
    if (!skip_expansions) {
        res->M = calloc((size_t)nn * nc, sizeof(double));
        if (!res->M) { st = ORC_ENOMEM; goto fail1; }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
        for (int64_t a = 0; a < nn; ++a)
            if (res->nchild[a] == 0)
                orc_p2m(p, res->count[a], xs + 3 * (int64_t)res->first[a], ms + res->first[a],
                        res->centre + 3 * a, res->M + a * nc);
        for (int l = depth - 1; l >= 0; --l) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
            for (int64_t a = res->level_off[l]; a < res->level_off[l + 1]; ++a)
                for (int c = 0; c < res->nchild[a]; ++c) {
                    int64_t ch = res->child0[a] + c;
                    double d[3] = {res->centre[3 * ch] - res->centre[3 * a],
                                   res->centre[3 * ch + 1] - res->centre[3 * a + 1],
                                   res->centre[3 * ch + 2] - res->centre[3 * a + 2]};
                    orc_m2m(p, res->M + ch * nc, d, res->M + a * nc);
                }
        }
    }
    t1 = now_s(); res->t_stage[2] = t1 - t0; t0 = t1;

    /* ---- stage 2: dual-tree walk from the pair (root, root) ---- */
    {
        prvec stack = {0}, m2l = {0}, p2p = {0};
        float th2f = (float)(theta * theta);
        double th2d = theta * theta;
        float *cf = NULL, *lf = NULL;
        if (dtype == ORC_DTYPE_F32) {
            cf = malloc(sizeof(float) * 3 * (size_t)nn); lf = malloc(sizeof(float) * 3 * (size_t)nn);
            if (!cf || !lf) { free(cf); free(lf); st = ORC_ENOMEM; goto fail1; }
            for (int64_t q = 0; q < 3 * nn; ++q) { cf[q] = (float)res->centre[q]; lf[q] = (float)res->half[q]; }
        }
        st = prpush(&stack, 0, 0);
        while (!st && stack.n > 0) {
            pr top = stack.v[--stack.n];
            int32_t A = top.r, B = top.s; /* A <= B */
            int leafA = res->nchild[A] == 0, leafB = res->nchild[B] == 0;
            if (A == B) {
                if (leafA) { st = prpush(&p2p, A, A); continue; }
                for (int i = 0; i < res->nchild[A] && !st; ++i)
                    for (int j = i; j < res->nchild[A] && !st; ++j)
                        st = prpush(&stack, res->child0[A] + i, res->child0[A] + j);
                continue;
            }
            int acc_ok = dtype == ORC_DTYPE_F32
                ? accept_f32(cf + 3 * A, lf + 3 * A, cf + 3 * B, lf + 3 * B, th2f)
                : accept_f64(res->centre + 3 * A, res->half + 3 * A, res->centre + 3 * B, res->half + 3 * B, th2d);
            if (acc_ok) { st = prpush(&m2l, A, B); continue; }
            if (leafA && leafB) { st = prpush(&p2p, A, B); continue; }
            int splitA;
            if (leafA) splitA = 0;
            else if (leafB) splitA = 1;
            else if (dtype == ORC_DTYPE_F32) splitA = norm2_f32(lf + 3 * A) >= norm2_f32(lf + 3 * B);
            else splitA = norm2_f64(res->half + 3 * A) >= norm2_f64(res->half + 3 * B);
            int32_t S = splitA ? A : B, O = splitA ? B : A;
            for (int i = 0; i < res->nchild[S] && !st; ++i) {
                int32_t C = res->child0[S] + i;
                st = prpush(&stack, C < O ? C : O, C < O ? O : C);
            }
        }
        free(stack.v); free(cf); free(lf);
        if (st) { free(m2l.v); free(p2p.v); goto fail1; }
        res->n_m2l_pairs = m2l.n; res->n_p2p_pairs = p2p.n;
        /* directed lists, then canonical order (receiver, source) and CSR */
        prvec dm = {0}, dp = {0};
        for (int64_t q = 0; q < m2l.n && !st; ++q) {
            st = prpush(&dm, m2l.v[q].r, m2l.v[q].s);
            if (!st) st = prpush(&dm, m2l.v[q].s, m2l.v[q].r);
        }
        for (int64_t q = 0; q < p2p.n && !st; ++q) {
            st = prpush(&dp, p2p.v[q].r, p2p.v[q].s);
            if (!st && p2p.v[q].r != p2p.v[q].s) st = prpush(&dp, p2p.v[q].s, p2p.v[q].r);
        }
        free(m2l.v); free(p2p.v);
        if (st) { free(dm.v); free(dp.v); goto fail1; }
        if (dm.n) qsort(dm.v, (size_t)dm.n, sizeof(pr), cmp_pr);
        if (dp.n) qsort(dp.v, (size_t)dp.n, sizeof(pr), cmp_pr);
        res->n_m2l = dm.n; res->n_p2p = dp.n;
        res->m2l_off = calloc((size_t)nn + 1, sizeof(int64_t));
        res->p2p_off = calloc((size_t)nn + 1, sizeof(int64_t));
        res->m2l_src = malloc(sizeof(int32_t) * (size_t)(dm.n ? dm.n : 1));
        res->p2p_src = malloc(sizeof(int32_t) * (size_t)(dp.n ? dp.n : 1));
        if (!res->m2l_off || !res->p2p_off || !res->m2l_src || !res->p2p_src) {
            free(dm.v); free(dp.v); st = ORC_ENOMEM; goto fail1;
        }
        for (int64_t q = 0; q < dm.n; ++q) { res->m2l_off[dm.v[q].r + 1]++; res->m2l_src[q] = dm.v[q].s; }
        for (int64_t q = 0; q < dp.n; ++q) {
            res->p2p_off[dp.v[q].r + 1]++; res->p2p_src[q] = dp.v[q].s;
            res->n_p2p_interactions += (int64_t)res->count[dp.v[q].r] * res->count[dp.v[q].s];
        }
        for (int64_t a = 0; a < nn; ++a) { res->m2l_off[a + 1] += res->m2l_off[a]; res->p2p_off[a + 1] += res->p2p_off[a]; }
        free(dm.v); free(dp.v);
    }
    t1 = now_s(); res->t_stage[3] = t1 - t0; t0 = t1;
    if (skip_expansions) goto done;

    /* which nodes must be evaluated: all, or the ancestors of the masked particles' leaves */
    uint8_t *need = calloc((size_t)nn, 1);
    int64_t *leaf_of = malloc(sizeof(int64_t) * (size_t)n);
    if (!need || !leaf_of) { free(need); free(leaf_of); st = ORC_ENOMEM; goto fail1; }
    for (int64_t a = 0; a < nn; ++a)
        if (res->nchild[a] == 0)
            for (int64_t i = res->first[a]; i < (int64_t)res->first[a] + res->count[a]; ++i) leaf_of[i] = a;
    for (int64_t i = 0; i < n; ++i) {
        if (eval_mask && !eval_mask[res->perm[i]]) continue;
        for (int64_t a = leaf_of[i]; a >= 0 && !need[a]; a = res->parent[a]) need[a] = 1;
    }

    /* ---- M2L: L_A += M2L(M_B, c_A - c_B) over A's sources, in list order ---- */
    res->Lm2l = calloc((size_t)nn * nc, sizeof(double));
    res->L = calloc((size_t)nn * nc, sizeof(double));
    if (!res->Lm2l || !res->L) { free(need); free(leaf_of); st = ORC_ENOMEM; goto fail1; }
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t a = 0; a < nn; ++a) {
        if (!need[a]) continue;
        for (int64_t q = res->m2l_off[a]; q < res->m2l_off[a + 1]; ++q) {
            int64_t b = res->m2l_src[q];
            double R[3] = {res->centre[3 * a] - res->centre[3 * b], res->centre[3 * a + 1] - res->centre[3 * b + 1],
                           res->centre[3 * a + 2] - res->centre[3 * b + 2]};
            orc_m2l(p, res->M + b * nc, R, res->Lm2l + a * nc);
        }
    }
    t1 = now_s(); res->t_stage[4] = t1 - t0; t0 = t1;

    /* ---- stage 3 (downward): L2L parent -> child, level by level ---- */
    for (int64_t a = 0; a < nn; ++a) {
        if (!need[a]) continue;
        double *La = res->L + a * nc;
        int64_t par = res->parent[a];
        if (par >= 0) {
            double e[3] = {res->centre[3 * a] - res->centre[3 * par], res->centre[3 * a + 1] - res->centre[3 * par + 1],
                           res->centre[3 * a + 2] - res->centre[3 * par + 2]};
            orc_l2l(p, res->L + par * nc, e, La);
        }
        for (int c = 0; c < nc; ++c) La[c] += res->Lm2l[a * nc + c];
    }
    t1 = now_s(); res->t_stage[5] = t1 - t0; t0 = t1;

    /* ---- leaves: L2P plus direct P2P with every source leaf in the list ---- */
    res->acc = malloc(sizeof(double) * 3 * (size_t)n);
    res->pot = malloc(sizeof(double) * (size_t)n);
    if (!res->acc || !res->pot) { free(need); free(leaf_of); st = ORC_ENOMEM; goto fail1; }
    for (int64_t i = 0; i < 3 * n; ++i) res->acc[i] = NAN;
    for (int64_t i = 0; i < n; ++i) res->pot[i] = NAN;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t a = 0; a < nn; ++a) {
        if (!need[a] || res->nchild[a] != 0) continue;
        for (int64_t i = res->first[a]; i < (int64_t)res->first[a] + res->count[a]; ++i) {
            int64_t o = res->perm[i];
            if (eval_mask && !eval_mask[o]) continue;
            double phi = 0.0, g[3] = {0.0, 0.0, 0.0};
            double dx[3] = {xs[3 * i] - res->centre[3 * a], xs[3 * i + 1] - res->centre[3 * a + 1],
                            xs[3 * i + 2] - res->centre[3 * a + 2]};
            orc_l2p(p, res->L + a * nc, dx, &phi, g);
            for (int64_t q = res->p2p_off[a]; q < res->p2p_off[a + 1]; ++q) {
                int64_t b = res->p2p_src[q];
                for (int64_t j = res->first[b]; j < (int64_t)res->first[b] + res->count[b]; ++j) {
                    double rx = xs[3 * j] - xs[3 * i], ry = xs[3 * j + 1] - xs[3 * i + 1], rz = xs[3 * j + 2] - xs[3 * i + 2];
                    double r2 = rx * rx + ry * ry + rz * rz;
                    if (r2 == 0.0) continue;
                    double r = sqrt(r2);
                    double mr3 = ms[j] / (r2 * r);
                    g[0] += mr3 * rx; g[1] += mr3 * ry; g[2] += mr3 * rz;
                    phi -= ms[j] / r;
                }
            }
            res->acc[3 * o] = g[0]; res->acc[3 * o + 1] = g[1]; res->acc[3 * o + 2] = g[2];
            res->pot[o] = phi;
        }
    }
    free(need); free(leaf_of);
    t1 = now_s(); res->t_stage[6] = t1 - t0; t0 = t1;

done:
    for (int q = 0; q < 7; ++q) res->t_stage[7] += res->t_stage[q];
    free(xs); free(ms); free(X); free(Mass);
    return ORC_OK;

fail1:
    free(first); free(count); free(child0); free(nchild); free(parent); free(level);
    free(xs); free(ms);
fail0:
    free(kvs); free(key); free(X); free(Mass);
    orc_result_free(res);
    return st;
}

/*
 * Kick-drift-kick leapfrog (Jaxion `_update`: half kick, full drift, half kick),
 * with the force from orc_fmm. `acc` holds a(x) on entry and a(x_new) on exit,
 * all in fp64. Returns the status of the force evaluation.
 */
int orc_kdk_step(int64_t n, double *pos, double *vel, const double *mass, double *acc, double dt,
                 int p, double theta, int leaf, int nthreads)
{
    for (int64_t i = 0; i < 3 * n; ++i) vel[i] += acc[i] * (0.5 * dt);
    for (int64_t i = 0; i < 3 * n; ++i) pos[i] += vel[i] * dt;
    orc_result r;
    int st = orc_fmm(ORC_DTYPE_F64, n, pos, mass, p, theta, leaf, NULL, 0, nthreads, &r);
    if (st) return st;
    memcpy(acc, r.acc, sizeof(double) * 3 * (size_t)n);
    orc_result_free(&r);
    for (int64_t i = 0; i < 3 * n; ++i) vel[i] += acc[i] * (0.5 * dt);
    return ORC_OK;
}

/*
 * Kick-drift-kick on an integer lattice (JZ-FMM page, "Why reversibility
 * matters": positions and velocities live on a lattice, the force stays
 * floating point, reversing an update subtracts the same increment).
 * Lattice spacings are 2^pos_exp and 2^vel_exp; every increment is rounded to
 * its lattice (round half to even, symmetric in the sign of dt), so a step
 * with -dt undoes a step with dt exactly when the force at a revisited state
 * is reproduced bit for bit. pos and vel are first rounded to their lattices
 * (a no-op once they lie on them). `acc` holds a(x) on entry, a(x_new) on exit.
 */
static double to_lattice(double y, double inv_spacing, double spacing) { return nearbyint(y * inv_spacing) * spacing; }

int orc_kdk_lattice_step(int64_t n, double *pos, double *vel, const double *mass, double *acc, double dt,
                         int pos_exp, int vel_exp, int p, double theta, int leaf, int nthreads)
{
    const double dx = ldexp(1.0, pos_exp), idx = ldexp(1.0, -pos_exp);
    const double dv = ldexp(1.0, vel_exp), idv = ldexp(1.0, -vel_exp);
    const double h = 0.5 * dt;
    for (int64_t i = 0; i < 3 * n; ++i) { pos[i] = to_lattice(pos[i], idx, dx); vel[i] = to_lattice(vel[i], idv, dv); }
    for (int64_t i = 0; i < 3 * n; ++i) vel[i] += to_lattice(acc[i] * h, idv, dv);
    for (int64_t i = 0; i < 3 * n; ++i) pos[i] += to_lattice(vel[i] * dt, idx, dx);
    orc_result r;
    int st = orc_fmm(ORC_DTYPE_F64, n, pos, mass, p, theta, leaf, NULL, 0, nthreads, &r);
    if (st) return st;
    memcpy(acc, r.acc, sizeof(double) * 3 * (size_t)n);
    orc_result_free(&r);
    for (int64_t i = 0; i < 3 * n; ++i) vel[i] += to_lattice(acc[i] * h, idv, dv);
    return ORC_OK;
}

/*
 * Vector-Jacobian product of one FMM evaluation (JZ-FMM page, "Differentiating the force
 * calculation": one contribution comes from the next higher derivative in the original evaluation,
 * the other from an FMM in which the force sensitivities act as dipole moments).
 *
 * Given cotangents abar_i of the accelerations and (optionally, NULL = 0) pbar_i of the potentials,
 * with the loss sensitivity sum_i abar_i . a_i + pbar_i phi_i, it returns
 *   xbar_k = m_k grad Phi_s(x_k) - Hess Phi(x_k) abar_k - pbar_k a_k,     mbar_k = Phi_s(x_k),
 * where Phi is the forward potential (its Hessian: L2P one order higher, plus the direct term of
 * every near pair) and Phi_s the potential of sources at every particle with monopole pbar_j and
 * dipole -abar_j,
 *   Phi_s(y) = -G sum_{j} [pbar_j / |y - x_j| - abar_j . (y - x_j) / |y - x_j|^3]   (r = 0 skipped),
 * evaluated by the same tree, centres, p, theta and lists as the forward evaluation (dipole P2M,
 * then the forward M2M, M2L, L2L and L2P, plus the direct near field). Why: with the centres and
 * lists fixed, the evaluation is a_i = -grad_{x_i} sum_k m_k K(x_i, x_k) with a pair kernel K that
 * is symmetric in its two particles (the total-degree truncation; D^m(-R) = (-1)^{|m|} D^m(R)),
 * so the derivative through a source's moments is the dipole FMM, and the derivative through the
 * evaluation point is the Hessian of the forward potential. These are therefore the exact
 * derivatives of the evaluation with the tree and the expansion centres held fixed.
 *
 * pos, mass in dtype (fp32 inputs are widened exactly); abar [n*3], pbar [n] or NULL, and the
 * outputs pos_bar [n*3], mass_bar [n] are fp64 in the caller's order.
 */
int orc_fmm_vjp(int dtype, int64_t n, const void *pos_in, const void *mass_in, const double *abar,
                const double *pbar, int p, double theta, int leaf, int nthreads, double *pos_bar, double *mass_bar)
{
    if (!abar || !pos_bar || !mass_bar) return ORC_EINVAL;
    orc_result r;
    int st = orc_fmm(dtype, n, pos_in, mass_in, p, theta, leaf, NULL, 0, nthreads, &r);
    if (st) return st;
    const int64_t nn = r.n_nodes;
    const int nc = r.nc;
    double *xs = malloc(sizeof(double) * 3 * (size_t)n), *ms = malloc(sizeof(double) * (size_t)n);
    double *as = malloc(sizeof(double) * 3 * (size_t)n), *qs = malloc(sizeof(double) * (size_t)n);
    double *ds = malloc(sizeof(double) * 3 * (size_t)n);
    double *Ms = calloc((size_t)nn * nc, sizeof(double)), *Lsm = calloc((size_t)nn * nc, sizeof(double));
    double *Ls = calloc((size_t)nn * nc, sizeof(double));
    if (!xs || !ms || !as || !qs || !ds || !Ms || !Lsm || !Ls) { st = ORC_ENOMEM; goto out; }
    /* sorted copies: positions, masses, cotangents; the dipole of particle j is -abar_j */
    for (int64_t i = 0; i < n; ++i) {
        int64_t o = r.perm[i];
        for (int d = 0; d < 3; ++d) {
            xs[3 * i + d] = dtype == ORC_DTYPE_F32 ? (double)((const float *)pos_in)[3 * o + d]
                                                   : ((const double *)pos_in)[3 * o + d];
            as[3 * i + d] = abar[3 * o + d];
            ds[3 * i + d] = -abar[3 * o + d];
        }
        ms[i] = dtype == ORC_DTYPE_F32 ? (double)((const float *)mass_in)[o] : ((const double *)mass_in)[o];
        qs[i] = pbar ? pbar[o] : 0.0;
    }
    /* source FMM, upward: dipole P2M at the leaves, M2M to the parents (same centres) */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
    for (int64_t a = 0; a < nn; ++a)
        if (r.nchild[a] == 0)
            orc_p2m_dipole(p, r.count[a], xs + 3 * (int64_t)r.first[a], qs + r.first[a], ds + 3 * (int64_t)r.first[a],
                           r.centre + 3 * a, Ms + a * nc);
    for (int l = r.depth - 1; l >= 0; --l) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 64)
#endif
        for (int64_t a = r.level_off[l]; a < r.level_off[l + 1]; ++a)
            for (int c = 0; c < r.nchild[a]; ++c) {
                int64_t ch = r.child0[a] + c;
                double dd[3] = {r.centre[3 * ch] - r.centre[3 * a], r.centre[3 * ch + 1] - r.centre[3 * a + 1],
                                r.centre[3 * ch + 2] - r.centre[3 * a + 2]};
                orc_m2m(p, Ms + ch * nc, dd, Ms + a * nc);
            }
    }
    /* M2L over the forward lists */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t a = 0; a < nn; ++a)
        for (int64_t q = r.m2l_off[a]; q < r.m2l_off[a + 1]; ++q) {
            int64_t b = r.m2l_src[q];
            double R[3] = {r.centre[3 * a] - r.centre[3 * b], r.centre[3 * a + 1] - r.centre[3 * b + 1],
                           r.centre[3 * a + 2] - r.centre[3 * b + 2]};
            orc_m2l(p, Ms + b * nc, R, Lsm + a * nc);
        }
    /* L2L, parents before children */
    for (int64_t a = 0; a < nn; ++a) {
        int64_t par = r.parent[a];
        if (par >= 0) {
            double e[3] = {r.centre[3 * a] - r.centre[3 * par], r.centre[3 * a + 1] - r.centre[3 * par + 1],
                           r.centre[3 * a + 2] - r.centre[3 * par + 2]};
            orc_l2l(p, Ls + par * nc, e, Ls + a * nc);
        }
        for (int c = 0; c < nc; ++c) Ls[a * nc + c] += Lsm[a * nc + c];
    }
    /* leaves: far parts from the local series, near parts over the P2P lists */
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 16)
#endif
    for (int64_t a = 0; a < nn; ++a) {
        if (r.nchild[a] != 0) continue;
        for (int64_t i = r.first[a]; i < (int64_t)r.first[a] + r.count[a]; ++i) {
            int64_t o = r.perm[i];
            double dx[3] = {xs[3 * i] - r.centre[3 * a], xs[3 * i + 1] - r.centre[3 * a + 1],
                            xs[3 * i + 2] - r.centre[3 * a + 2]};
            double phis = 0.0, ngs[3] = {0.0, 0.0, 0.0}, H[6] = {0, 0, 0, 0, 0, 0};
            orc_l2p(p, Ls + a * nc, dx, &phis, ngs);      /* Phi_s and -grad Phi_s */
            orc_l2p_hess(p, r.L + a * nc, dx, H);         /* Hessian of the forward potential */
            double gs[3] = {-ngs[0], -ngs[1], -ngs[2]};
            for (int64_t q = r.p2p_off[a]; q < r.p2p_off[a + 1]; ++q) {
                int64_t b = r.p2p_src[q];
                for (int64_t j = r.first[b]; j < (int64_t)r.first[b] + r.count[b]; ++j) {
                    double u[3] = {xs[3 * i] - xs[3 * j], xs[3 * i + 1] - xs[3 * j + 1], xs[3 * i + 2] - xs[3 * j + 2]};
                    double r2 = u[0] * u[0] + u[1] * u[1] + u[2] * u[2];
                    if (r2 == 0.0) continue;
                    double rr = sqrt(r2), ir3 = 1.0 / (r2 * rr), ir5 = ir3 / r2;
                    /* forward: Phi += -m_j / r, Hessian m_j (r^2 delta - 3 u u) / r^5 */
                    H[0] += ms[j] * (r2 - 3.0 * u[0] * u[0]) * ir5;
                    H[1] += ms[j] * (-3.0 * u[0] * u[1]) * ir5;
                    H[2] += ms[j] * (-3.0 * u[0] * u[2]) * ir5;
                    H[3] += ms[j] * (r2 - 3.0 * u[1] * u[1]) * ir5;
                    H[4] += ms[j] * (-3.0 * u[1] * u[2]) * ir5;
                    H[5] += ms[j] * (r2 - 3.0 * u[2] * u[2]) * ir5;
                    /* sources: Phi_s += -q_j / r - d_j . u / r^3 and its gradient
                       q_j u / r^3 - d_j / r^3 + 3 (d_j . u) u / r^5 */
                    const double *dj = ds + 3 * j;
                    double du = dj[0] * u[0] + dj[1] * u[1] + dj[2] * u[2];
                    phis += -qs[j] / rr - du * ir3;
                    for (int d = 0; d < 3; ++d) gs[d] += qs[j] * u[d] * ir3 - dj[d] * ir3 + 3.0 * du * u[d] * ir5;
                }
            }
            const double *ab = as + 3 * i;
            double Ha[3] = {H[0] * ab[0] + H[1] * ab[1] + H[2] * ab[2], H[1] * ab[0] + H[3] * ab[1] + H[4] * ab[2],
                            H[2] * ab[0] + H[4] * ab[1] + H[5] * ab[2]};
            for (int d = 0; d < 3; ++d) pos_bar[3 * o + d] = ms[i] * gs[d] - Ha[d] - qs[i] * r.acc[3 * o + d];
            mass_bar[o] = phis;
        }
    }
out:
    free(xs); free(ms); free(as); free(qs); free(ds); free(Ms); free(Lsm); free(Ls);
    orc_result_free(&r);
    return st;
}
