/*
 * nbody_oracle.c -- the oracle for the all-pairs softened gravity path.
 *
 * TEST INFRASTRUCTURE ONLY. This is the slow, plain CPU statement of what the
 * CUDA library computes. The test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it; the library never does, and the two share no code,
 * header, table or helper.
 *
 * What it computes (G = 1):
 *
 *   a_i =  sum_j m_j (x_j - x_i) / (|x_j - x_i|^2 + eps^2)^(3/2)
 *   p_i = -sum_j m_j             / (|x_j - x_i|^2 + eps^2)^(1/2)
 *
 *   - The acceleration is the softened law of the "N体問題" lecture slides
 *     (Nagaoka), slide 4 (equation of motion) and slide 12 (the softening
 *     factor replaces the i != j branch); the same pair term is
 *     bodyBodyInteraction in the "Cuda Nbody笔记" notes and section 1 of the
 *     GPU Gems 3 ch.31 study page ("Fast N-Body Simulation with CUDA").
 *   - The potential is the second quantity of the "ATI Stream SDK による天文物理
 *     計算の高速化" slides (Aizu), slide No.4; its minus sign is lost in the
 *     extraction and is restored (a bound system has negative potential).
 *   - The sum runs over EVERY source j, the target itself included, with no
 *     branch: that is the point of slide 12.  The self term adds exactly 0 to
 *     a_i (its numerator is 0) and -m_i/eps to p_i, as the branch-free IL loop
 *     of the Aizu slides (No.7, No.9, softening kept in the dp4 fourth lane)
 *     also does.
 *   - r_ij = x_j - x_i points from the target to the source (the lecture's
 *     kernel code, and section 1 of the study page), so a_i is attractive.
 *
 * Arithmetic: the fp32 inputs are widened to fp64 exactly, every operation is
 * fp64, 1/sqrt comes from the host libm, and the sum runs over j in index
 * order.  Nothing is blocked, fused or reordered.
 *
 * The Euler step is the lecture's integrate() (slides 6 and 15, where the
 * positions are advanced before the velocities): x <- x + dt*v with the OLD
 * v, then v <- v + dt*a.  The pages compute it in fp32; here every product and sum is
 * rounded to fp32 separately (the file is compiled with -ffp-contract=off).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Number of OpenMP threads a call with nthreads <= 0 uses. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Target/source form of the definition above.
 *
 *   targets : nt bodies, 4 floats each (x, y, z, w); w is not read.
 *   sources : ns bodies, 4 floats each (x, y, z, m).
 *   eps2    : the softening eps^2 exactly as the fp32 library receives it.
 *   out     : nt rows of 4 doubles (ax, ay, az, p).
 *   nthreads: OpenMP threads over targets (<= 0: the OpenMP default).
 *
 * The all-pairs evaluation is the case where the targets are (rows of) the
 * sources themselves.  Returns 0, or -1 on a bad argument.
 */
int oracle_forces_ts(const float *targets, int64_t nt,
                     const float *sources, int64_t ns,
                     float eps2, double *out, int nthreads)
{
    if (nt < 0 || ns < 0) return -1;
    if ((nt > 0 && (targets == NULL || out == NULL)) || (ns > 0 && sources == NULL))
        return -1;
    const double e2 = (double)eps2;
#ifdef _OPENMP
    int nth = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(nth)
#else
    (void)nthreads;
#endif
    for (int64_t t = 0; t < nt; ++t) {
        const double xi = (double)targets[4 * t + 0];
        const double yi = (double)targets[4 * t + 1];
        const double zi = (double)targets[4 * t + 2];
        double ax = 0.0, ay = 0.0, az = 0.0, p = 0.0;
        for (int64_t j = 0; j < ns; ++j) {
            const double rx = (double)sources[4 * j + 0] - xi;
            const double ry = (double)sources[4 * j + 1] - yi;
            const double rz = (double)sources[4 * j + 2] - zi;
            const double mj = (double)sources[4 * j + 3];
            const double d2 = rx * rx + ry * ry + rz * rz + e2;   /* |r|^2 + eps^2 */
            const double inv = 1.0 / sqrt(d2);                    /* (|r|^2+eps^2)^(-1/2) */
            const double s = mj * inv * inv * inv;                /* m_j (|r|^2+eps^2)^(-3/2) */
            ax += s * rx;
            ay += s * ry;
            az += s * rz;
            p -= mj * inv;
        }
        out[4 * t + 0] = ax;
        out[4 * t + 1] = ay;
        out[4 * t + 2] = az;
        out[4 * t + 3] = p;
    }
    return 0;
}

/*
 * The same definition with fp64 bodies: all-pairs over n bodies whose
 * positions and masses are doubles, for the fp64 reference trajectory (an
 * Euler integration kept in fp64 throughout).  On bodies that fp32 holds
 * exactly it gives the same bits as oracle_forces_ts with targets ==
 * sources, the same arithmetic in the same order.
 *
 *   bodies  : n bodies, 4 doubles each (x, y, z, m).
 *   eps2    : the softening eps^2.
 *   out     : n rows of 4 doubles (ax, ay, az, p).
 *
 * Returns 0, or -1 on a bad argument.
 */
int oracle_forces_f64(const double *bodies, int64_t n, double eps2, double *out, int nthreads)
{
    if (n < 0) return -1;
    if (n > 0 && (bodies == NULL || out == NULL)) return -1;
#ifdef _OPENMP
    int nth = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 8) num_threads(nth)
#else
    (void)nthreads;
#endif
    for (int64_t i = 0; i < n; ++i) {
        const double *b = bodies + 4 * i;
        double sx = 0.0, sy = 0.0, sz = 0.0, pot = 0.0;
        for (int64_t q = 0; q < n; ++q) {
            const double *src = bodies + 4 * q;
            const double dx = src[0] - b[0];
            const double dy = src[1] - b[1];
            const double dz = src[2] - b[2];
            const double m = src[3];
            const double dd = dx * dx + dy * dy + dz * dz + eps2;   /* |r|^2 + eps^2 */
            const double w = 1.0 / sqrt(dd);
            const double k = m * w * w * w;                        /* m (|r|^2 + eps^2)^(-3/2) */
            sx += k * dx;
            sy += k * dy;
            sz += k * dz;
            pot -= m * w;
        }
        out[4 * i + 0] = sx;
        out[4 * i + 1] = sy;
        out[4 * i + 2] = sz;
        out[4 * i + 3] = pot;
    }
    return 0;
}

/*
 * Explicit Euler step in fp32, in place.
 *
 *   pos_mass: n bodies (x, y, z, m); x, y, z updated, m untouched.
 *   vel     : n bodies (vx, vy, vz, w); vx, vy, vz updated, w untouched.
 *   acc_pot : n rows (ax, ay, az, p); p is not read.
 *
 * Every component: x' = fl(x + fl(dt*v)), then v' = fl(v + fl(dt*a)).
 * Returns 0, or -1 on a bad argument.
 */
int oracle_euler(float *pos_mass, float *vel, const float *acc_pot,
                 int64_t n, float dt)
{
    if (n < 0) return -1;
    if (n > 0 && (pos_mass == NULL || vel == NULL || acc_pot == NULL)) return -1;
    for (int64_t i = 0; i < n; ++i) {
        for (int c = 0; c < 3; ++c) {
            const float v_old = vel[4 * i + c];
            const float step_x = dt * v_old;          /* rounded to fp32 */
            pos_mass[4 * i + c] = pos_mass[4 * i + c] + step_x;
        }
        for (int c = 0; c < 3; ++c) {
            const float step_v = dt * acc_pot[4 * i + c];
            vel[4 * i + c] = vel[4 * i + c] + step_v;
        }
    }
    return 0;
}
