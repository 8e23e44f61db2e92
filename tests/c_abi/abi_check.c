/*
 * abi_check.c -- the C ABI used from plain C99: device buffers from
 * cudaMalloc, nbody_forces, nbody_euler_step and nbody_simulate, checked
 * against a direct double-precision sum written here (G = 1, every source
 * including the body itself).  Exit status 0 on success.
 */
#include <math.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "nbody.h"

#define N 777
#define EPS2 1e-3f

static unsigned long long state = 88172645463325252ULL;
static float uniform(float lo, float hi) {       /* xorshift64, enough for a test */
    state ^= state << 13;
    state ^= state >> 7;
    state ^= state << 17;
    return lo + (hi - lo) * (float)((state >> 11) * (1.0 / 9007199254740992.0));
}

int main(void) {
    static float pm[N * 4], vel[N * 4], acc[N * 4], pm2[N * 4];
    for (int i = 0; i < N; ++i) {
        pm[4 * i + 0] = uniform(-1.f, 1.f);
        pm[4 * i + 1] = uniform(-1.f, 1.f);
        pm[4 * i + 2] = uniform(-1.f, 1.f);
        pm[4 * i + 3] = uniform(0.5f, 1.5f);
        vel[4 * i + 0] = vel[4 * i + 1] = vel[4 * i + 2] = 0.25f;
        vel[4 * i + 3] = 0.f;
    }
    float *d_pm = NULL, *d_vel = NULL, *d_acc = NULL;
    if (cudaMalloc((void **)&d_pm, sizeof pm) != cudaSuccess ||
        cudaMalloc((void **)&d_vel, sizeof vel) != cudaSuccess ||
        cudaMalloc((void **)&d_acc, sizeof acc) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 2;
    }
    cudaMemcpy(d_pm, pm, sizeof pm, cudaMemcpyHostToDevice);
    cudaMemcpy(d_vel, vel, sizeof vel, cudaMemcpyHostToDevice);

    nbody_status st = nbody_forces(d_pm, N, EPS2, d_acc, 0);
    if (st != NBODY_OK) {
        fprintf(stderr, "nbody_forces: %s\n", nbody_status_string(st));
        return 3;
    }
    if (nbody_forces(d_pm, N, EPS2, d_pm, 0) != NBODY_ERR_ALIAS) return 4;   /* rejected on the host */
    cudaMemcpy(acc, d_acc, sizeof acc, cudaMemcpyDeviceToHost);

    double worst = 0.0;
    for (int i = 0; i < N; ++i) {
        double a[3] = {0, 0, 0}, p = 0;
        for (int j = 0; j < N; ++j) {
            double r[3], d2 = EPS2;
            for (int c = 0; c < 3; ++c) {
                r[c] = (double)pm[4 * j + c] - (double)pm[4 * i + c];
                d2 += r[c] * r[c];
            }
            const double inv = 1.0 / sqrt(d2);
            for (int c = 0; c < 3; ++c) a[c] += pm[4 * j + 3] * r[c] * inv * inv * inv;
            p -= pm[4 * j + 3] * inv;
        }
        const double na = sqrt(a[0] * a[0] + a[1] * a[1] + a[2] * a[2]);
        double da = 0;
        for (int c = 0; c < 3; ++c) da += (acc[4 * i + c] - a[c]) * (acc[4 * i + c] - a[c]);
        const double ea = sqrt(da) / na, ep = fabs(acc[4 * i + 3] - p) / fabs(p);
        if (ea > worst) worst = ea;
        if (ep > worst) worst = ep;
    }
    printf("nbody_forces from C: worst per-body relative error %.3e\n", worst);
    if (!(worst <= 1e-4)) return 5;

    /* the symmetric path forced through the options struct, and the planner's
     * automatic choice at 2^20 bodies, from C */
    nbody_forces_opts opts = {NBODY_PATH_SYMMETRIC, -1, 0, NBODY_PRECISION_DEFAULT,
                              NBODY_QUANTITIES_ACC_POT, 0};
    static float acc_sym[N * 4];
    if ((st = nbody_forces_ex(d_pm, N, EPS2, d_vel, &opts, 0)) != NBODY_OK) return 10;
    cudaMemcpy(acc_sym, d_vel, sizeof acc_sym, cudaMemcpyDeviceToHost);
    cudaMemcpy(d_vel, vel, sizeof vel, cudaMemcpyHostToDevice);         /* restore */
    double worst_sym = 0.0;
    for (int i = 0; i < N; ++i) {
        double d = 0, na = 0;
        for (int c = 0; c < 3; ++c) {
            d += (double)(acc_sym[4 * i + c] - acc[4 * i + c]) * (acc_sym[4 * i + c] - acc[4 * i + c]);
            na += (double)acc[4 * i + c] * acc[4 * i + c];
        }
        const double e = sqrt(d / na);
        if (e > worst_sym) worst_sym = e;
    }
    printf("symmetric path from C: worst per-body difference %.3e\n", worst_sym);
    if (!(worst_sym <= 2e-4)) return 11;
    nbody_plan plan;
    nbody_forces_opts autoo = {NBODY_PATH_AUTO, -1, 0, NBODY_PRECISION_DEFAULT,
                              NBODY_QUANTITIES_ACC_POT, 0};
    if (nbody_plan_forces(1 << 20, 152, 0, &autoo, &plan) != NBODY_OK) return 12;
    if (plan.path != NBODY_PATH_SYMMETRIC || plan.scratch_bytes <= 0 ||
        plan.scratch_bytes > NBODY_DEFAULT_WORKSPACE_BYTES)
        return 13;
    /* the target/source planner: few sources take the row-split path, with
     * no workspace and one CTA per SM */
    if (nbody_plan_forces_ts(3000, 500, 152, 0, &autoo, -1, &plan) != NBODY_OK) return 19;
    if (plan.path != NBODY_PATH_ROWS || plan.scratch_bytes != 0 || plan.grid > 152) return 20;

    /* the symmetric path again within a caller-owned workspace: ask for its
     * size, give it exactly that, and get the same bits */
    size_t ws_bytes = 0;
    if (nbody_forces_ws(NULL, N, EPS2, NULL, &opts, NULL, &ws_bytes, 0) != NBODY_OK) return 14;
    void *ws = NULL;
    if (ws_bytes > 0 && cudaMalloc(&ws, ws_bytes) != cudaSuccess) return 15;
    if (nbody_forces_ws(d_pm, N, EPS2, d_vel, &opts, ws ? ws : (void *)d_vel, &ws_bytes, 0) != NBODY_OK)
        return 16;
    static float acc_ws[N * 4];
    cudaMemcpy(acc_ws, d_vel, sizeof acc_ws, cudaMemcpyDeviceToHost);
    cudaMemcpy(d_vel, vel, sizeof vel, cudaMemcpyHostToDevice);         /* restore */
    for (int k = 0; k < N * 4; ++k)
        if (acc_ws[k] != acc_sym[k]) return 17;
    if (ws) cudaFree(ws);
    printf("nbody_forces_ws from C: %zu bytes of workspace, same bits\n", ws_bytes);

    /* one Euler step, then the same step through nbody_simulate on a copy */
    cudaMemcpy(pm2, d_pm, sizeof pm2, cudaMemcpyDeviceToHost);
    if ((st = nbody_euler_step(d_pm, d_vel, d_acc, N, 1e-3f, 0)) != NBODY_OK) return 6;
    float *s_pm = NULL, *s_vel = NULL, *s_acc = NULL;
    cudaMalloc((void **)&s_pm, sizeof pm);
    cudaMalloc((void **)&s_vel, sizeof vel);
    cudaMalloc((void **)&s_acc, sizeof acc);
    cudaMemcpy(s_pm, pm2, sizeof pm2, cudaMemcpyHostToDevice);
    cudaMemcpy(s_vel, vel, sizeof vel, cudaMemcpyHostToDevice);
    if ((st = nbody_simulate(s_pm, s_vel, s_acc, N, EPS2, 1e-3f, 1, 0)) != NBODY_OK) return 7;
    static float a1[N * 4], a2[N * 4];
    cudaMemcpy(a1, d_pm, sizeof a1, cudaMemcpyDeviceToHost);
    cudaMemcpy(a2, s_pm, sizeof a2, cudaMemcpyDeviceToHost);
    for (int k = 0; k < N * 4; ++k)
        if (a1[k] != a2[k]) return 8;
    if (cudaDeviceSynchronize() != cudaSuccess) return 9;
    if (nbody_release_cached() != NBODY_OK) return 18;
    printf("nbody_euler_step and nbody_simulate agree bit for bit\n");
    return 0;
}
