/*
 * A plain C program that uses the library the way a non-Python caller would: device memory from
 * the CUDA runtime, one decode token for N sequences through gdn_recurrent_step (fp32 q, k, v,
 * d = 64, state updated in place), results copied back.  The same inputs go through the fp64
 * oracle's C entry point (test infrastructure, linked from oracle/_build), and the program prints
 * the worst relative L2 error per (sequence, head) of the outputs and of the new states.
 * Exit status 0 when both are within the fp32 tolerance (1e-4), 1 when not, 2 on a CUDA or
 * library error.  Built and run by tests/test_zzz_gpu_c_program.py.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "gdn.h"

/* the oracle's C entry point (form 0: the token-by-token recurrence) */
int gdn_oracle_forward(int form, const double* q, const double* k, const double* v,
                       const double* g, const double* beta, const int32_t* cu_seqlens,
                       int num_seqs, int H, int Hk, int dk, int dv, int g_per_channel,
                       double scale, int use_qk_l2norm, const double* S0, double* y,
                       double* S_final, int C, int n_threads);

enum { N = 8, H = 4, D = 64 };

/* seeded draws (64-bit LCG, Box-Muller); both sides receive the same float values */
static uint64_t rng_state = 0x2545F4914F6CDD1Dull;
static double uniform01(void) {
    rng_state = rng_state * 6364136223846793005ull + 1442695040888963407ull;
    return ((double)(rng_state >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}
static double normal(void) {
    const double u1 = uniform01(), u2 = uniform01();
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

#define CUDA_OK(call)                                                              \
    do {                                                                           \
        cudaError_t e_ = (call);                                                   \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));            \
            return 2;                                                              \
        }                                                                          \
    } while (0)

static double rel_l2(const float* x, const double* ref, long n) {
    double num = 0.0, den = 0.0;
    for (long i = 0; i < n; ++i) {
        const double d = (double)x[i] - ref[i];
        num += d * d;
        den += ref[i] * ref[i];
    }
    return sqrt(num) / (den > 0.0 ? sqrt(den) : 1e-300);
}

int main(void) {
    const long n_tok = (long)N * H * D, n_gate = (long)N * H, n_state = (long)N * H * D * D;
    float *q = malloc(n_tok * 4), *k = malloc(n_tok * 4), *v = malloc(n_tok * 4);
    float *g = malloc(n_gate * 4), *beta = malloc(n_gate * 4), *S = malloc(n_state * 4);
    float *y = malloc(n_tok * 4);
    double *qd = malloc(n_tok * 8), *kd = malloc(n_tok * 8), *vd = malloc(n_tok * 8);
    double *gd = malloc(n_gate * 8), *bd = malloc(n_gate * 8), *Sd = malloc(n_state * 8);
    double *y_ref = malloc(n_tok * 8), *S_ref = malloc(n_state * 8);
    int32_t cu[N + 1];
    for (long i = 0; i < n_tok; ++i) { q[i] = (float)normal(); k[i] = (float)normal(); v[i] = (float)normal(); }
    for (long i = 0; i < n_gate; ++i) {
        g[i] = (float)(-0.05 - 1.45 * uniform01());  /* log alpha in (-1.5, -0.05) */
        beta[i] = (float)uniform01();
    }
    for (long i = 0; i < n_state; ++i) S[i] = (float)(0.1 * normal());
    for (long i = 0; i < n_tok; ++i) { qd[i] = q[i]; kd[i] = k[i]; vd[i] = v[i]; }
    for (long i = 0; i < n_gate; ++i) { gd[i] = g[i]; bd[i] = beta[i]; }
    for (long i = 0; i < n_state; ++i) Sd[i] = S[i];
    for (int n = 0; n <= N; ++n) cu[n] = n;   /* every sequence: one token */

    float *dq, *dk, *dv, *dg, *db, *dS, *dy;
    CUDA_OK(cudaMalloc((void**)&dq, n_tok * 4));
    CUDA_OK(cudaMalloc((void**)&dk, n_tok * 4));
    CUDA_OK(cudaMalloc((void**)&dv, n_tok * 4));
    CUDA_OK(cudaMalloc((void**)&dg, n_gate * 4));
    CUDA_OK(cudaMalloc((void**)&db, n_gate * 4));
    CUDA_OK(cudaMalloc((void**)&dS, n_state * 4));
    CUDA_OK(cudaMalloc((void**)&dy, n_tok * 4));
    CUDA_OK(cudaMemcpy(dq, q, n_tok * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dk, k, n_tok * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dv, v, n_tok * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dg, g, n_gate * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(db, beta, n_gate * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dS, S, n_state * 4, cudaMemcpyHostToDevice));

    int rc = gdn_recurrent_step(dq, dk, dv, dg, db, dS, N, H, H, D, D, GDN_F32, GDN_DECAY_PER_HEAD,
                                0.0f, 1, NULL, NULL, NULL, NULL, NULL, 1e-6f, dy, GDN_F32, NULL);
    if (rc != GDN_OK) {
        fprintf(stderr, "gdn_recurrent_step: %s\n", gdn_status_string(rc));
        return 2;
    }
    int dev_status = -100;
    rc = gdn_get_device_error(NULL, &dev_status);
    if (rc != GDN_OK || dev_status != GDN_OK) {
        fprintf(stderr, "device status %d (%s)\n", dev_status, gdn_status_string(dev_status));
        return 2;
    }
    CUDA_OK(cudaMemcpy(y, dy, n_tok * 4, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(S, dS, n_state * 4, cudaMemcpyDeviceToHost));

    if (gdn_oracle_forward(0, qd, kd, vd, gd, bd, cu, N, H, H, D, D, 0, 1.0 / sqrt((double)D), 1,
                           Sd, y_ref, S_ref, 64, 1) != 0) {
        fprintf(stderr, "oracle rejected its arguments\n");
        return 2;
    }
    double worst_y = 0.0, worst_S = 0.0;
    for (long u = 0; u < (long)N * H; ++u) {
        const double ey = rel_l2(y + u * D, y_ref + u * D, D);
        const double eS = rel_l2(S + u * D * D, S_ref + u * D * D, (long)D * D);
        if (ey > worst_y) worst_y = ey;
        if (eS > worst_S) worst_S = eS;
    }
    printf("max_rel_y %.3e max_rel_S %.3e\n", worst_y, worst_S);
    cudaFree(dq); cudaFree(dk); cudaFree(dv); cudaFree(dg); cudaFree(db); cudaFree(dS); cudaFree(dy);
    return (worst_y <= 1e-4 && worst_S <= 1e-4) ? 0 : 1;
}
