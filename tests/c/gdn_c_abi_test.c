/*
 * gdn_c_abi_test.c -- liblinattn used from C through its ABI alone (no Python, no PyTorch).
 *
 * Seeded synthetic inputs (splitmix64 + Box-Muller, bf16 by round-to-nearest-even) with the
 * cuDNN Linear Attention page's distributions in their slow-decay variant; a ragged batch with
 * grouped heads, an fp32 start state and fp32 checkpoints every 64 tokens:
 *   1. gdn_fwd on device buffers (cudaMalloc) against the fp64 oracle (test infrastructure,
 *      linked in): max|x - ref| / max|ref| <= 1e-2 for o, <= 2e-3 for the final state and the
 *      checkpoints;
 *   2. gdn_fwd_host on pinned host buffers: bitwise the same o, final state and checkpoints;
 *   3. argument errors come back synchronously with their codes.
 * Exit status 0 when every check passes.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "liblinattn.h"

int gdn_oracle_run(const double *q, const double *k, const double *v, const double *g, const double *beta,
                   const int64_t *cu, int64_t T, int N, int HK, int HV, int K, int V, double scale, int l2norm,
                   const double *s0, double *o, double *final_state, double *ckpt, int64_t ckpt_n,
                   const int64_t *ckpt_off, double *transition, const unsigned char *unit_mask, int nthreads,
                   int mutation);

static uint64_t rng_state = 0x5eed2026ull;
static uint64_t splitmix64(void) {
    uint64_t z = (rng_state += 0x9e3779b97f4a7c15ull);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}
static double uniform01(void) { return ((splitmix64() >> 11) + 0.5) * (1.0 / 9007199254740992.0); }
static double normal(void) {
    const double u1 = uniform01(), u2 = uniform01();
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}
static uint16_t to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

#define CUDA_OK(x)                                                              \
    do {                                                                        \
        cudaError_t e_ = (x);                                                   \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            return 2;                                                           \
        }                                                                       \
    } while (0)

static double rel_err(const double *got, const double *ref, size_t n) {
    double num = 0, den = 0;
    for (size_t i = 0; i < n; ++i) {
        const double d = fabs(got[i] - ref[i]);
        if (d > num) num = d;
        if (fabs(ref[i]) > den) den = fabs(ref[i]);
    }
    return den > 0 ? num / den : (num > 0 ? INFINITY : 0);
}

int main(void) {
    enum { N = 5, HK = 2, HV = 4, K = 128, V = 64, CK = 64 };
    const int64_t lengths[N] = {100, 64, 1, 0, 257};
    int32_t cu32[N + 1];
    int64_t cu64[N + 1], ckoff[N], R = 0;
    cu32[0] = 0;
    cu64[0] = 0;
    for (int i = 0; i < N; ++i) {
        cu64[i + 1] = cu64[i] + lengths[i];
        cu32[i + 1] = (int32_t)cu64[i + 1];
        ckoff[i] = R;
        R += (lengths[i] + CK - 1) / CK;
    }
    const int64_t T = cu64[N];
    const size_t nq = (size_t)T * HK * K, nv = (size_t)T * HV * V, ng = (size_t)T * HV;
    const size_t ns = (size_t)N * HV * K * V, nck = (size_t)R * HV * K * V;
    const double scale = 1.0 / sqrt((double)K);

    /* inputs (pinned host memory: gdn_fwd_host reads it asynchronously) */
    uint16_t *q, *k, *v, *o_h, *o_d2h;
    float *g, *beta, *s0, *fin_h, *ck_h, *fin_d2h, *ck_d2h;
    CUDA_OK(cudaMallocHost((void **)&q, nq * 2));
    CUDA_OK(cudaMallocHost((void **)&k, nq * 2));
    CUDA_OK(cudaMallocHost((void **)&v, nv * 2));
    CUDA_OK(cudaMallocHost((void **)&g, ng * 4));
    CUDA_OK(cudaMallocHost((void **)&beta, ng * 4));
    CUDA_OK(cudaMallocHost((void **)&s0, ns * 4));
    CUDA_OK(cudaMallocHost((void **)&o_h, nv * 2));
    CUDA_OK(cudaMallocHost((void **)&fin_h, ns * 4));
    CUDA_OK(cudaMallocHost((void **)&ck_h, nck * 4));
    o_d2h = malloc(nv * 2);
    fin_d2h = malloc(ns * 4);
    ck_d2h = malloc(nck * 4);
    double *dq = malloc(nq * 8), *dk = malloc(nq * 8), *dv = malloc(nv * 8), *dg = malloc(ng * 8),
           *db = malloc(ng * 8), *ds0 = malloc(ns * 8), *ro = malloc(nv * 8), *rfin = malloc(ns * 8),
           *rck = malloc(nck * 8), *got = malloc((nck > nv ? nck : nv) * 8);
    for (size_t i = 0; i < nq; ++i) { q[i] = to_bf16((float)normal()); dq[i] = from_bf16(q[i]); }
    for (size_t i = 0; i < nq; ++i) { k[i] = to_bf16((float)normal()); dk[i] = from_bf16(k[i]); }
    for (size_t i = 0; i < nv; ++i) { v[i] = to_bf16((float)normal()); dv[i] = from_bf16(v[i]); }
    for (size_t i = 0; i < ng; ++i) {
        const double z = normal(), y = normal();
        g[i] = (float)(-log1p(exp(z)) * 1e-3);  /* slow decay: the state reaches every chunk */
        beta[i] = (float)(0.2 / (1.0 + exp(-y)));
        dg[i] = g[i];
        db[i] = beta[i];
    }
    for (size_t i = 0; i < ns; ++i) { s0[i] = (float)(0.1 * normal()); ds0[i] = s0[i]; }

    /* the oracle */
    if (gdn_oracle_run(dq, dk, dv, dg, db, cu64, T, N, HK, HV, K, V, scale, 1, ds0, ro, rfin, rck, CK, ckoff, NULL,
                       NULL, 8, 0) != 0) {
        fprintf(stderr, "oracle rejected the inputs\n");
        return 2;
    }

    /* 1. gdn_fwd on device buffers */
    void *d_q, *d_k, *d_v, *d_g, *d_b, *d_s0, *d_o, *d_fin, *d_ck, *d_cu;
    int32_t *d_status;
    CUDA_OK(cudaMalloc(&d_q, nq * 2));
    CUDA_OK(cudaMalloc(&d_k, nq * 2));
    CUDA_OK(cudaMalloc(&d_v, nv * 2));
    CUDA_OK(cudaMalloc(&d_g, ng * 4));
    CUDA_OK(cudaMalloc(&d_b, ng * 4));
    CUDA_OK(cudaMalloc(&d_s0, ns * 4));
    CUDA_OK(cudaMalloc(&d_o, nv * 2));
    CUDA_OK(cudaMalloc(&d_fin, ns * 4));
    CUDA_OK(cudaMalloc(&d_ck, nck * 4));
    CUDA_OK(cudaMalloc(&d_cu, sizeof(cu32)));
    CUDA_OK(cudaMalloc((void **)&d_status, 4));
    CUDA_OK(cudaMemset(d_status, 0, 4));
    CUDA_OK(cudaMemcpy(d_q, q, nq * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_k, k, nq * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_v, v, nv * 2, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_g, g, ng * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_b, beta, ng * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_s0, s0, ns * 4, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_cu, cu32, sizeof(cu32), cudaMemcpyHostToDevice));

    la_gdn_fwd_params p;
    memset(&p, 0, sizeof(p));
    p.q = d_q; p.q_stride_t = HK * K; p.q_stride_h = K;
    p.k = d_k; p.k_stride_t = HK * K; p.k_stride_h = K;
    p.v = d_v; p.v_stride_t = HV * V; p.v_stride_h = V;
    p.g = (const float *)d_g; p.g_stride_t = HV; p.g_stride_h = 1;
    p.beta = (const float *)d_b; p.beta_stride_t = HV; p.beta_stride_h = 1;
    p.cu_seqlens = d_cu; p.cu_seqlens_bits = 32;
    p.T = T; p.N = N; p.HK = HK; p.HV = HV; p.K = K; p.V = V;
    p.scale = (float)scale;
    p.use_qk_l2norm = 1;
    p.initial_state = d_s0; p.initial_state_dtype = LA_DTYPE_F32;
    p.o = d_o; p.o_stride_t = HV * V; p.o_stride_h = V;
    p.final_state = (float *)d_fin;
    p.checkpoints = d_ck; p.checkpoint_dtype = LA_DTYPE_F32; p.checkpoint_every_n = CK;
    p.status = d_status;
    la_status st = gdn_fwd(&p, NULL);
    if (st != LA_OK) { fprintf(stderr, "gdn_fwd: %s\n", la_status_string(st)); return 1; }
    int32_t dev_status = -1;
    if (la_read_status(d_status, NULL, &dev_status) != LA_OK || dev_status != LA_OK) {
        fprintf(stderr, "device status %d\n", dev_status);
        return 1;
    }
    CUDA_OK(cudaMemcpy(o_d2h, d_o, nv * 2, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(fin_d2h, d_fin, ns * 4, cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(ck_d2h, d_ck, nck * 4, cudaMemcpyDeviceToHost));
    for (size_t i = 0; i < nv; ++i) got[i] = from_bf16(o_d2h[i]);
    const double e_o = rel_err(got, ro, nv);
    for (size_t i = 0; i < ns; ++i) got[i] = fin_d2h[i];
    const double e_f = rel_err(got, rfin, ns);
    for (size_t i = 0; i < nck; ++i) got[i] = ck_d2h[i];
    const double e_c = rel_err(got, rck, nck);
    printf("[parity] C ABI gdn_fwd: o %.2e, final %.2e, checkpoints %.2e\n", e_o, e_f, e_c);
    int fail = !(e_o <= 1e-2 && e_f <= 2e-3 && e_c <= 2e-3);

    /* 2. gdn_fwd_host on pinned host buffers: the same bits */
    la_gdn_fwd_host_params hp;
    memset(&hp, 0, sizeof(hp));
    hp.fwd = p;
    hp.fwd.q = q; hp.fwd.k = k; hp.fwd.v = v; hp.fwd.g = g; hp.fwd.beta = beta;
    hp.fwd.cu_seqlens = cu32; hp.fwd.initial_state = s0;
    hp.fwd.o = o_h; hp.fwd.final_state = fin_h; hp.fwd.checkpoints = ck_h;
    hp.ranges = 4;
    const size_t need = la_gdn_fwd_host_staging_bytes(&hp);
    void *staging;
    if (need == 0) { fprintf(stderr, "staging size query failed\n"); return 1; }
    CUDA_OK(cudaMalloc(&staging, need));
    hp.staging = staging;
    hp.staging_bytes = need;
    st = gdn_fwd_host(&hp, NULL);
    if (st != LA_OK) { fprintf(stderr, "gdn_fwd_host: %s\n", la_status_string(st)); return 1; }
    CUDA_OK(cudaStreamSynchronize(NULL));
    const int same = memcmp(o_h, o_d2h, nv * 2) == 0 && memcmp(fin_h, fin_d2h, ns * 4) == 0 &&
                     memcmp(ck_h, ck_d2h, nck * 4) == 0;
    printf("[parity] C ABI gdn_fwd_host bitwise equal to gdn_fwd: %s\n", same ? "yes" : "no");
    fail |= !same;

    /* 3. argument errors, synchronously */
    la_gdn_fwd_params bad = p;
    bad.K = 96;
    const int e1 = gdn_fwd(&bad, NULL) == LA_ERR_UNSUPPORTED;
    bad = p;
    bad.q = (const char *)d_q + 8;  /* not 16-byte aligned */
    const int e2 = gdn_fwd(&bad, NULL) == LA_ERR_INVALID_ARG;
    la_gdn_fwd_host_params hbad = hp;
    hbad.staging_bytes = 256;
    const int e3 = gdn_fwd_host(&hbad, NULL) == LA_ERR_WORKSPACE;
    printf("argument errors: %d %d %d (%s)\n", e1, e2, e3, la_status_string(LA_ERR_UNSUPPORTED));
    fail |= !(e1 && e2 && e3);

    printf("%s\n", fail ? "FAIL" : "OK");
    return fail ? 1 : 0;
}
