/* Three fused steps driven from plain C through zr.h: cudaMalloc'd buffers, no Python and
 * no torch. Every gradient is 1.0 on W = 4 workers with loss scale 1, so the mean
 * gradient is 1 at every step; with a constant gradient, bias-corrected m and v are both
 * 1 at every step t (m = 1 - 0.9^t and v = 1 - 0.999^t before correction), so each step
 * (no weight decay) moves every master value by -lr / (1 + eps): 0.5 - t * lr / (1 + eps)
 * after step t. Step 1 runs zr_step as the plan chose, step 2 zr_step with bulk-copy
 * staging, step 3 zr_step_noalloc on the plan's bucket table. Prints "ok" and returns 0
 * on success. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "zr.h"

#define NWORKERS 4

static int fail_cuda(const char* what, cudaError_t e) {
    printf("%s: %s\n", what, cudaGetErrorString(e));
    return 1;
}

/* every master value after step t: 0.5 - t * lr / (1 + eps), lr = 1e-3, eps = 1e-8 */
static int check_master(const float* dev, float* host, int64_t n, int t) {
    cudaError_t e = cudaMemcpy(host, dev, (size_t)n * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda("read back", e);
    const double want = 0.5 - t * 1e-3 / (1.0 + 1e-8);
    for (int64_t i = 0; i < n; ++i) {
        if (fabs((double)host[i] - want) > 2e-6) {
            printf("step %d: master[%lld] = %.9g, want %.9g\n", t, (long long)i, host[i], want);
            return 1;
        }
    }
    return 0;
}

int main(void) {
    const int64_t numels[3] = {1000, 37, 5000};
    zr_plan_desc d = {0};
    d.W = NWORKERS;
    d.A = 1;
    d.dtype = ZR_BF16;
    d.stage = 2;
    d.align = ZR_ALIGN;
    d.cap = 4096;
    d.ntensors = 3;
    d.numels = numels;
    d.order = NULL;
    d.scaler.init_scale = 1.0f;
    d.scaler.backoff = 0.5f;
    d.scaler.growth = 2.0f;
    d.scaler.min_scale = 1.0f;
    d.scaler.growth_interval = 1000;
    d.scaler.dynamic = 0;
    d.fp32_grads = 0;
    zr_plan* p = NULL;
    if (zr_plan_create(&d, &p) != ZR_OK) {
        printf("zr_plan_create: %s\n", zr_last_error());
        return 1;
    }
    const int64_t n = zr_plan_numel(p);

    uint16_t* g16 = (uint16_t*)malloc((size_t)n * 2);
    float* f32 = (float*)malloc((size_t)n * 4);
    if (!g16 || !f32) return 1;
    for (int64_t i = 0; i < n; ++i) {
        g16[i] = 0x3F80; /* bf16 1.0 */
        f32[i] = 0.5f;
    }
    void* grads[NWORKERS];
    for (int w = 0; w < NWORKERS; ++w) {
        cudaError_t e = cudaMalloc(&grads[w], (size_t)n * 2);
        if (e == cudaSuccess) e = cudaMemcpy(grads[w], g16, (size_t)n * 2, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail_cuda("grads", e);
    }
    zr_state st;
    for (int k = 0; k < 2; ++k) {
        cudaError_t e = cudaMalloc((void**)&st.master[k], (size_t)n * 4);
        if (e == cudaSuccess) e = cudaMalloc((void**)&st.m[k], (size_t)n * 4);
        if (e == cudaSuccess) e = cudaMalloc((void**)&st.v[k], (size_t)n * 4);
        if (e == cudaSuccess) e = cudaMalloc(&st.param[k], (size_t)n * 2);
        if (e == cudaSuccess) e = cudaMemset(st.m[k], 0, (size_t)n * 4);
        if (e == cudaSuccess) e = cudaMemset(st.v[k], 0, (size_t)n * 4);
        if (e != cudaSuccess) return fail_cuda("state", e);
    }
    cudaError_t e = cudaMemcpy(st.master[0], f32, (size_t)n * 4, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda("master", e);

    const zr_adamw_hyper h = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.0f};
    zr_step_report rep;
    if (zr_step(p, 2, (const void* const*)grads, &st, &h, NULL, &rep) != ZR_OK) {
        printf("zr_step: %s\n", zr_last_error());
        return 1;
    }
    if (rep.t != 1 || rep.overflow != 0 || rep.current != 1 || rep.n_real != 6037) {
        printf("report: t=%lld overflow=%d current=%d n_real=%lld\n", (long long)rep.t, rep.overflow, rep.current,
               (long long)rep.n_real);
        return 1;
    }
    if (check_master(st.master[1], f32, n, 1) != 0) return 1;

    /* step 2: loads staged through shared memory by bulk copies */
    if (zr_plan_set_staging(p, ZR_STAGING_BULK, 0, 0) != ZR_OK || zr_plan_staging(p) != ZR_STAGING_BULK) {
        printf("zr_plan_set_staging: %s\n", zr_last_error());
        return 1;
    }
    if (zr_step(p, 2, (const void* const*)grads, &st, &h, NULL, &rep) != ZR_OK || rep.t != 2 || rep.current != 0) {
        printf("zr_step (bulk): %s t=%lld current=%d\n", zr_last_error(), (long long)rep.t, rep.current);
        return 1;
    }
    if (check_master(st.master[0], f32, n, 2) != 0) return 1;

    /* step 3: the no-allocation entry point on the plan's bucket table; the caller carries the
     * live set (0), the loss scale (1) and t (3) */
    const int nb = zr_plan_nbuckets(p);
    zr_bucket* buckets = (zr_bucket*)malloc((size_t)nb * sizeof(zr_bucket));
    int32_t* overflow = NULL;
    if (!buckets || zr_plan_buckets(p, buckets, NULL) != ZR_OK) return 1;
    e = cudaMalloc((void**)&overflow, sizeof(int32_t));
    if (e != cudaSuccess) return fail_cuda("overflow", e);
    if (zr_step_noalloc(buckets, nb, NWORKERS, 1, ZR_BF16, NULL, (const void* const*)grads, &st, 0, &h, 1.0f, 3,
                        overflow, NULL) != ZR_OK) {
        printf("zr_step_noalloc: %s\n", zr_last_error());
        return 1;
    }
    int32_t flag = -1;
    e = cudaMemcpy(&flag, overflow, sizeof flag, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda("overflow read back", e);
    if (flag != 0) {
        printf("zr_step_noalloc: overflow %d\n", flag);
        return 1;
    }
    if (check_master(st.master[1], f32, n, 3) != 0) return 1;
    cudaFree(overflow);
    free(buckets);
    zr_plan_destroy(p);
    for (int w = 0; w < NWORKERS; ++w) cudaFree(grads[w]);
    for (int k = 0; k < 2; ++k) {
        cudaFree(st.master[k]);
        cudaFree(st.m[k]);
        cudaFree(st.v[k]);
        cudaFree(st.param[k]);
    }
    free(g16);
    free(f32);
    printf("ok\n");
    return 0;
}
