/* One fused step driven from plain C through zr.h: cudaMalloc'd buffers, no Python and
 * no torch. Every gradient is 1.0 on W = 4 workers with loss scale 1, so the mean
 * gradient is 1 and the first AdamW step (m = 0.1, v = 0.001, bias corrections 0.1 and
 * 0.001, no weight decay) moves every master value from 0.5 to 0.5 - lr / (1 + eps).
 * Prints "ok" and returns 0 on success. */
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
    e = cudaMemcpy(f32, st.master[1], (size_t)n * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda("read back", e);
    const double want = 0.5 - 1e-3 / (1.0 + 1e-8);
    for (int64_t i = 0; i < n; ++i) {
        if (fabs((double)f32[i] - want) > 1e-6) {
            printf("master[%lld] = %.9g, want %.9g\n", (long long)i, f32[i], want);
            return 1;
        }
    }
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
