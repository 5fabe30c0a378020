// ZeRO-Offload step: the reduce-scatter stays on the GPU, the optimizer moves to the
// host CPU. The fp32 master/m/v live in host memory; the reduced gradients go down
// to the host (4 bytes/param over the host link), the CPU runs the owner-side AdamW
// (zr_offload_adamw), and the updated 16-bit parameters come back (2 bytes/param).
// Buckets are pipelined: bucket b's sums are copied down while the CPU updates
// bucket b-1 and bucket b-2's parameters are copied up.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <vector>

#include "zr_internal.h"
#include "zr_nvtx.h"
#include "zr_plan.h"

using zr::fail;

namespace {

zr_status cuda_err(const char* what, cudaError_t e) {
  return fail(ZR_ERR_CUDA, "zr_offload_step: %s: %s", what, cudaGetErrorString(e));
}

}  // namespace

extern "C" zr_status zr_offload_step(zr_plan* p, int stage, const void* const* grads, float* sums_dev, float* sums_host,
                                     float* master, float* m, float* v, void* param_host, void* param_dev,
                                     const zr_adamw_hyper* h, float loss_scale, int64_t t, int nthreads,
                                     void* stream, int32_t* overflow) {
  zr::Range range("zr_offload_step");
  zr::clear_error();
  if (!p || !grads || !sums_dev || !sums_host || !master || !m || !v || !param_host || !param_dev || !h || !overflow)
    return fail(ZR_ERR_INVALID, "zr_offload_step: null argument");
  if (stage < 1 || stage > 3) return fail(ZR_ERR_INVALID, "zr_offload_step: stage=%d not in 1..3", stage);
  if (p->A != 1) return fail(ZR_ERR_UNSUPPORTED, "zr_offload_step: plans with A > 1 (accumulate first)");
  if (t < 1) return fail(ZR_ERR_INVALID, "zr_offload_step: t must be >= 1");
  if (!zr::aligned16(sums_dev) || !zr::aligned16(param_dev))
    return fail(ZR_ERR_INVALID, "zr_offload_step: misaligned device buffer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const zr_dtype gdt = p->fp32_grads ? ZR_F32 : p->dtype;
  const size_t gsz = p->fp32_grads ? 4 : 2;
  int32_t* flag_dev = &p->ctrl_dev->offload_flag;
  cudaError_t e = cudaMemsetAsync(flag_dev, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_err("memset", e);
  // 1. reduce-scatter of every bucket on the GPU (fp32 sums, global flag)
  std::vector<const void*> views(p->W);
  for (const zr_bucket& b : p->buckets) {
    for (int w = 0; w < p->W; ++w) views[w] = static_cast<const char*>(grads[w]) + (size_t)b.start * gsz;
    zr_status st = zr_reduce_scatter(views.data(), gdt, b.len, p->W, p->order, sums_dev + b.start, flag_dev, stream);
    if (st != ZR_OK) return st;
  }
  // 2. the flag decides before any state changes
  int32_t flag = 0;
  e = cudaMemcpyAsync(&flag, flag_dev, sizeof flag, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_err("flag", e);
  if (flag) {
    *overflow = 1;
    return ZR_OK;
  }
  // 3. pipeline per bucket: copy sums down (event), update on the CPU, copy params up
  const size_t nb = p->buckets.size();
  std::vector<cudaEvent_t> down(nb, nullptr);
  for (size_t b = 0; b < nb && e == cudaSuccess; ++b) e = cudaEventCreateWithFlags(&down[b], cudaEventDisableTiming);
  for (size_t b = 0; b < nb && e == cudaSuccess; ++b) {
    const zr_bucket& bk = p->buckets[b];
    e = cudaMemcpyAsync(sums_host + bk.start, sums_dev + bk.start, (size_t)bk.len * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaEventRecord(down[b], s);
  }
  zr_status st = ZR_OK;
  for (size_t b = 0; b < nb && e == cudaSuccess && st == ZR_OK; ++b) {
    const zr_bucket& bk = p->buckets[b];
    e = cudaEventSynchronize(down[b]);
    if (e != cudaSuccess) break;
    int32_t of = 0;
    st = zr_offload_adamw(sums_host + bk.start, master + bk.start, m + bk.start, v + bk.start,
                          static_cast<char*>(param_host) + (size_t)bk.start * 2, p->dtype, bk.len, h, loss_scale,
                          p->W, t, nthreads, &of);
    if (st == ZR_OK)
      e = cudaMemcpyAsync(static_cast<char*>(param_dev) + (size_t)bk.start * 2,
                          static_cast<const char*>(param_host) + (size_t)bk.start * 2, (size_t)bk.len * 2,
                          cudaMemcpyHostToDevice, s);
  }
  for (cudaEvent_t ev : down)
    if (ev) cudaEventDestroy(ev);
  if (st != ZR_OK) return st;
  if (e != cudaSuccess) return cuda_err("pipeline", e);
  *overflow = 0;
  return ZR_OK;
}
