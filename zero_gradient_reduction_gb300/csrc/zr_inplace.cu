// The in-place step: the fused update on ONE state set, for runs with no room for a
// second one. The whole step is skipped when any reduced gradient is not finite, and
// that is known only after every bucket has been summed, so the step is two launches of
// fused_step_kernel: a flag pass (ring sums, flag only) and the in-place update, which
// writes nothing if the flag is set. The two fold every sum with the same code, so the
// flag the update obeys is exactly the flag of the sums it applies.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "zr_device.cuh"
#include "zr_internal.h"
#include "zr_nvtx.h"

using zr::fail;

#include "zr_plan.h"
#include "zr_step_kernel.cuh"

zr_status zr::init_inplace(zr_plan* p) {
  const bool f32 = p->fp32_grads != 0;
  const bool f16 = p->dtype == ZR_F16;
  KernelFn f = f16 ? pick_kernel<zr::DT_F16, kFlagPass>(p->W, p->A, f32)
                   : pick_kernel<zr::DT_BF16, kFlagPass>(p->W, p->A, f32);
  KernelFn u = f16 ? pick_kernel<zr::DT_F16, kInPlace>(p->W, p->A, f32)
                   : pick_kernel<zr::DT_BF16, kInPlace>(p->W, p->A, f32);
  p->ip_flag_kernel = reinterpret_cast<void*>(f);
  p->ip_update_kernel = reinterpret_cast<void*>(u);
  p->ip_flag_grid = zr::step_grid(p, p->ntiles);
  p->ip_update_grid = zr::step_grid(p, p->ntiles);
  return ZR_OK;
}

extern "C" zr_status zr_step_inplace(zr_plan* p, int stage, const void* const* grads, const zr_state1* st,
                                     const zr_adamw_hyper* h, void* stream, zr_step_report* rep) {
  zr::Range range("zr_step_inplace");
  zr::clear_error();
  if (!p || !st || !h || !grads) return fail(ZR_ERR_INVALID, "zr_step_inplace: null argument");
  if (stage < 0 || stage > 3) return fail(ZR_ERR_INVALID, "zr_step_inplace: stage=%d not in 0..3", stage);
  // a plan with no parameters: empty (possibly null) arrays, and a step that only runs the
  // scaler rule (two launches of one block over no tiles)
  if (p->numel > 0) {
    for (int r = 0; r < p->W * p->A; ++r)
      if (!grads[r] || !zr::aligned16(grads[r]))
        return fail(ZR_ERR_INVALID, "zr_step_inplace: grads[%d] null or misaligned", r);
    if (!st->master || !st->m || !st->v || !st->param)
      return fail(ZR_ERR_INVALID, "zr_step_inplace: the state set has a null array");
    if (!zr::aligned16(st->master) || !zr::aligned16(st->m) || !zr::aligned16(st->v) || !zr::aligned16(st->param))
      return fail(ZR_ERR_INVALID, "zr_step_inplace: the state set is misaligned");
  }

  // The single set goes in both slots: the in-place kernel reads and writes slot 0 and
  // the flag pass touches neither.
  float* const master[2] = {st->master, st->master};
  float* const m[2] = {st->m, st->m};
  float* const v[2] = {st->v, st->v};
  void* const param[2] = {st->param, st->param};
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const FusedArgs flag_args = make_args(p, stage, grads, master, m, v, param, h, 0, p->ntiles, 0);
  reinterpret_cast<KernelFn>(p->ip_flag_kernel)<<<p->ip_flag_grid, kThreads, 0, cs>>>(flag_args);
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) {
    const FusedArgs upd_args =
        make_args(p, stage, grads, master, m, v, param, h, 0, p->ntiles, (unsigned)p->ip_update_grid);
    reinterpret_cast<KernelFn>(p->ip_update_kernel)<<<p->ip_update_grid, kThreads, 0, cs>>>(upd_args);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step_inplace: launch failed: %s", cudaGetErrorString(e));
  return rep ? zr_plan_report(p, stream, rep) : ZR_OK;
}

extern "C" zr_status zr_step_inplace_from_host(zr_plan* p, int stage, const void* const* host_grads,
                                               void* const* dev_grads, const zr_state1* st, const zr_adamw_hyper* h,
                                               void* stream, zr_step_report* rep) {
  zr::Range range("zr_step_inplace_from_host");
  zr::clear_error();
  if (!p || !host_grads || !dev_grads || !rep)
    return fail(ZR_ERR_INVALID, "zr_step_inplace_from_host: null argument");
  const int R = p->W * p->A;
  for (int r = 0; r < R && p->numel > 0; ++r)
    if (!host_grads[r] || !dev_grads[r] || !zr::aligned16(dev_grads[r]))
      return fail(ZR_ERR_INVALID, "zr_step_inplace_from_host: replica %d: null pointer or misaligned device buffer", r);
  if (!st || !h) return fail(ZR_ERR_INVALID, "zr_step_inplace_from_host: null argument");
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t esz = p->fp32_grads ? 4 : 2;
  for (const zr_bucket& b : p->buckets) {
    for (int r = 0; r < R; ++r) {
      const size_t off = (size_t)b.start * esz, bytes = (size_t)b.len * esz;
      const cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dev_grads[r]) + off,
                                            static_cast<const char*>(host_grads[r]) + off, bytes,
                                            cudaMemcpyHostToDevice, cs);
      if (e != cudaSuccess)
        return fail(ZR_ERR_CUDA, "zr_step_inplace_from_host: copy: %s", cudaGetErrorString(e));
    }
  }
  return zr_step_inplace(p, stage, const_cast<const void* const*>(dev_grads), st, h, stream, rep);
}
