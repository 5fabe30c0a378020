// ZeRO-Offload step: the reduce-scatter stays on the GPU, the optimizer moves to the
// host CPU. The fp32 master/m/v live in host memory; the reduced gradients go down
// to the host (4 bytes/param over the host link), the CPU runs the owner-side AdamW
// (zr_offload_adamw), and the updated 16-bit parameters come back (2 bytes/param).
// Buckets are pipelined: later buckets' sums are copied down while the CPU updates
// bucket b, and earlier buckets' parameters are copied up on a second stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <memory>
#include <thread>
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
  if (!p || !grads || !h || !overflow) return fail(ZR_ERR_INVALID, "zr_offload_step: null argument");
  // a plan with no parameters has empty (possibly null) arrays
  if (p->numel > 0 && (!sums_dev || !sums_host || !master || !m || !v || !param_host || !param_dev))
    return fail(ZR_ERR_INVALID, "zr_offload_step: null array");
  if (stage < 0 || stage > 3) return fail(ZR_ERR_INVALID, "zr_offload_step: stage=%d not in 0..3", stage);
  if (p->A != 1) return fail(ZR_ERR_UNSUPPORTED, "zr_offload_step: plans with A > 1 (accumulate first)");
  if (t < 1) return fail(ZR_ERR_INVALID, "zr_offload_step: t must be >= 1");
  if (!zr::betas_ok(*h)) return fail(ZR_ERR_INVALID, "zr_offload_step: betas must lie in [0, 1)");
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
  // 3. pipeline per bucket. Every bucket's sums are queued down on `stream`, each followed
  //    by an event. A team of nthreads host threads walks the buckets in order: each waits
  //    for a bucket's event and updates its slice of the bucket (AdamW and the cast in one
  //    pass), and the last thread to finish the bucket queues its parameters up on a second
  //    stream, so that copies up overlap copies down and the host never waits for them.
  const size_t nb = p->buckets.size();
  cudaStream_t up = nullptr;
  std::vector<cudaEvent_t> down(nb, nullptr);
  cudaEvent_t up_done = nullptr;
  e = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&up_done, cudaEventDisableTiming);
  for (size_t b = 0; b < nb && e == cudaSuccess; ++b) e = cudaEventCreateWithFlags(&down[b], cudaEventDisableTiming);
  for (size_t b = 0; b < nb && e == cudaSuccess; ++b) {
    const zr_bucket& bk = p->buckets[b];
    e = cudaMemcpyAsync(sums_host + bk.start, sums_dev + bk.start, (size_t)bk.len * 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaEventRecord(down[b], s);
  }
  if (e == cudaSuccess) {
    const zr::OffloadConsts k = zr::offload_consts(*h, loss_scale, p->W, t);
    const int nt = nthreads < 1 ? 1 : (nthreads > 256 ? 256 : nthreads);
    std::unique_ptr<std::atomic<int>[]> left(new std::atomic<int>[nb]);
    for (size_t b = 0; b < nb; ++b) left[b].store(nt);
    std::atomic<int> err{(int)cudaSuccess};
    auto note = [&](cudaError_t ee) {
      int ok = (int)cudaSuccess;
      if (ee != cudaSuccess) err.compare_exchange_strong(ok, (int)ee);
    };
    auto work = [&](int tid) {
      for (size_t b = 0; b < nb; ++b) {
        const zr_bucket& bk = p->buckets[b];
        if (err.load() == (int)cudaSuccess) {
          const cudaError_t ee = cudaEventSynchronize(down[b]);
          note(ee);
          if (ee == cudaSuccess) {
            const int64_t per = (bk.len + nt - 1) / nt;
            const int64_t lo = std::min(per * tid, bk.len), hi = std::min(per * (tid + 1), bk.len);
            zr::offload_update(sums_host, master, m, v, param_host, p->dtype, bk.start + lo, bk.start + hi, k);
          }
        }
        if (left[b].fetch_sub(1) == 1 && err.load() == (int)cudaSuccess)
          note(cudaMemcpyAsync(static_cast<char*>(param_dev) + (size_t)bk.start * 2,
                               static_cast<const char*>(param_host) + (size_t)bk.start * 2, (size_t)bk.len * 2,
                               cudaMemcpyHostToDevice, up));
      }
    };
    std::vector<std::thread> team;
    for (int i = 1; i < nt; ++i) team.emplace_back(work, i);
    work(0);
    for (auto& th : team) th.join();
    e = (cudaError_t)err.load();
    // the caller's stream sees the parameters once every copy up is done
    if (e == cudaSuccess) e = cudaEventRecord(up_done, up);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, up_done, 0);
  }
  for (cudaEvent_t ev : down)
    if (ev) cudaEventDestroy(ev);
  if (up_done) cudaEventDestroy(up_done);
  if (up) cudaStreamDestroy(up);
  if (e != cudaSuccess) return cuda_err("pipeline", e);
  *overflow = 0;
  return ZR_OK;
}
