// Standalone (unfused) kernels of the post-backward step: ring reduce-scatter,
// the owner-side AdamW shard update (flag pass + conditional update), and the
// parameter all-gather. Each is one HBM stream over its arrays; they are the
// building blocks the fused step is measured against.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "zr_device.cuh"
#include "zr_internal.h"
#include "zr_nvtx.h"

using zr::fail;

namespace {

constexpr int kThreads = 256;

// Work is cut into chunks of kChunkElems consecutive elements, one block per chunk (a
// block moves on to chunk + gridDim.x only if the grid was capped). The hardware hands
// blocks out in index order, so the elements in flight stay a compact window of every
// array; a grid-stride loop would spread each block's accesses over the whole array.
constexpr int64_t kChunkElems = 32768;

// Blocks for n elements.
int chunk_grid(int64_t n) {
  int64_t want = (n + kChunkElems - 1) / kChunkElems;
  if (want < 1) want = 1;
  return (int)(want < (1 << 30) ? want : (1 << 30));
}

// Calls f(i) for this block's items of PER elements each, out of nitems.
template <int PER, class F>
__device__ __forceinline__ void for_block_items(int64_t nitems, F&& f) {
  constexpr int64_t kItems = kChunkElems / PER;
  for (int64_t c = blockIdx.x; c * kItems < nitems; c += gridDim.x) {
    const int64_t end = (c + 1) * kItems < nitems ? (c + 1) * kItems : nitems;
    for (int64_t i = c * kItems + threadIdx.x; i < end; i += blockDim.x) f(i);
  }
}

zr_status launch_status(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return ZR_OK;
}

// Block-wide OR of a per-thread flag, then one atomicOr per block.
__device__ __forceinline__ void block_flag_or(bool mine, int32_t* flag_out) {
  __shared__ int s_any;
  if (threadIdx.x == 0) s_any = 0;
  __syncthreads();
  if (__any_sync(0xFFFFFFFFu, mine) && (threadIdx.x & 31) == 0) s_any = 1;
  __syncthreads();
  if (threadIdx.x == 0 && s_any) atomicOr(flag_out, 1);
}

// ---------------------------------------------------------------- reduce-scatter
struct RsArgs {
  const void* grads[ZR_MAX_W];   // indexed by worker
  int order[ZR_MAX_W];           // ring position -> worker
  float* out[ZR_MAX_REPLICAS];   // R copies of the sums: 1 for the reduce-scatter, R for the all-reduce
  int32_t* overflow;
  int64_t n, C;
  int W, R;
};

// Ring-order fp32 sum of the W values of element group e (8 elements, or the
// ragged tail). Block c of the bucket starts at position c. DT: input type.
template <int DT, int WT>
__global__ void __launch_bounds__(kThreads) rs_kernel(const __grid_constant__ RsArgs a) {
  const int W = WT > 0 ? WT : a.W;
  bool bad = false;
  const int64_t ngroups = (a.n + 7) / 8;
  for_block_items<8>(ngroups, [&](int64_t g) {
    const int64_t e = g * 8;
    const int c = (int)(e / a.C);
    if (e + 8 <= a.n) {
      float s[8];
      if (WT > 0) {
        float xs[WT > 0 ? WT : 1][8];
#pragma unroll
        for (int h = 0; h < (WT > 0 ? WT : 1); ++h) {
          int pos = c + h;
          pos -= pos >= W ? W : 0;
          zr::load8<DT>(a.grads[a.order[pos]], e, xs[h]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = xs[0][j];
#pragma unroll
        for (int h = 1; h < (WT > 0 ? WT : 1); ++h)
#pragma unroll
          for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], xs[h][j]);
      } else {
        zr::load8<DT>(a.grads[a.order[c]], e, s);
        for (int h = 1; h < W; ++h) {
          int pos = c + h;
          pos -= pos >= W ? W : 0;
          float x[8];
          zr::load8<DT>(a.grads[a.order[pos]], e, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) bad |= zr::nonfinite(s[j]);
      const float4 lo = make_float4(s[0], s[1], s[2], s[3]), hi = make_float4(s[4], s[5], s[6], s[7]);
      for (int r = 0; r < a.R; ++r) {
        zr::st_once_f4(a.out[r] + e, lo);
        zr::st_once_f4(a.out[r] + e + 4, hi);
      }
    } else {
      for (int64_t i = e; i < a.n; ++i) {
        float s = zr::load1<DT>(a.grads[a.order[c]], i);
        for (int h = 1; h < W; ++h) {
          int pos = c + h;
          pos -= pos >= W ? W : 0;
          s = __fadd_rn(s, zr::load1<DT>(a.grads[a.order[pos]], i));
        }
        bad |= zr::nonfinite(s);
        for (int r = 0; r < a.R; ++r) a.out[r][i] = s;
      }
    }
  });
  block_flag_or(bad, a.overflow);
}

template <int DT>
void launch_rs(const RsArgs& a, int grid, cudaStream_t s) {
  switch (a.W) {
    case 1: rs_kernel<DT, 1><<<grid, kThreads, 0, s>>>(a); break;
    case 2: rs_kernel<DT, 2><<<grid, kThreads, 0, s>>>(a); break;
    case 3: rs_kernel<DT, 3><<<grid, kThreads, 0, s>>>(a); break;
    case 4: rs_kernel<DT, 4><<<grid, kThreads, 0, s>>>(a); break;
    case 8: rs_kernel<DT, 8><<<grid, kThreads, 0, s>>>(a); break;
    default: rs_kernel<DT, 0><<<grid, kThreads, 0, s>>>(a); break;
  }
}

// ---------------------------------------------------------------- AdamW shard step
// A read-only stream: with one 16-byte load per thread in flight it ran at 0.84 of the
// copy rate, so each thread issues kFlagLoads loads (128 bytes) before testing any of them.
constexpr int kFlagLoads = 8;

__global__ void __launch_bounds__(kThreads) flag_pass_kernel(const float* __restrict__ x, int64_t n,
                                                              int32_t* overflow) {
  constexpr int64_t kItems = kChunkElems / 4;  // float4 words per chunk
  static_assert(kItems % (kThreads * kFlagLoads) == 0, "a chunk is whole rounds of loads");
  bool bad = false;
  const int64_t nv = n / 4;
  for (int64_t c = blockIdx.x; c * kItems < nv; c += gridDim.x) {
    const int64_t base = c * kItems;
    if (base + kItems <= nv) {
#pragma unroll 1
      for (int r = 0; r < (int)(kItems / (kThreads * kFlagLoads)); ++r) {
        const float* p = x + 4 * (base + (int64_t)r * kThreads * kFlagLoads + threadIdx.x);
        float4 v[kFlagLoads];
#pragma unroll
        for (int u = 0; u < kFlagLoads; ++u) v[u] = zr::ld_once_f4(p + 4 * u * kThreads);
#pragma unroll
        for (int u = 0; u < kFlagLoads; ++u)
          bad |= zr::nonfinite(v[u].x) | zr::nonfinite(v[u].y) | zr::nonfinite(v[u].z) | zr::nonfinite(v[u].w);
      }
    } else {
      for (int64_t i = base + threadIdx.x; i < nv; i += blockDim.x) {
        const float4 v = zr::ld_once_f4(x + 4 * i);
        bad |= zr::nonfinite(v.x) | zr::nonfinite(v.y) | zr::nonfinite(v.z) | zr::nonfinite(v.w);
      }
    }
  }
  for (int64_t i = nv * 4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    bad |= zr::nonfinite(x[i]);
  block_flag_or(bad, overflow);
}

struct AdamArgs {
  const float* sums;
  float* m;
  float* v;
  float* master;
  const int32_t* overflow;
  int64_t n;
  float r;  // fp32(1/(S*W))
  zr::AdamConsts k;
};

__global__ void __launch_bounds__(kThreads) adamw_kernel(const __grid_constant__ AdamArgs a) {
  __shared__ int s_skip;
  if (threadIdx.x == 0) s_skip = *reinterpret_cast<const volatile int32_t*>(a.overflow);
  __syncthreads();
  if (s_skip) return;
  const int64_t nv = a.n / 4;
  for_block_items<4>(nv, [&](int64_t i) {
    const int64_t e = 4 * i;
    float4 s = zr::ld_once_f4(a.sums + e), p = zr::ld_once_f4(a.master + e), m = zr::ld_once_f4(a.m + e),
           v = zr::ld_once_f4(a.v + e);
    zr::adamw_elem(__fmul_rn(s.x, a.r), p.x, m.x, v.x, a.k);
    zr::adamw_elem(__fmul_rn(s.y, a.r), p.y, m.y, v.y, a.k);
    zr::adamw_elem(__fmul_rn(s.z, a.r), p.z, m.z, v.z, a.k);
    zr::adamw_elem(__fmul_rn(s.w, a.r), p.w, m.w, v.w, a.k);
    zr::st_once_f4(a.master + e, p);
    zr::st_once_f4(a.m + e, m);
    zr::st_once_f4(a.v + e, v);
  });
  for (int64_t i = nv * 4 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < a.n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float p = a.master[i], m = a.m[i], v = a.v[i];
    zr::adamw_elem(__fmul_rn(a.sums[i], a.r), p, m, v, a.k);
    a.master[i] = p;
    a.m[i] = m;
    a.v[i] = v;
  }
}

// ---------------------------------------------------------------- all-gather
struct AgArgs {
  void* out[ZR_MAX_REPLICAS];
  const float* master;
  int64_t n;
  int R;
};

template <int DT>
__global__ void __launch_bounds__(kThreads) ag_kernel(const __grid_constant__ AgArgs a) {
  const int64_t ngroups = (a.n + 7) / 8;
  for_block_items<8>(ngroups, [&](int64_t g) {
    const int64_t e = g * 8;
    if (e + 8 <= a.n) {
      float4 lo = zr::ld_once_f4(a.master + e), hi = zr::ld_once_f4(a.master + e + 4);
      const float f[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
      const uint4 packed = zr::pack8<DT>(f);
      for (int r = 0; r < a.R; ++r) zr::st_once(static_cast<uint16_t*>(a.out[r]) + e, packed);
    } else {
      for (int64_t i = e; i < a.n; ++i) {
        const uint16_t b = zr::from_f32<DT>(a.master[i]);
        for (int r = 0; r < a.R; ++r) static_cast<uint16_t*>(a.out[r])[i] = b;
      }
    }
  });
}

}  // namespace

namespace zr {
double beta_power_from(double p, int64_t k, float beta, int64_t n) {
  const double b = (double)beta;
  for (; k < n; ++k) {
    const double q = p * b;
    if (q == p) break;  // every later factor leaves it unchanged
    p = q;
  }
  return p;
}

float bias_correction_host(float beta, int64_t t) { return (float)(1.0 - beta_power_from(1.0, 0, beta, t)); }

bool betas_ok(const zr_adamw_hyper& h) {
  return h.beta1 >= 0.0f && h.beta1 < 1.0f && h.beta2 >= 0.0f && h.beta2 < 1.0f;
}

AdamConsts adam_consts_host(const zr_adamw_hyper& h, float bc1, float bc2) {
  AdamConsts k;
  k.b1 = h.beta1;
  k.b2 = h.beta2;
  k.omb1 = 1.0f - h.beta1;
  k.omb2 = 1.0f - h.beta2;
  k.lr = h.lr;
  k.eps = h.eps;
  const float lrwd = h.lr * h.weight_decay;
  k.decay = 1.0f - lrwd;
  k.bc1 = bc1;
  k.bc2 = bc2;
  return k;
}
}  // namespace zr

namespace {
// The ring sums of one bucket written to R outputs: the reduce-scatter (R = 1) and the
// all-reduce (every worker's copy) share the kernel; `what` names the caller in errors.
zr_status ring_sums(const char* what, const void* const* grads, zr_dtype dt, int64_t n, int W, const int* order,
                    float* const* out, int R, int32_t* overflow, void* stream) {
  if (n < 0) return fail(ZR_ERR_INVALID, "%s: n < 0", what);
  if (W < 1 || W > ZR_MAX_W) return fail(ZR_ERR_INVALID, "%s: W=%d outside [1, %d]", what, W, ZR_MAX_W);
  if (dt != ZR_F16 && dt != ZR_BF16 && dt != ZR_F32)
    return fail(ZR_ERR_INVALID, "%s: dtype must be F16, BF16 or F32", what);
  if (R < 1 || R > ZR_MAX_REPLICAS) return fail(ZR_ERR_INVALID, "%s: R=%d outside [1, %d]", what, R, ZR_MAX_REPLICAS);
  if (!grads || !out || !overflow) return fail(ZR_ERR_INVALID, "%s: null pointer", what);
  if (reinterpret_cast<uintptr_t>(overflow) & 3u) return fail(ZR_ERR_INVALID, "%s: misaligned overflow flag", what);
  RsArgs a{};
  for (int r = 0; r < R; ++r) {
    if (!out[r] || !zr::aligned16(out[r])) return fail(ZR_ERR_INVALID, "%s: output %d null or misaligned", what, r);
    a.out[r] = out[r];
  }
  bool seen[ZR_MAX_W] = {};
  for (int p = 0; p < W; ++p) {
    const int w = order ? order[p] : p;
    if (w < 0 || w >= W || seen[w]) return fail(ZR_ERR_INVALID, "%s: order is not a permutation", what);
    seen[w] = true;
    a.order[p] = w;
  }
  for (int w = 0; w < W; ++w) {
    if (!grads[w] || !zr::aligned16(grads[w])) return fail(ZR_ERR_INVALID, "%s: grads[%d] null or misaligned", what, w);
    a.grads[w] = grads[w];
  }
  if (n == 0) return ZR_OK;
  a.overflow = overflow;
  a.n = n;
  a.C = zr_chunk_size(n, W, ZR_ALIGN);
  a.W = W;
  a.R = R;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = chunk_grid(n);
  if (dt == ZR_F16) launch_rs<zr::DT_F16>(a, grid, s);
  else if (dt == ZR_BF16) launch_rs<zr::DT_BF16>(a, grid, s);
  else launch_rs<zr::DT_F32>(a, grid, s);
  return launch_status(what);
}
}  // namespace

extern "C" zr_status zr_reduce_scatter(const void* const* grads, zr_dtype dt, int64_t n, int W, const int* order,
                                       float* sums, int32_t* overflow, void* stream) {
  zr::Range range("zr_reduce_scatter");
  zr::clear_error();
  float* const out[1] = {sums};
  return ring_sums("zr_reduce_scatter", grads, dt, n, W, order, out, 1, overflow, stream);
}

extern "C" zr_status zr_all_reduce(const void* const* grads, zr_dtype dt, int64_t n, int W, const int* order,
                                   float* const* out, int R, int32_t* overflow, void* stream) {
  zr::Range range("zr_all_reduce");
  zr::clear_error();
  return ring_sums("zr_all_reduce", grads, dt, n, W, order, out, R, overflow, stream);
}

// ---------------------------------------------------------------- accumulate
namespace {
template <int DT, bool FIRST>
__global__ void __launch_bounds__(kThreads) accumulate_kernel(const void* __restrict__ g, float* __restrict__ acc,
                                                              int64_t n) {
  const int64_t ngroups = n / 8;
  for_block_items<8>(ngroups, [&](int64_t q) {
    const int64_t e = q * 8;
    float x[8];
    zr::load8<DT>(g, e, x);
    if (!FIRST) {
      const float4 a0 = zr::ld_once_f4(acc + e), a1 = zr::ld_once_f4(acc + e + 4);
      x[0] = __fadd_rn(a0.x, x[0]); x[1] = __fadd_rn(a0.y, x[1]); x[2] = __fadd_rn(a0.z, x[2]);
      x[3] = __fadd_rn(a0.w, x[3]); x[4] = __fadd_rn(a1.x, x[4]); x[5] = __fadd_rn(a1.y, x[5]);
      x[6] = __fadd_rn(a1.z, x[6]); x[7] = __fadd_rn(a1.w, x[7]);
    }
    zr::st_once_f4(acc + e, make_float4(x[0], x[1], x[2], x[3]));
    zr::st_once_f4(acc + e + 4, make_float4(x[4], x[5], x[6], x[7]));
  });
  for (int64_t i = ngroups * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = zr::load1<DT>(g, i);
    acc[i] = FIRST ? x : __fadd_rn(acc[i], x);
  }
}
}  // namespace

extern "C" zr_status zr_accumulate(const void* grad, zr_dtype dt, float* acc, int64_t n, int first, void* stream) {
  zr::Range range("zr_accumulate");
  zr::clear_error();
  if (n < 0) return fail(ZR_ERR_INVALID, "zr_accumulate: n < 0");
  if (dt != ZR_F16 && dt != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_accumulate: dtype must be F16 or BF16");
  if (!grad || !acc || !zr::aligned16(grad) || !zr::aligned16(acc))
    return fail(ZR_ERR_INVALID, "zr_accumulate: null or misaligned pointer");
  if (n == 0) return ZR_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = chunk_grid(n);
  if (dt == ZR_F16) {
    if (first) accumulate_kernel<zr::DT_F16, true><<<grid, kThreads, 0, s>>>(grad, acc, n);
    else accumulate_kernel<zr::DT_F16, false><<<grid, kThreads, 0, s>>>(grad, acc, n);
  } else {
    if (first) accumulate_kernel<zr::DT_BF16, true><<<grid, kThreads, 0, s>>>(grad, acc, n);
    else accumulate_kernel<zr::DT_BF16, false><<<grid, kThreads, 0, s>>>(grad, acc, n);
  }
  return launch_status("zr_accumulate");
}

extern "C" zr_status zr_adamw_shard_step(const float* shard_sums, float* m, float* v, float* master, int64_t len,
                                         const zr_adamw_hyper* h, float loss_scale, int W, int64_t t,
                                         int32_t* overflow, void* stream) {
  zr::Range range("zr_adamw_shard_step");
  zr::clear_error();
  if (len < 0) return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: len < 0");
  if (!h) return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: null hyperparameters");
  if (t < 1) return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: t must be >= 1");
  if (W < 1) return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: W < 1");
  if (!zr::betas_ok(*h)) return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: betas must lie in [0, 1)");
  if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
    return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: loss_scale must be positive and finite");
  if (!shard_sums || !m || !v || !master || !overflow) return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: null pointer");
  if (!zr::aligned16(shard_sums) || !zr::aligned16(m) || !zr::aligned16(v) || !zr::aligned16(master))
    return fail(ZR_ERR_INVALID, "zr_adamw_shard_step: misaligned array");
  if (len == 0) return ZR_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  flag_pass_kernel<<<chunk_grid(len), kThreads, 0, s>>>(shard_sums, len, overflow);
  zr_status st = launch_status("zr_adamw_shard_step flag pass");
  if (st != ZR_OK) return st;
  AdamArgs a{};
  a.sums = shard_sums;
  a.m = m;
  a.v = v;
  a.master = master;
  a.overflow = overflow;
  a.n = len;
  a.r = (float)(1.0 / ((double)loss_scale * (double)W));
  a.k = zr::adam_consts_host(*h, zr::bias_correction_host(h->beta1, t), zr::bias_correction_host(h->beta2, t));
  adamw_kernel<<<chunk_grid(len), kThreads, 0, s>>>(a);
  return launch_status("zr_adamw_shard_step update");
}

extern "C" zr_status zr_all_gather(const float* master, int64_t n, zr_dtype out_dt, void* const* replicas,
                                   int n_replicas, void* stream) {
  zr::Range range("zr_all_gather");
  zr::clear_error();
  if (n < 0) return fail(ZR_ERR_INVALID, "zr_all_gather: n < 0");
  if (out_dt != ZR_F16 && out_dt != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_all_gather: dtype must be F16 or BF16");
  if (n_replicas < 1 || n_replicas > ZR_MAX_REPLICAS)
    return fail(ZR_ERR_INVALID, "zr_all_gather: n_replicas=%d outside [1, %d]", n_replicas, ZR_MAX_REPLICAS);
  if (!master || !replicas || !zr::aligned16(master)) return fail(ZR_ERR_INVALID, "zr_all_gather: null or misaligned master");
  AgArgs a{};
  for (int r = 0; r < n_replicas; ++r) {
    if (!replicas[r] || !zr::aligned16(replicas[r])) return fail(ZR_ERR_INVALID, "zr_all_gather: replica %d null or misaligned", r);
    a.out[r] = replicas[r];
  }
  if (n == 0) return ZR_OK;
  a.master = master;
  a.n = n;
  a.R = n_replicas;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int grid = chunk_grid(n);
  if (out_dt == ZR_F16) ag_kernel<zr::DT_F16><<<grid, kThreads, 0, s>>>(a);
  else ag_kernel<zr::DT_BF16><<<grid, kThreads, 0, s>>>(a);
  return launch_status("zr_all_gather");
}
