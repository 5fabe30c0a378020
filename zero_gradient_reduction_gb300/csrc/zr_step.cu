// The fused post-backward step: one launch per step over a precomputed tile
// schedule. For every 8-element group of every bucket a thread
//   - loads the W*A 16-bit gradient values (16-byte streaming loads),
//   - forms each worker's fp32 micro-batch sum and the ring-order fp32 sum,
//   - unscales (x 1/(S*W)), tests for non-finite values,
//   - runs AdamW on the fp32 master/m/v of state set k,
//   - writes master/m/v and the 16-bit parameter into state set 1-k.
// The last block to finish (atomic ticket, no waiting) ORs the flags, applies the
// loss-scale rule and, on a clean step, advances t and flips k. Pure HBM stream:
// (2*W*A + 26) bytes per parameter, no tensor cores (no contraction here).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "zr_device.cuh"
#include "zr_internal.h"

using zr::fail;

namespace zr {
float bias_correction_host(float beta, int64_t t);
}

namespace {

constexpr int kThreads = 256;
constexpr int kTileElems = 16384;  // elements per tile (a multiple of 8 * kThreads)

struct FusedArgs {
  const uint16_t* grads[ZR_MAX_REPLICAS];  // replica w*A + a
  int order[ZR_MAX_W];                     // ring position -> worker
  const int4* tiles;                       // {start lo, start hi, groups, block index c}
  int64_t ntiles;
  float* master[2];
  float* m[2];
  float* v[2];
  uint16_t* param[2];
  zr::Ctrl* ctrl;
  float lr, beta1, beta2, eps, weight_decay;
  int W, A, stage;
};

// Per-block view of the control block, read once at the start of the step.
struct StepConsts {
  zr::AdamConsts k;
  float r;  // fp32(1/(S*W))
  int cur;  // live state set
};

__device__ void read_consts(const FusedArgs& a, StepConsts& out) {
  const volatile zr::Ctrl* c = a.ctrl;
  const double S = (double)c->scale;
  const double p1 = c->prod1, p2 = c->prod2;
  out.cur = c->k;
  out.r = (float)__ddiv_rn(1.0, __dmul_rn(S, (double)a.W));
  out.k.b1 = a.beta1;
  out.k.b2 = a.beta2;
  out.k.omb1 = __fsub_rn(1.0f, a.beta1);
  out.k.omb2 = __fsub_rn(1.0f, a.beta2);
  out.k.lr = a.lr;
  out.k.eps = a.eps;
  out.k.decay = __fsub_rn(1.0f, __fmul_rn(a.lr, a.weight_decay));
  out.k.bc1 = (float)__dsub_rn(1.0, __dmul_rn(p1, (double)a.beta1));
  out.k.bc2 = (float)__dsub_rn(1.0, __dmul_rn(p2, (double)a.beta2));
}

// The loss-scale rule and commit, run by one thread of the last block.
__device__ void finish_step(const FusedArgs& a) {
  volatile zr::Ctrl* c = a.ctrl;
  const int of = c->overflow;
  float scale = c->scale;
  c->last_overflow = of;
  c->scale_used = scale;
  c->stage = a.stage;
  c->steps = c->steps + 1;
  if (of) {
    c->skipped = c->skipped + 1;
    if (c->dynamic) {
      const float s2 = __fmul_rn(scale, c->backoff);
      scale = s2 > c->min_scale ? s2 : c->min_scale;
      c->good = 0;
    }
  } else {
    c->t = c->t + 1;
    c->prod1 = __dmul_rn(c->prod1, (double)a.beta1);
    c->prod2 = __dmul_rn(c->prod2, (double)a.beta2);
    c->k = 1 - c->k;
    c->good = c->good + 1;
    if (c->dynamic && c->good >= c->interval) {
      scale = __fmul_rn(scale, c->growth);
      c->good = 0;
    }
  }
  c->scale = scale;
  c->overflow = 0;
  c->ticket = 0;
  __threadfence();
}

// AdamW on one 8-element group whose ring sums are s[0..7], reading state set `cur`
// at flat element e and writing set 1-cur; returns whether any sum was not finite.
template <int DT>
__device__ __forceinline__ bool update_group(const FusedArgs& a, const StepConsts& K, int64_t e, const float s[8],
                                             float4 p0, float4 p1, float4 m0, float4 m1, float4 v0, float4 v1) {
  float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bad |= zr::nonfinite(s[j]);
    zr::adamw_elem(__fmul_rn(s[j], K.r), p[j], m[j], v[j], K.k);
  }
  const int out = 1 - K.cur;
  zr::st_once_f4(a.master[out] + e, make_float4(p[0], p[1], p[2], p[3]));
  zr::st_once_f4(a.master[out] + e + 4, make_float4(p[4], p[5], p[6], p[7]));
  zr::st_once_f4(a.m[out] + e, make_float4(m[0], m[1], m[2], m[3]));
  zr::st_once_f4(a.m[out] + e + 4, make_float4(m[4], m[5], m[6], m[7]));
  zr::st_once_f4(a.v[out] + e, make_float4(v[0], v[1], v[2], v[3]));
  zr::st_once_f4(a.v[out] + e + 4, make_float4(v[4], v[5], v[6], v[7]));
  zr::st_once(a.param[out] + e, zr::pack8<DT>(p));
  return bad;
}

// Ring-position pointers are computed per tile from the grid constants (block index c
// is uniform over the tile), so tiles need no shared table and no block barrier. For
// A = 1 with a compile-time W all W gradient loads and the six state loads of a group
// are issued before any arithmetic.
template <int DT, int WT, int AT>
__global__ void __launch_bounds__(kThreads, 2) fused_step_kernel(const __grid_constant__ FusedArgs a) {
  __shared__ StepConsts s_k;
  __shared__ int s_bad;
  __shared__ unsigned s_ticket;
  if (threadIdx.x == 0) {
    read_consts(a, s_k);
    s_bad = 0;
  }
  __syncthreads();
  const StepConsts K = s_k;
  const int W = WT > 0 ? WT : a.W;
  const int A = AT > 0 ? AT : a.A;
  const float* __restrict__ mst_in = a.master[K.cur];
  const float* __restrict__ m_in = a.m[K.cur];
  const float* __restrict__ v_in = a.v[K.cur];
  bool bad = false;

  for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    const int4 d = a.tiles[tile];
    const int64_t start = (int64_t)(((uint64_t)(uint32_t)d.y << 32) | (uint32_t)d.x);
    const int groups = d.z, c = d.w;
    if (WT > 0 && AT == 1) {
      constexpr int WN = WT > 0 ? WT : 1;
      const uint16_t* gp[WN];
#pragma unroll
      for (int h = 0; h < WN; ++h) {
        int pos = c + h;
        pos -= pos >= WN ? WN : 0;
        gp[h] = a.grads[a.order[pos]] + start;
      }
      // U groups per thread and iteration, all of their loads issued before any arithmetic:
      // with few replicas one group holds too few bytes in flight to cover HBM latency.
      constexpr int UN = WN <= 3 ? 2 : 1;
      for (int g0 = threadIdx.x; g0 < groups; g0 += UN * blockDim.x) {
        uint4 raw[UN][WN];
        float4 st[UN][6];
#pragma unroll
        for (int u = 0; u < UN; ++u) {
          const int g = g0 + u * (int)blockDim.x;
          if (g < groups) {
            const int64_t off = (int64_t)g * 8, e = start + off;
#pragma unroll
            for (int h = 0; h < WN; ++h) raw[u][h] = zr::ld_once(gp[h] + off);
            st[u][0] = zr::ld_once_f4(mst_in + e);
            st[u][1] = zr::ld_once_f4(mst_in + e + 4);
            st[u][2] = zr::ld_once_f4(m_in + e);
            st[u][3] = zr::ld_once_f4(m_in + e + 4);
            st[u][4] = zr::ld_once_f4(v_in + e);
            st[u][5] = zr::ld_once_f4(v_in + e + 4);
          }
        }
#pragma unroll
        for (int u = 0; u < UN; ++u) {
          const int g = g0 + u * (int)blockDim.x;
          if (g < groups) {
            float s[8];
            zr::unpack8<DT>(raw[u][0], s);
#pragma unroll
            for (int h = 1; h < WN; ++h) {
              float x[8];
              zr::unpack8<DT>(raw[u][h], x);
#pragma unroll
              for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x[j]);
            }
            bad |= update_group<DT>(a, K, start + (int64_t)g * 8, s, st[u][0], st[u][1], st[u][2], st[u][3],
                                    st[u][4], st[u][5]);
          }
        }
      }
    } else {
      for (int g = threadIdx.x; g < groups; g += blockDim.x) {
        const int64_t off = (int64_t)g * 8, e = start + off;
        float s[8];
        for (int h = 0; h < W; ++h) {
          int pos = c + h;
          pos -= pos >= W ? W : 0;
          const uint16_t* const* rep = a.grads + a.order[pos] * A;  // worker's A micro-batches
          float w8[8];
          zr::unpack8<DT>(zr::ld_once(rep[0] + e), w8);
          for (int q = 1; q < A; ++q) {
            float x[8];
            zr::unpack8<DT>(zr::ld_once(rep[q] + e), x);
#pragma unroll
            for (int j = 0; j < 8; ++j) w8[j] = __fadd_rn(w8[j], x[j]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) s[j] = h == 0 ? w8[j] : __fadd_rn(s[j], w8[j]);
        }
        const float4 p0 = zr::ld_once_f4(mst_in + e), p1 = zr::ld_once_f4(mst_in + e + 4);
        const float4 m0 = zr::ld_once_f4(m_in + e), m1 = zr::ld_once_f4(m_in + e + 4);
        const float4 v0 = zr::ld_once_f4(v_in + e), v1 = zr::ld_once_f4(v_in + e + 4);
        bad |= update_group<DT>(a, K, e, s, p0, p1, m0, m1, v0, v1);
      }
    }
  }

  // Block flag -> control block, then the ticket: the last block to arrive decides.
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) s_bad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s_bad) atomicOr(&a.ctrl->overflow, 1);
    __threadfence();
    s_ticket = atomicAdd(&a.ctrl->ticket, 1u);
  }
  __syncthreads();
  if (s_ticket == gridDim.x - 1 && threadIdx.x == 0) {
    __threadfence();
    finish_step(a);
  }
}

using KernelFn = void (*)(FusedArgs);

template <int DT>
KernelFn pick_kernel(int W, int A) {
  if (A == 1) {
    switch (W) {
      case 1: return fused_step_kernel<DT, 1, 1>;
      case 2: return fused_step_kernel<DT, 2, 1>;
      case 3: return fused_step_kernel<DT, 3, 1>;
      case 4: return fused_step_kernel<DT, 4, 1>;
      case 8: return fused_step_kernel<DT, 8, 1>;
      default: return fused_step_kernel<DT, 0, 1>;
    }
  }
  if (A == 4) {
    switch (W) {
      case 2: return fused_step_kernel<DT, 2, 4>;
      case 4: return fused_step_kernel<DT, 4, 4>;
      case 8: return fused_step_kernel<DT, 8, 4>;
      default: return fused_step_kernel<DT, 0, 4>;
    }
  }
  return fused_step_kernel<DT, 0, 0>;
}

}  // namespace

struct zr_plan {
  int W = 0, A = 0, stage = 0, align = 0;
  zr_dtype dtype = ZR_BF16;
  int64_t numel = 0, n_real = 0;
  std::vector<zr_bucket> buckets;
  std::vector<int64_t> tensor_offsets;
  int order[ZR_MAX_W] = {};
  zr_scaler_cfg scaler{};
  int4* tiles_dev = nullptr;
  int64_t ntiles = 0;
  zr::Ctrl* ctrl_dev = nullptr;
  KernelFn kernel = nullptr;
  int grid = 0;
  int device = 0;
};

namespace {

zr::Ctrl initial_ctrl(const zr_scaler_cfg& sc) {
  zr::Ctrl c;
  std::memset(&c, 0, sizeof c);
  c.k = 0;
  c.scale = sc.init_scale;
  c.scale_used = sc.init_scale;
  c.dynamic = sc.dynamic ? 1 : 0;
  c.interval = sc.growth_interval;
  c.backoff = sc.backoff;
  c.growth = sc.growth;
  c.min_scale = sc.min_scale;
  c.prod1 = 1.0;
  c.prod2 = 1.0;
  return c;
}

zr_status cuda_fail(const char* what, cudaError_t e) {
  return fail(e == cudaErrorMemoryAllocation ? ZR_ERR_OOM : ZR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace

extern "C" zr_status zr_plan_create(const zr_plan_desc* d, zr_plan** out) {
  zr::clear_error();
  if (!d || !out) return fail(ZR_ERR_INVALID, "zr_plan_create: null argument");
  *out = nullptr;
  if (d->W < 1 || d->W > ZR_MAX_W) return fail(ZR_ERR_INVALID, "zr_plan_create: W=%d outside [1, %d]", d->W, ZR_MAX_W);
  if (d->A < 1 || (int64_t)d->W * d->A > ZR_MAX_REPLICAS)
    return fail(ZR_ERR_INVALID, "zr_plan_create: A=%d (W*A must be in [1, %d])", d->A, ZR_MAX_REPLICAS);
  if (d->dtype != ZR_F16 && d->dtype != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_plan_create: dtype must be F16 or BF16");
  if (d->stage < 1 || d->stage > 3) return fail(ZR_ERR_INVALID, "zr_plan_create: stage=%d not in 1..3", d->stage);
  if (d->align != ZR_ALIGN) return fail(ZR_ERR_INVALID, "zr_plan_create: align must be %d", ZR_ALIGN);
  if (d->ntensors < 1 || !d->numels) return fail(ZR_ERR_INVALID, "zr_plan_create: empty tensor list");
  if (d->cap < 1) return fail(ZR_ERR_INVALID, "zr_plan_create: cap < 1");
  if (!(d->scaler.init_scale > 0.0f) || !std::isfinite(d->scaler.init_scale))
    return fail(ZR_ERR_INVALID, "zr_plan_create: init_scale must be positive and finite");
  if (d->scaler.dynamic && (!(d->scaler.backoff > 0.0f) || !(d->scaler.growth > 0.0f) ||
                            !(d->scaler.min_scale > 0.0f) || d->scaler.growth_interval < 1))
    return fail(ZR_ERR_INVALID, "zr_plan_create: bad dynamic scaler settings");

  zr_plan* p = new (std::nothrow) zr_plan();
  if (!p) return fail(ZR_ERR_OOM, "zr_plan_create: host allocation");
  p->W = d->W;
  p->A = d->A;
  p->dtype = d->dtype;
  p->stage = d->stage;
  p->align = d->align;
  p->scaler = d->scaler;
  bool seen[ZR_MAX_W] = {};
  for (int i = 0; i < d->W; ++i) {
    const int w = d->order ? d->order[i] : i;
    if (w < 0 || w >= d->W || seen[w]) {
      delete p;
      return fail(ZR_ERR_INVALID, "zr_plan_create: order is not a permutation");
    }
    seen[w] = true;
    p->order[i] = w;
  }
  p->buckets.resize(d->ntensors);
  p->tensor_offsets.resize(d->ntensors);
  int nb = 0;
  zr_status st = zr_bucket_plan(d->numels, d->ntensors, d->cap, d->W, d->align, p->buckets.data(), &nb,
                                p->tensor_offsets.data());
  if (st != ZR_OK) {
    delete p;
    return st;
  }
  p->buckets.resize(nb);
  p->n_real = 0;
  for (int t = 0; t < d->ntensors; ++t) p->n_real += d->numels[t];
  p->numel = nb ? p->buckets.back().start + p->buckets.back().len : 0;

  // Tile schedule: every block of every bucket cut into pieces of at most kTileElems.
  std::vector<int4> tiles;
  for (const zr_bucket& b : p->buckets) {
    for (int c = 0; c < p->W; ++c) {
      int64_t lo = b.start + (int64_t)c * b.chunk, hi = lo + b.chunk;
      const int64_t end = b.start + b.len;
      if (lo > end) lo = end;
      if (hi > end) hi = end;
      for (int64_t x = lo; x < hi; x += kTileElems) {
        const int64_t len = (hi - x) < kTileElems ? (hi - x) : kTileElems;
        tiles.push_back(make_int4((int)(uint32_t)(uint64_t)x, (int)(uint32_t)((uint64_t)x >> 32), (int)(len / 8), c));
      }
    }
  }
  p->ntiles = (int64_t)tiles.size();
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess && !tiles.empty()) e = cudaMalloc(&p->tiles_dev, tiles.size() * sizeof(int4));
  if (e == cudaSuccess && !tiles.empty())
    e = cudaMemcpy(p->tiles_dev, tiles.data(), tiles.size() * sizeof(int4), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMalloc(&p->ctrl_dev, sizeof(zr::Ctrl));
  if (e == cudaSuccess) {
    zr::Ctrl c = initial_ctrl(p->scaler);
    e = cudaMemcpy(p->ctrl_dev, &c, sizeof c, cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) {
    p->kernel = p->dtype == ZR_F16 ? pick_kernel<zr::DT_F16>(p->W, p->A) : pick_kernel<zr::DT_BF16>(p->W, p->A);
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, p->kernel, kThreads, 0);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e == cudaSuccess) {
      if (per_sm < 1) per_sm = 1;
      const int64_t full = (int64_t)sms * per_sm;
      p->grid = (int)(p->ntiles < full ? (p->ntiles > 0 ? p->ntiles : 1) : full);
    }
  }
  if (e != cudaSuccess) {
    zr_status s = cuda_fail("zr_plan_create", e);
    zr_plan_destroy(p);
    return s;
  }
  *out = p;
  return ZR_OK;
}

extern "C" zr_status zr_plan_destroy(zr_plan* p) {
  if (!p) return ZR_OK;
  if (p->tiles_dev) cudaFree(p->tiles_dev);
  if (p->ctrl_dev) cudaFree(p->ctrl_dev);
  delete p;
  return ZR_OK;
}

extern "C" int64_t zr_plan_numel(const zr_plan* p) { return p ? p->numel : -1; }
extern "C" int32_t zr_plan_nbuckets(const zr_plan* p) { return p ? (int32_t)p->buckets.size() : -1; }

extern "C" zr_status zr_plan_buckets(const zr_plan* p, zr_bucket* buckets, int64_t* tensor_offsets) {
  zr::clear_error();
  if (!p) return fail(ZR_ERR_INVALID, "zr_plan_buckets: null plan");
  if (buckets) std::memcpy(buckets, p->buckets.data(), p->buckets.size() * sizeof(zr_bucket));
  if (tensor_offsets)
    std::memcpy(tensor_offsets, p->tensor_offsets.data(), p->tensor_offsets.size() * sizeof(int64_t));
  return ZR_OK;
}

extern "C" zr_status zr_plan_reset(zr_plan* p, void* stream) {
  zr::clear_error();
  if (!p) return fail(ZR_ERR_INVALID, "zr_plan_reset: null plan");
  zr::Ctrl c = initial_ctrl(p->scaler);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(p->ctrl_dev, &c, sizeof c, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? ZR_OK : cuda_fail("zr_plan_reset", e);
}

extern "C" zr_status zr_plan_report(zr_plan* p, void* stream, zr_step_report* rep) {
  zr::clear_error();
  if (!p || !rep) return fail(ZR_ERR_INVALID, "zr_plan_report: null argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  zr::Ctrl c;
  cudaError_t e = cudaMemcpyAsync(&c, p->ctrl_dev, sizeof c, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("zr_plan_report", e);
  rep->overflow = c.last_overflow;
  rep->skipped = c.last_overflow;
  rep->current = c.k;
  rep->stage = c.stage;
  rep->scale_used = c.scale_used;
  rep->scale = c.scale;
  rep->t = c.t;
  rep->steps = c.steps;
  rep->skipped_total = c.skipped;
  rep->good = c.good;
  rep->n_real = p->n_real;
  rep->bytes_alg = (int64_t)(2 * p->W * p->A + 26) * p->n_real;
  return ZR_OK;
}

static zr_status check_step_args(const zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                                 const zr_adamw_hyper* h) {
  if (!p || !st || !h || !grads) return fail(ZR_ERR_INVALID, "zr_step: null argument");
  if (stage < 1 || stage > 3) return fail(ZR_ERR_INVALID, "zr_step: stage=%d not in 1..3", stage);
  for (int r = 0; r < p->W * p->A; ++r)
    if (!grads[r] || !zr::aligned16(grads[r])) return fail(ZR_ERR_INVALID, "zr_step: grads[%d] null or misaligned", r);
  for (int k = 0; k < 2; ++k) {
    if (!st->master[k] || !st->m[k] || !st->v[k] || !st->param[k])
      return fail(ZR_ERR_INVALID, "zr_step: state set %d has a null array", k);
    if (!zr::aligned16(st->master[k]) || !zr::aligned16(st->m[k]) || !zr::aligned16(st->v[k]) ||
        !zr::aligned16(st->param[k]))
      return fail(ZR_ERR_INVALID, "zr_step: state set %d misaligned", k);
  }
  if (st->master[0] == st->master[1] || st->m[0] == st->m[1] || st->v[0] == st->v[1] || st->param[0] == st->param[1])
    return fail(ZR_ERR_INVALID, "zr_step: the two state sets must be distinct buffers");
  return ZR_OK;
}

static zr_status launch_step(zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                             const zr_adamw_hyper* h, cudaStream_t s) {
  if (p->ntiles == 0) return ZR_OK;
  FusedArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < p->W * p->A; ++r) a.grads[r] = static_cast<const uint16_t*>(grads[r]);
  for (int i = 0; i < p->W; ++i) a.order[i] = p->order[i];
  a.tiles = p->tiles_dev;
  a.ntiles = p->ntiles;
  for (int k = 0; k < 2; ++k) {
    a.master[k] = st->master[k];
    a.m[k] = st->m[k];
    a.v[k] = st->v[k];
    a.param[k] = static_cast<uint16_t*>(st->param[k]);
  }
  a.ctrl = p->ctrl_dev;
  a.lr = h->lr;
  a.beta1 = h->beta1;
  a.beta2 = h->beta2;
  a.eps = h->eps;
  a.weight_decay = h->weight_decay;
  a.W = p->W;
  a.A = p->A;
  a.stage = stage;
  p->kernel<<<p->grid, kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ZR_OK : fail(ZR_ERR_CUDA, "zr_step: launch failed: %s", cudaGetErrorString(e));
}

extern "C" zr_status zr_step(zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                             const zr_adamw_hyper* h, void* stream, zr_step_report* rep) {
  zr::clear_error();
  zr_status s = check_step_args(p, stage, grads, st, h);
  if (s != ZR_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  s = launch_step(p, stage, grads, st, h, cs);
  if (s != ZR_OK || !rep) return s;
  return zr_plan_report(p, stream, rep);
}

extern "C" zr_status zr_step_from_host(zr_plan* p, int stage, const void* const* host_grads, void* const* dev_grads,
                                       const zr_state* st, const zr_adamw_hyper* h, void* stream,
                                       zr_step_report* rep) {
  zr::clear_error();
  if (!p || !host_grads || !dev_grads || !rep) return fail(ZR_ERR_INVALID, "zr_step_from_host: null argument");
  const int R = p->W * p->A;
  for (int r = 0; r < R; ++r)
    if (!host_grads[r]) return fail(ZR_ERR_INVALID, "zr_step_from_host: host_grads[%d] is null", r);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // Page-locked host memory the device can address (cudaHostAlloc, cudaHostRegister) is read
  // in place by the step kernel: each byte crosses the host link once and the HBM half of
  // the step overlaps the transfer. Anything else is copied into dev_grads first.
  bool direct = true;
  const void* mapped[ZR_MAX_REPLICAS];
  for (int r = 0; r < R && direct; ++r) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, host_grads[r]) != cudaSuccess) {
      cudaGetLastError();  // clear the sticky-free error of an unknown pointer
      direct = false;
    } else if (at.type != cudaMemoryTypeHost || !at.devicePointer) {
      direct = false;
    } else {
      mapped[r] = at.devicePointer;
    }
  }
  if (direct) {
    zr_status s = check_step_args(p, stage, mapped, st, h);
    if (s != ZR_OK) return s;
    s = launch_step(p, stage, mapped, st, h, cs);
    if (s != ZR_OK) return s;
    return zr_plan_report(p, stream, rep);
  }
  zr_status s = check_step_args(p, stage, const_cast<const void* const*>(dev_grads), st, h);
  if (s != ZR_OK) return s;
  for (const zr_bucket& b : p->buckets) {
    for (int r = 0; r < R; ++r) {
      const size_t off = (size_t)b.start * 2, bytes = (size_t)b.len * 2;
      cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dev_grads[r]) + off,
                                      static_cast<const char*>(host_grads[r]) + off, bytes,
                                      cudaMemcpyHostToDevice, cs);
      if (e != cudaSuccess) return cuda_fail("zr_step_from_host: copy", e);
    }
  }
  s = launch_step(p, stage, const_cast<const void* const*>(dev_grads), st, h, cs);
  if (s != ZR_OK) return s;
  return zr_plan_report(p, stream, rep);
}
