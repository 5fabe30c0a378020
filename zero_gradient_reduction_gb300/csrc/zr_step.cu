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

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "zr_device.cuh"
#include "zr_internal.h"
#include "zr_nvtx.h"

using zr::fail;

namespace zr {
void take_cuda_error() { (void)cudaGetLastError(); }
}  // namespace zr

#include "zr_plan.h"
#include "zr_step_kernel.cuh"
#include "zr_step_bulk.cuh"
#include "zr_step_bulk_chunked.cuh"

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

// Blocks of each zr_step_bucket launch: one per tile (or a persistent grid for a small
// bucket), capped at max_blocks if that is > 0; a step's launches add up to bucket_blocks.
static void set_bucket_grids(zr_plan* p, int max_blocks) {
  p->bucket_grid.clear();
  p->bucket_blocks = 0;
  for (size_t b = 0; b + 1 < p->tile_begin.size(); ++b) {
    const int64_t nt = p->tile_begin[b + 1] - p->tile_begin[b];
    int g = nt > 0 ? zr::step_grid(p, nt) : 0;  // a bucket without tiles launches nothing
    if (max_blocks > 0 && g > max_blocks) g = max_blocks;
    p->bucket_grid.push_back(g);
    p->bucket_blocks += (unsigned)g;
  }
}

// Automatic shape: two blocks per SM (at most kBulkBudget of shared memory each, which with
// the per-block reserve fills an SM's 228 KB), stages of 2048 elements (one 8-element group
// per consumer thread) where two of them fit, else smaller; as many stages as the budget
// holds, up to kBulkMaxStages. Measured on the 7B (W = 2) and 1.3B (W = 8) workloads:
// 2048 x 3 and 2048 x 2 beat every other shape, and smaller stages (1024) or one block per
// SM (4096) lose 10-25 %.
void zr::bulk_auto_shape(int R, int* E, int* NS) {
  constexpr int kBulkBudget = 113 * 1024;
  if (*E == 0) {
    *E = 2048;
    while (*E > 256 && 2 * bulk_stage_bytes(R, *E) > kBulkBudget) *E /= 2;
  }
  if (*NS == 0) {  // a stage larger than the budget (hundreds of replica slices) runs alone on its SM
    const int ns = kBulkBudget / bulk_stage_bytes(R, *E);
    *NS = ns < 1 ? 1 : ns > kBulkMaxStages ? kBulkMaxStages : ns;
  }
}

// Bulk staging is chosen where the automatic shape keeps stages of 2048 elements (W * A <=
// 8: every consumer thread gets one 8-element group per stage) and the plan streams from HBM
// (at least four waves of tiles): measured 0.6-1.2 % faster than register staging on the 7B
// (W = 2), 1.3B (W = 8) and W = 2, A = 4 workloads. With more replica slices the stages
// shrink, consumers sit idle and bulk staging loses (W = 4, A = 4: 11.9 against 10.6 ms;
// W = 8, A = 4: 27.5 against 17.4 ms). A small plan is launch-bound, and there the ring's
// fill costs more than it hides (the 786,432-param workload: 14.5 us against 12.5 us).
bool zr::bulk_preferred(int E, int64_t ntiles, int64_t resident) { return E >= 2048 && ntiles >= 4 * resident; }

// Automatic shape of the chunked stages (more than kChunkSlices replica slices per element):
// 2048 elements, as many stages as kBulkBudget holds (two of 56 KB), up to kBulkMaxStages.
static void chunked_auto_shape(int* E, int* NS) {
  constexpr int kBulkBudget = 113 * 1024;
  if (*E == 0) *E = kChunkMaxElems;
  if (*NS == 0) {
    const int ns = kBulkBudget / chunked_stage_bytes(*E);
    *NS = ns < 1 ? 1 : ns > kBulkMaxStages ? kBulkMaxStages : ns;
  }
}

// Chooses how zr_step stages its loads (the body of zr_plan_set_staging; zr_plan_create
// also calls it to make bulk staging the default where it applies).
static zr_status configure_staging(zr_plan* p, int staging, int stage_elems, int stages) {
  if (staging == ZR_STAGING_REGISTERS) {
    p->staging = ZR_STAGING_REGISTERS;
    return ZR_OK;
  }
  if (staging != ZR_STAGING_BULK && staging != ZR_STAGING_BULK_IO)
    return fail(ZR_ERR_INVALID, "zr_plan_set_staging: unknown staging %d", staging);
  const bool sb = staging == ZR_STAGING_BULK_IO;
  if (p->fp32_grads) return fail(ZR_ERR_UNSUPPORTED, "zr_plan_set_staging: bulk staging needs 16-bit gradients");
  const int R = p->W * p->A;  // replica slices per element
  // more slices than one stage takes: the chunked kernel spreads them over consecutive stages
  const bool chunked = !sb && R > kChunkSlices;
  const int max_elems = chunked ? kChunkMaxElems : 65536;
  if (stage_elems < 0 || (stage_elems % 8) != 0 || stage_elems > max_elems)
    return fail(ZR_ERR_INVALID, "zr_plan_set_staging: stage_elems must be 0 or a multiple of 8 up to %d%s", max_elems,
                chunked ? " (stages of 8 replica slices)" : "");
  if (stages < 0 || stages > kBulkMaxStages)
    return fail(ZR_ERR_INVALID, "zr_plan_set_staging: stages must be 0 or 1..%d", kBulkMaxStages);
  int E = stage_elems, NS = stages;
  if (chunked) chunked_auto_shape(&E, &NS);
  else zr::bulk_auto_shape(R, &E, &NS);
  const int64_t smem64 = (int64_t)NS * (chunked ? chunked_stage_bytes(E) : bulk_stage_bytes(R, E));
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, p->device);
  if (e != cudaSuccess) return cuda_fail("zr_plan_set_staging", e);
  if (smem64 > optin)
    return fail(ZR_ERR_UNSUPPORTED, "zr_plan_set_staging: %d stages of %d elements need %lld bytes of shared memory "
                "(a block may have %d)", NS, E, (long long)smem64, optin);
  const int smem = (int)smem64;
  BulkKernelFn k = sb ? (p->dtype == ZR_F16 ? pick_bulk_kernel<zr::DT_F16, true>(p->W, p->A)
                                            : pick_bulk_kernel<zr::DT_BF16, true>(p->W, p->A))
                 : chunked ? (p->dtype == ZR_F16 ? pick_chunked_kernel<zr::DT_F16>(p->A)
                                                 : pick_chunked_kernel<zr::DT_BF16>(p->A))
                      : (p->dtype == ZR_F16 ? pick_bulk_kernel<zr::DT_F16, false>(p->W, p->A)
                                            : pick_bulk_kernel<zr::DT_BF16, false>(p->W, p->A));
  const int threads = bulk_threads(sb);
  int per_sm = 0, sms = 0;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
  if (e != cudaSuccess) return cuda_fail("zr_plan_set_staging", e);
  if (per_sm < 1)
    return fail(ZR_ERR_UNSUPPORTED, "zr_plan_set_staging: %d stages of %d elements (%d bytes) do not fit an SM", NS, E,
                smem);
  const int64_t resident = (int64_t)sms * per_sm, nt = p->ntiles;
  int grid = 1;
  if (nt >= 4 * resident) grid = (int)(nt < (1 << 30) ? nt : (1 << 30));
  else if (nt > 0) grid = (int)(nt < resident ? nt : resident);
  p->bulk_kernel = reinterpret_cast<void*>(k);
  p->bulk_E = E;
  p->bulk_NS = NS;
  p->bulk_smem = smem;
  p->bulk_grid = grid;
  p->bulk_threads = threads;
  p->bulk_resident = resident;
  p->staging = staging;
  return ZR_OK;
}

extern "C" zr_status zr_plan_set_staging(zr_plan* p, int staging, int stage_elems, int stages) {
  zr::clear_error();
  if (!p) return fail(ZR_ERR_INVALID, "zr_plan_set_staging: null plan");
  return configure_staging(p, staging, stage_elems, stages);
}

extern "C" int zr_plan_staging(const zr_plan* p) { return p ? p->staging : -1; }

extern "C" zr_status zr_plan_stall_bulk_waits(zr_plan* p, int on) {
  zr::clear_error();
  if (!p) return fail(ZR_ERR_INVALID, "zr_plan_stall_bulk_waits: null plan");
  p->bulk_stall = on ? 1 : 0;
  return ZR_OK;
}

extern "C" zr_status zr_plan_create(const zr_plan_desc* d, zr_plan** out) {
  zr::clear_error();
  if (!d || !out) return fail(ZR_ERR_INVALID, "zr_plan_create: null argument");
  *out = nullptr;
  if (d->W < 1 || d->W > ZR_MAX_W) return fail(ZR_ERR_INVALID, "zr_plan_create: W=%d outside [1, %d]", d->W, ZR_MAX_W);
  if (d->A < 1 || (int64_t)d->W * d->A > ZR_MAX_REPLICAS)
    return fail(ZR_ERR_INVALID, "zr_plan_create: A=%d (W*A must be in [1, %d])", d->A, ZR_MAX_REPLICAS);
  if (d->dtype != ZR_F16 && d->dtype != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_plan_create: dtype must be F16 or BF16");
  if (d->stage < 0 || d->stage > 3) return fail(ZR_ERR_INVALID, "zr_plan_create: stage=%d not in 0..3", d->stage);
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
  p->fp32_grads = d->fp32_grads ? 1 : 0;
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

  // Kernel for (dtype, W, A) and the number of its blocks that fit on the GPU at once.
  const bool f32 = p->fp32_grads != 0;
  KernelFn k = p->dtype == ZR_F16 ? pick_kernel<zr::DT_F16, kPingPong>(p->W, p->A, f32)
                                  : pick_kernel<zr::DT_BF16, kPingPong>(p->W, p->A, f32);
  p->kernel = reinterpret_cast<void*>(k);
  int per_sm = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&p->device);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kThreads, 0);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, p->device);
  if (per_sm < 1) per_sm = 1;
  const int64_t full = (int64_t)(sms > 0 ? sms : 1) * per_sm;

  // Tile schedule: every block of every bucket cut into pieces of at most `tile` elements.
  // A large plan takes kTileElems, one thread block per tile (step_grid). A plan of fewer
  // than four waves of such tiles runs at most `full` blocks at once and its slowest block
  // sets the time, so its tile is the multiple of one block iteration (8 * kThreads * U
  // elements, U groups per thread) up to kTileElems with the fewest waves x iterations
  // per tile, ties going to the larger tile: no last wave and no iteration runs mostly
  // empty.
  int64_t tile = kTileElems;
  if (p->numel < 4 * full * kTileElems) {
    const int64_t iter = 8 * kThreads * ((!f32 && p->A == 1 && p->W <= 3) ? 2 : 1);
    std::vector<int64_t> pieces;
    for (const zr_bucket& b : p->buckets)
      for (int c = 0; c < p->W; ++c) {
        const int64_t end = b.start + b.len;
        const int64_t lo = std::min(b.start + (int64_t)c * b.chunk, end), hi = std::min(lo + b.chunk, end);
        if (hi > lo) pieces.push_back(hi - lo);
      }
    int64_t best = -1;
    for (int64_t t = iter; t <= kTileElems && pieces.size() <= 65536; t += iter) {
      int64_t nt = 0;
      for (int64_t len : pieces) nt += (len + t - 1) / t;
      const int64_t cost = (nt + full - 1) / full * (t / iter);
      if (best < 0 || cost <= best) {
        best = cost;
        tile = t;
      }
    }
  }
  std::vector<int4> tiles;
  for (const zr_bucket& b : p->buckets) {
    p->tile_begin.push_back((int64_t)tiles.size());
    for (int c = 0; c < p->W; ++c) {
      int64_t lo = b.start + (int64_t)c * b.chunk, hi = lo + b.chunk;
      const int64_t end = b.start + b.len;
      if (lo > end) lo = end;
      if (hi > end) hi = end;
      for (int64_t x = lo; x < hi; x += tile) {
        const int64_t len = (hi - x) < tile ? (hi - x) : tile;
        tiles.push_back(make_int4((int)(uint32_t)(uint64_t)x, (int)(uint32_t)((uint64_t)x >> 32), (int)(len / 8), c));
      }
    }
  }
  p->ntiles = (int64_t)tiles.size();
  p->tile_begin.push_back(p->ntiles);
  p->resident = full;
  p->grid = zr::step_grid(p, p->ntiles);
  set_bucket_grids(p, 0);
  if (e == cudaSuccess && !tiles.empty()) e = cudaMalloc(&p->tiles_dev, tiles.size() * sizeof(int4));
  if (e == cudaSuccess && !tiles.empty())
    e = cudaMemcpy(p->tiles_dev, tiles.data(), tiles.size() * sizeof(int4), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMalloc(&p->ctrl_dev, sizeof(zr::Ctrl));
  if (e == cudaSuccess) {
    zr::Ctrl c = initial_ctrl(p->scaler);
    e = cudaMemcpy(p->ctrl_dev, &c, sizeof c, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) {
    zr_status s = cuda_fail("zr_plan_create", e);
    zr_plan_destroy(p);
    return s;
  }
  zr_status ss = zr::build_shard_tables(p);
  if (ss == ZR_OK) ss = zr::init_inplace(p);
  if (ss != ZR_OK) {
    zr_plan_destroy(p);
    return ss;
  }
  // zr_step stages its loads by bulk copies where zr::bulk_preferred says so; other plans
  // keep register staging, and so do plans with more than kChunkSlices replica slices per
  // element, whose chunked bulk stages measured as fast as register staging at best.
  if (!p->fp32_grads && p->ntiles > 0) {
    if (p->W * p->A > kChunkSlices || configure_staging(p, ZR_STAGING_BULK, 0, 0) != ZR_OK ||
        !zr::bulk_preferred(p->bulk_E, p->ntiles, p->bulk_resident))
      p->staging = ZR_STAGING_REGISTERS;
    zr::clear_error();
  }
  *out = p;
  return ZR_OK;
}

extern "C" zr_status zr_plan_destroy(zr_plan* p) {
  if (!p) return ZR_OK;
  if (p->tiles_dev) cudaFree(p->tiles_dev);
  if (p->ctrl_dev) cudaFree(p->ctrl_dev);
  if (p->shard_tiles_dev) cudaFree(p->shard_tiles_dev);
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
  if (c.error)
    return fail(ZR_ERR_TIMEOUT, "zr_plan_report: a wait of the bulk-staged step gave up; that step was skipped "
                "(state unchanged); zr_plan_reset clears the error");
  return ZR_OK;
}

extern "C" zr_status zr_plan_checkpoint(zr_plan* p, void* stream, zr_checkpoint* out) {
  zr::clear_error();
  if (!p || !out) return fail(ZR_ERR_INVALID, "zr_plan_checkpoint: null argument");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  zr::Ctrl c;
  cudaError_t e = cudaMemcpyAsync(&c, p->ctrl_dev, sizeof c, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail("zr_plan_checkpoint", e);
  out->current = c.k;
  out->scale = c.scale;
  out->good = c.good;
  out->t = c.t;
  out->steps = c.steps;
  out->skipped = c.skipped;
  out->beta1_pow = c.prod1;
  out->beta2_pow = c.prod2;
  return ZR_OK;
}

extern "C" zr_status zr_plan_restore(zr_plan* p, const zr_checkpoint* in, void* stream) {
  zr::clear_error();
  if (!p || !in) return fail(ZR_ERR_INVALID, "zr_plan_restore: null argument");
  if (in->current != 0 && in->current != 1) return fail(ZR_ERR_INVALID, "zr_plan_restore: current must be 0 or 1");
  if (!(in->scale > 0.0f) || !std::isfinite(in->scale))
    return fail(ZR_ERR_INVALID, "zr_plan_restore: scale must be positive and finite");
  if (in->good < 0 || in->t < 0 || in->steps < 0 || in->skipped < 0)
    return fail(ZR_ERR_INVALID, "zr_plan_restore: negative counter");
  // running products of betas in [0, 1): a value outside [0, 1] (or NaN) is no such product
  if (!(in->beta1_pow >= 0.0 && in->beta1_pow <= 1.0) || !(in->beta2_pow >= 0.0 && in->beta2_pow <= 1.0))
    return fail(ZR_ERR_INVALID, "zr_plan_restore: beta powers must lie in [0, 1]");
  zr::Ctrl c = initial_ctrl(p->scaler);
  c.k = in->current;
  c.scale = in->scale;
  c.scale_used = in->scale;
  c.good = in->good;
  c.t = in->t;
  c.steps = in->steps;
  c.skipped = in->skipped;
  c.prod1 = in->beta1_pow;
  c.prod2 = in->beta2_pow;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(p->ctrl_dev, &c, sizeof c, cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? ZR_OK : cuda_fail("zr_plan_restore", e);
}

static zr_status check_step_args(const zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                                 const zr_adamw_hyper* h) {
  if (!p || !st || !h || !grads) return fail(ZR_ERR_INVALID, "zr_step: null argument");
  if (stage < 0 || stage > 3) return fail(ZR_ERR_INVALID, "zr_step: stage=%d not in 0..3", stage);
  if (p->numel == 0) return ZR_OK;  // no parameters: the arrays are empty and may be null
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

// One launch of the fused kernel over tiles [tile0, tile1) with `grid` blocks; the step's
// launches add up to `total` blocks, and the last of those blocks decides the step. A plan
// with no parameters has no tiles: its step is one block that only runs that decision
// (a clean step), as the method's step over nothing is.
static zr_status launch_step(zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                             const zr_adamw_hyper* h, cudaStream_t s, int64_t tile0, int64_t tile1, int grid,
                             unsigned total) {
  if (tile1 < tile0 || (tile1 == tile0 && p->ntiles > 0) || grid < 1) return ZR_OK;
  const FusedArgs a = make_args(p, stage, grads, st->master, st->m, st->v, st->param, h, tile0, tile1, total);
  reinterpret_cast<KernelFn>(p->kernel)<<<grid, kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ZR_OK : fail(ZR_ERR_CUDA, "zr_step: launch failed: %s", cudaGetErrorString(e));
}

extern "C" zr_status zr_step(zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                             const zr_adamw_hyper* h, void* stream, zr_step_report* rep) {
  zr::Range range("zr_step");
  zr::clear_error();
  zr_status s = check_step_args(p, stage, grads, st, h);
  if (s != ZR_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (p->staging != ZR_STAGING_REGISTERS && p->ntiles > 0) {
    const FusedArgs a = make_args(p, stage, grads, st->master, st->m, st->v, st->param, h, 0, p->ntiles,
                                  (unsigned)p->bulk_grid);
    const BulkCfg cfg{p->bulk_E, p->bulk_NS, p->bulk_stall ? 16u : 0u};
    reinterpret_cast<BulkKernelFn>(p->bulk_kernel)<<<p->bulk_grid, p->bulk_threads, p->bulk_smem, cs>>>(a, cfg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step: launch failed: %s", cudaGetErrorString(e));
  } else {
    s = launch_step(p, stage, grads, st, h, cs, 0, p->ntiles, p->grid, (unsigned)p->grid);
  }
  if (s != ZR_OK || !rep) return s;
  return zr_plan_report(p, stream, rep);
}


extern "C" zr_status zr_step_bucket(zr_plan* p, int stage, int bucket, const void* const* grads, const zr_state* st,
                                    const zr_adamw_hyper* h, void* stream) {
  zr::Range range("zr_step_bucket");
  zr::clear_error();
  zr_status s = check_step_args(p, stage, grads, st, h);
  if (s != ZR_OK) return s;
  if (bucket < 0 || bucket >= (int)p->buckets.size())
    return fail(ZR_ERR_INVALID, "zr_step_bucket: bucket %d outside [0, %d)", bucket, (int)p->buckets.size());
  return launch_step(p, stage, grads, st, h, static_cast<cudaStream_t>(stream), p->tile_begin[bucket],
                     p->tile_begin[bucket + 1], p->bucket_grid[bucket], p->bucket_blocks);
}

extern "C" zr_status zr_plan_set_bucket_blocks(zr_plan* p, int max_blocks) {
  zr::clear_error();
  if (!p) return fail(ZR_ERR_INVALID, "zr_plan_set_bucket_blocks: null plan");
  if (max_blocks < 0) return fail(ZR_ERR_INVALID, "zr_plan_set_bucket_blocks: max_blocks=%d < 0", max_blocks);
  set_bucket_grids(p, max_blocks);
  return ZR_OK;
}

extern "C" zr_status zr_step_from_host(zr_plan* p, int stage, const void* const* host_grads, void* const* dev_grads,
                                       const zr_state* st, const zr_adamw_hyper* h, void* stream,
                                       zr_step_report* rep) {
  zr::Range range("zr_step_from_host");
  zr::clear_error();
  if (!p || !host_grads || !dev_grads || !rep) return fail(ZR_ERR_INVALID, "zr_step_from_host: null argument");
  const int R = p->W * p->A;
  for (int r = 0; r < R && p->numel > 0; ++r)
    if (!host_grads[r]) return fail(ZR_ERR_INVALID, "zr_step_from_host: host_grads[%d] is null", r);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // Page-locked host memory the device can address (cudaHostAlloc, cudaHostRegister) is read
  // in place by the step kernel: each byte crosses the host link once and the HBM half of
  // the step overlaps the transfer. Anything else is copied into dev_grads first.
  bool direct = p->numel > 0;
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
    s = launch_step(p, stage, mapped, st, h, cs, 0, p->ntiles, p->grid, (unsigned)p->grid);
    if (s != ZR_OK) return s;
    return zr_plan_report(p, stream, rep);
  }
  zr_status s = check_step_args(p, stage, const_cast<const void* const*>(dev_grads), st, h);
  if (s != ZR_OK) return s;
  for (const zr_bucket& b : p->buckets) {
    for (int r = 0; r < R; ++r) {
      const size_t esz = p->fp32_grads ? 4 : 2;
      const size_t off = (size_t)b.start * esz, bytes = (size_t)b.len * esz;
      cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dev_grads[r]) + off,
                                      static_cast<const char*>(host_grads[r]) + off, bytes,
                                      cudaMemcpyHostToDevice, cs);
      if (e != cudaSuccess) return cuda_fail("zr_step_from_host: copy", e);
    }
  }
  s = launch_step(p, stage, const_cast<const void* const*>(dev_grads), st, h, cs, 0, p->ntiles, p->grid,
                  (unsigned)p->grid);
  if (s != ZR_OK) return s;
  return zr_plan_report(p, stream, rep);
}
