// ZeRO-3 parameter sharding and the parameter all-gather that precedes forward and
// backward. A ZeRO-3 worker keeps only its own block of every bucket of the 16-bit
// parameters; before a layer runs, the layer's buckets are all-gathered from the W
// shards into a transient full replica, used and dropped. Both directions are tiled
// 16-byte copies over a per-plan table of (bucket, block) pieces: 2 bytes read and 2
// bytes written per parameter, an HBM copy.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <vector>

#include "zr_device.cuh"
#include "zr_internal.h"
#include "zr_nvtx.h"
#include "zr_plan.h"

using zr::fail;

namespace {

constexpr int kThreads = 256;
constexpr int kShardTileElems = 16384;
constexpr int kGroupsPerIter = 4;  // 16-byte copies in flight per thread

struct ShardArgs {
  uint16_t* shards[ZR_MAX_W];  // by worker id
  uint16_t* replica;
  const int4* tiles;           // two int4 per tile
  int64_t t0, t1;              // tile range
};

// GATHER: shards -> replica (the all-gather before forward/backward);
// otherwise replica -> shards (what a ZeRO-3 worker keeps after the step).
template <bool GATHER>
__global__ void __launch_bounds__(kThreads) shard_copy_kernel(const __grid_constant__ ShardArgs a) {
  for (int64_t t = a.t0 + blockIdx.x; t < a.t1; t += gridDim.x) {
    const int4 d0 = a.tiles[2 * t], d1 = a.tiles[2 * t + 1];
    const int64_t flat = (int64_t)(((uint64_t)(uint32_t)d0.y << 32) | (uint32_t)d0.x);
    const int64_t sh = (int64_t)(((uint64_t)(uint32_t)d0.w << 32) | (uint32_t)d0.z);
    const int groups = d1.x;
    uint16_t* rep = a.replica + flat;
    uint16_t* shd = a.shards[d1.y] + sh;
    const uint16_t* src = GATHER ? shd : rep;
    uint16_t* dst = GATHER ? rep : shd;
    for (int g0 = threadIdx.x; g0 < groups; g0 += kGroupsPerIter * blockDim.x) {
      uint4 v[kGroupsPerIter];
#pragma unroll
      for (int u = 0; u < kGroupsPerIter; ++u) {
        const int g = g0 + u * (int)blockDim.x;
        if (g < groups) v[u] = zr::ld_once(src + (int64_t)g * 8);
      }
#pragma unroll
      for (int u = 0; u < kGroupsPerIter; ++u) {
        const int g = g0 + u * (int)blockDim.x;
        if (g < groups) zr::st_once(dst + (int64_t)g * 8, v[u]);
      }
    }
  }
}

zr_status launch_copy(zr_plan* p, bool gather, int64_t t0, int64_t t1, void* const* shards, void* replica,
                      void* stream, const char* what) {
  if (t1 <= t0) return ZR_OK;
  ShardArgs a;
  std::memset(&a, 0, sizeof a);
  for (int w = 0; w < p->W; ++w) a.shards[w] = static_cast<uint16_t*>(shards[w]);
  a.replica = static_cast<uint16_t*>(replica);
  a.tiles = p->shard_tiles_dev;
  a.t0 = t0;
  a.t1 = t1;
  // One block per tile, handed out in index order (see step_grid).
  const int64_t want = t1 - t0, cap = (int64_t)1 << 30;
  const int grid = (int)(want < cap ? want : cap);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (gather) shard_copy_kernel<true><<<grid, kThreads, 0, s>>>(a);
  else shard_copy_kernel<false><<<grid, kThreads, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? ZR_OK : fail(ZR_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
}

zr_status check_shards(const zr_plan* p, const void* const* shards, const void* replica, const char* what) {
  if (!p || !shards || !replica) return fail(ZR_ERR_INVALID, "%s: null argument", what);
  if (!zr::aligned16(replica)) return fail(ZR_ERR_INVALID, "%s: replica misaligned", what);
  for (int w = 0; w < p->W; ++w)
    if (!shards[w] || !zr::aligned16(shards[w])) return fail(ZR_ERR_INVALID, "%s: shard %d null or misaligned", what, w);
  return ZR_OK;
}

}  // namespace

namespace zr {

zr_status build_shard_tables(zr_plan* p) {
  const int W = p->W;
  const size_t nb = p->buckets.size();
  p->shard_numel.assign(W, 0);
  p->shard_off.assign(nb * W, 0);
  p->shard_tile_begin.assign(nb + 1, 0);
  auto block = [](const zr_bucket& b, int c, int64_t& lo, int64_t& hi) {
    lo = (int64_t)c * b.chunk;
    hi = lo + b.chunk;
    if (lo > b.len) lo = b.len;
    if (hi > b.len) hi = b.len;
  };
  for (size_t b = 0; b < nb; ++b) {
    for (int pos = 0; pos < W; ++pos) {
      const int w = p->order[pos];
      int64_t lo, hi;
      block(p->buckets[b], (pos + 1) % W, lo, hi);
      p->shard_off[b * W + w] = p->shard_numel[w];
      p->shard_numel[w] += hi - lo;
    }
  }
  std::vector<int4> tiles;
  for (size_t b = 0; b < nb; ++b) {
    p->shard_tile_begin[b] = (int64_t)(tiles.size() / 2);
    const zr_bucket& bk = p->buckets[b];
    for (int c = 0; c < W; ++c) {
      const int w = p->order[(c - 1 + W) % W];  // the position before c owns block c
      int64_t lo, hi;
      block(bk, c, lo, hi);
      for (int64_t x = lo; x < hi; x += kShardTileElems) {
        const int64_t len = (hi - x) < kShardTileElems ? (hi - x) : kShardTileElems;
        const uint64_t flat = (uint64_t)(bk.start + x), sh = (uint64_t)(p->shard_off[b * W + w] + (x - lo));
        tiles.push_back(make_int4((int)(uint32_t)flat, (int)(uint32_t)(flat >> 32), (int)(uint32_t)sh,
                                  (int)(uint32_t)(sh >> 32)));
        tiles.push_back(make_int4((int)(len / 8), w, 0, 0));
      }
    }
  }
  p->shard_tile_begin[nb] = (int64_t)(tiles.size() / 2);
  p->nshard_tiles = (int64_t)(tiles.size() / 2);
  if (tiles.empty()) return ZR_OK;
  cudaError_t e = cudaMalloc(&p->shard_tiles_dev, tiles.size() * sizeof(int4));
  if (e == cudaSuccess)
    e = cudaMemcpy(p->shard_tiles_dev, tiles.data(), tiles.size() * sizeof(int4), cudaMemcpyHostToDevice);
  if (e != cudaSuccess)
    return fail(e == cudaErrorMemoryAllocation ? ZR_ERR_OOM : ZR_ERR_CUDA, "zr_plan_create: shard table: %s",
                cudaGetErrorString(e));
  return ZR_OK;
}

}  // namespace zr

extern "C" int64_t zr_plan_shard_numel(const zr_plan* p, int worker) {
  if (!p || worker < 0 || worker >= p->W) return -1;
  return p->shard_numel[worker];
}

extern "C" zr_status zr_plan_shard_offset(const zr_plan* p, int bucket, int worker, int64_t* offset) {
  zr::clear_error();
  if (!p || !offset) return fail(ZR_ERR_INVALID, "zr_plan_shard_offset: null argument");
  if (bucket < 0 || bucket >= (int)p->buckets.size() || worker < 0 || worker >= p->W)
    return fail(ZR_ERR_INVALID, "zr_plan_shard_offset: bucket or worker out of range");
  *offset = p->shard_off[(size_t)bucket * p->W + worker];
  return ZR_OK;
}

extern "C" zr_status zr_shard_params(zr_plan* p, const void* replica, void* const* shards, void* stream) {
  zr::Range range("zr_shard_params");
  zr::clear_error();
  zr_status s = check_shards(p, const_cast<const void* const*>(shards), replica, "zr_shard_params");
  if (s != ZR_OK) return s;
  return launch_copy(p, false, 0, p->nshard_tiles, shards, const_cast<void*>(replica), stream, "zr_shard_params");
}

extern "C" zr_status zr_gather_params(zr_plan* p, int bucket_lo, int bucket_hi, const void* const* shards,
                                      void* replica, void* stream) {
  zr::Range range("zr_gather_params");
  zr::clear_error();
  zr_status s = check_shards(p, shards, replica, "zr_gather_params");
  if (s != ZR_OK) return s;
  const int nb = (int)p->buckets.size();
  if (bucket_lo < 0 || bucket_hi > nb || bucket_lo > bucket_hi)
    return fail(ZR_ERR_INVALID, "zr_gather_params: bucket range [%d, %d) outside [0, %d]", bucket_lo, bucket_hi, nb);
  return launch_copy(p, true, p->shard_tile_begin[bucket_lo], p->shard_tile_begin[bucket_hi],
                     const_cast<void* const*>(shards), replica, stream, "zr_gather_params");
}
