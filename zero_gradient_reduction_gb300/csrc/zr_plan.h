// The plan object behind the zr_plan handle (host side, internal to libzr).
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "zr_internal.h"

struct zr_plan {
  int W = 0, A = 0, stage = 0, align = 0;
  zr_dtype dtype = ZR_BF16;
  int64_t numel = 0, n_real = 0;
  std::vector<zr_bucket> buckets;
  std::vector<int64_t> tensor_offsets;
  int order[ZR_MAX_W] = {};
  zr_scaler_cfg scaler{};
  int fp32_grads = 0;  // gradients are fp32 (4 bytes) instead of the param type
  // fused step: tile schedule, control block, kernel and grid
  int4* tiles_dev = nullptr;
  int64_t ntiles = 0;
  zr::Ctrl* ctrl_dev = nullptr;
  void* kernel = nullptr;  // the fused_step_kernel instantiation for (dtype, W, A)
  int grid = 0;
  int64_t resident = 0;    // blocks of that kernel that fit on the GPU at once
  // zr_step with its loads staged by bulk copies (zr_plan_set_staging): the kernel, its
  // stage size and count, dynamic shared memory per block and grid
  int staging = 0;         // ZR_STAGING_REGISTERS or ZR_STAGING_BULK
  void* bulk_kernel = nullptr;
  int bulk_E = 0, bulk_NS = 0, bulk_smem = 0, bulk_grid = 0, bulk_threads = 0;
  int64_t bulk_resident = 0;  // blocks of the bulk kernel that fit on the GPU at once
  int bulk_stall = 0;         // test hook (zr_plan_stall_bulk_waits): stages announce bytes never sent
  int device = 0;
  // bucketed launches (zr_step_bucket): bucket b's tiles are [tile_begin[b], tile_begin[b+1]),
  // launched with bucket_grid[b] blocks; a step's launches add up to bucket_blocks blocks
  std::vector<int64_t> tile_begin;
  std::vector<int> bucket_grid;
  unsigned bucket_blocks = 0;
  // in-place step (zr_step_inplace): the flag-pass and in-place instantiations for
  // (dtype, W, A) and their grids (one block per tile)
  void* ip_flag_kernel = nullptr;
  void* ip_update_kernel = nullptr;
  int ip_flag_grid = 0, ip_update_grid = 0;
  // ZeRO-3 parameter shards: the worker at ring position p keeps block (p+1) mod W of
  // every bucket, packed in bucket order. shard_off[b*W + w] is where bucket b's block
  // starts in worker w's shard; the shard tile table cuts every (bucket, block) piece
  // into copies of at most 16K elements (two int4 per tile: {flat lo, flat hi, shard lo,
  // shard hi}, {groups of 8, worker, 0, 0}); bucket b's tiles are
  // [shard_tile_begin[b], shard_tile_begin[b+1]).
  std::vector<int64_t> shard_numel;
  std::vector<int64_t> shard_off;
  std::vector<int64_t> shard_tile_begin;
  int4* shard_tiles_dev = nullptr;
  int64_t nshard_tiles = 0;
};

namespace zr {
// Builds the ZeRO-3 shard bookkeeping and its device tile table (zr_zero3.cu).
zr_status build_shard_tables(zr_plan* p);
// Picks the in-place step's kernels and grids once the tile table exists (zr_inplace.cu).
zr_status init_inplace(zr_plan* p);
// The automatic stage shape of bulk-copy staging for R = W*A replica slices (zr_step.cu):
// fills *E if it is 0 and *NS if it is 0.
void bulk_auto_shape(int R, int* E, int* NS);
// Whether the automatic shape suits a step of R replica slices over ntiles tiles when
// `resident` blocks of the bulk kernel fit on the GPU at once: stages of 2048 elements
// and at least four waves of tiles (the rule zr_plan_create and zr_step_noalloc apply).
bool bulk_preferred(int E, int64_t ntiles, int64_t resident);

// Blocks for a launch over `ntiles` tiles. A large launch gets one block per tile: the
// hardware hands blocks out in index order as earlier ones finish, so the tiles in flight
// stay a compact window of the address space and every block ends within one tile of the
// others (a persistent grid striding over the tiles measured 3-9 % slower on the 1.3B and
// 7B workloads). Under four waves of tiles a persistent grid of at most `resident` blocks
// striding over them avoids a last, partly filled wave.
inline int step_grid(const zr_plan* p, int64_t ntiles) {
  constexpr int64_t kMaxBlocks = 1 << 30;  // a step's launches stay below 2^32 blocks
  if (ntiles < 1) return 1;
  if (ntiles >= 4 * p->resident) return (int)(ntiles < kMaxBlocks ? ntiles : kMaxBlocks);
  return (int)(ntiles < p->resident ? ntiles : p->resident);
}
}  // namespace zr
