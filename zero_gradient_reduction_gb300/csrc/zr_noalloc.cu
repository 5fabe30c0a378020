// zr_step_noalloc: the fused step for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: an embedding runtime that owns every byte of
// device memory through its own pool and forbids allocations behind its back, code
// running under a hard memory budget that was sized before the first step, or a
// caller on a path where an allocation would implicitly synchronise the device.
// zr_plan_create allocates a tile table and a control block, so such callers cannot
// use zr_step. This entry point runs zr_step's kernel with its scratch (the tile
// schedule and a control block) kept in one static device array of this file, sized
// at compile time. The caller passes every input
// and output, and carries the step state (live set, loss scale, step count) itself.
//
// Sharing and lifetime: the array exists once per GPU that loads this library and
// stays allocated until the process exits. Every call on a device uses the same
// array and leaves its contents behind; each call rebuilds the schedule and clears
// the ticket and the flag itself before the step kernel runs. Calls whose kernels
// overlap on the GPU (different streams without ordering between them) race on the
// array and must not be issued. The first call on a device resolves the array's
// device address with cudaGetSymbolAddress; make that first call before any stream
// capture begins.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "zr_device.cuh"
#include "zr_internal.h"
#include "zr_nvtx.h"

using zr::fail;

#include "zr_plan.h"
#include "zr_step_kernel.cuh"
#include "zr_step_bulk.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kSetupBuckets = 64;  // bucket descriptors carried by one set-up launch

// Scratch layout: [0, 256) a control block for fused_step_kernel; then ZR_NOALLOC_MAX_TILES
// tiles of 16 bytes. The step runs the same kernel as zr_step, with this control block
// standing in for a plan's: the set-up launch writes the caller's live set, loss scale and
// the running beta products for t - 1 into it, and clears its flag and ticket.
constexpr size_t kHeaderBytes = 256;
static_assert(sizeof(zr::Ctrl) <= kHeaderBytes, "the control block must fit the scratch header");
constexpr size_t kScratchBytes = kHeaderBytes + (size_t)ZR_NOALLOC_MAX_TILES * sizeof(int4);

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch, resolved once per device (host code may not use the
// symbol itself as a device address).
std::mutex g_addr_mu;
void* g_addr[kMaxDevices] = {};

zr_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(ZR_ERR_UNSUPPORTED, "zr_step_noalloc: device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_addr_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return fail(ZR_ERR_CUDA, "zr_step_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return ZR_OK;
}

struct SetupArgs {
  int64_t start[kSetupBuckets];
  int64_t len[kSetupBuckets];
  int64_t chunk[kSetupBuckets];
  int32_t first_tile[kSetupBuckets];  // index of each bucket's first tile in the table
  int nb;
  int W;
  int64_t tile;        // elements per tile
  int init_ctrl;       // the first set-up launch of a call writes the control block
  int current;         // live state set
  float scale;         // loss scale of this step
  double prod1, prod2; // beta1^(t-1), beta2^(t-1) as running products
  unsigned char* scratch;
};

// One block per bucket: writes the bucket's tiles (block by block, pieces of at most
// `tile` elements) into the table, in the same order zr_plan_create uses. The first
// launch of a call also writes the control block the step kernel reads.
__global__ void setup_tiles_kernel(const __grid_constant__ SetupArgs a) {
  if (a.init_ctrl && blockIdx.x == 0 && threadIdx.x == 0) {
    zr::Ctrl* c = reinterpret_cast<zr::Ctrl*>(a.scratch);
    uint32_t* words = reinterpret_cast<uint32_t*>(a.scratch);
    for (size_t i = 0; i < sizeof(zr::Ctrl) / 4; ++i) words[i] = 0;
    c->k = a.current;
    c->scale = a.scale;
    c->scale_used = a.scale;
    c->prod1 = a.prod1;
    c->prod2 = a.prod2;
    c->interval = 1;
  }
  const int b = blockIdx.x;
  if (b >= a.nb) return;
  int4* table = reinterpret_cast<int4*>(a.scratch + kHeaderBytes);
  const int64_t end = a.start[b] + a.len[b];
  int32_t tile = a.first_tile[b];
  for (int c = 0; c < a.W; ++c) {
    int64_t lo = a.start[b] + (int64_t)c * a.chunk[b], hi = lo + a.chunk[b];
    if (lo > end) lo = end;
    if (hi > end) hi = end;
    const int64_t pieces = (hi - lo + a.tile - 1) / a.tile;
    for (int64_t i = threadIdx.x; i < pieces; i += blockDim.x) {
      const int64_t x = lo + i * a.tile;
      const int64_t ln = (hi - x) < a.tile ? (hi - x) : a.tile;
      table[tile + i] = make_int4((int)(uint32_t)(uint64_t)x, (int)(uint32_t)((uint64_t)x >> 32), (int)(ln / 8), c);
    }
    tile += (int32_t)pieces;
  }
}

// beta1^(t-1) and beta2^(t-1) as the running products a plan keeps, so that the bias
// corrections match zr_step's bit for bit. The last result is kept per process: a caller
// stepping t = 1, 2, 3, ... extends it by one factor per call instead of redoing t - 1
// multiplications; going back in t, or other betas, starts again from 1.0 (bounded by
// the fixed point of zr::beta_power_from).
struct PowCache {
  float beta1 = 0.0f, beta2 = 0.0f;
  int64_t n = -1;  // exponent of the cached products (-1: empty)
  double p1 = 1.0, p2 = 1.0;
};
std::mutex g_pow_mu;
PowCache g_pow;

void beta_powers(float beta1, float beta2, int64_t n, double* p1, double* p2) {
  std::lock_guard<std::mutex> lock(g_pow_mu);
  PowCache& c = g_pow;
  const bool same = c.n >= 0 && std::memcmp(&c.beta1, &beta1, sizeof(float)) == 0 &&
                    std::memcmp(&c.beta2, &beta2, sizeof(float)) == 0;
  if (!same || c.n > n) {
    c.beta1 = beta1;
    c.beta2 = beta2;
    c.n = 0;
    c.p1 = 1.0;
    c.p2 = 1.0;
  }
  c.p1 = zr::beta_power_from(c.p1, c.n, beta1, n);
  c.p2 = zr::beta_power_from(c.p2, c.n, beta2, n);
  c.n = n;
  *p1 = c.p1;
  *p2 = c.p2;
}

// Tiles the ring blocks of the buckets need at `tile` elements per tile.
int64_t count_tiles(const zr_bucket* buckets, int nbuckets, int W, int64_t tile) {
  int64_t n = 0;
  for (int b = 0; b < nbuckets; ++b)
    for (int c = 0; c < W; ++c) {
      int64_t lo = (int64_t)c * buckets[b].chunk, hi = lo + buckets[b].chunk;
      if (lo > buckets[b].len) lo = buckets[b].len;
      if (hi > buckets[b].len) hi = buckets[b].len;
      n += (hi - lo + tile - 1) / tile;
    }
  return n;
}

}  // namespace

extern "C" zr_status zr_step_noalloc(const zr_bucket* buckets, int nbuckets, int W, int A, zr_dtype dtype,
                                     const int* order, const void* const* grads, const zr_state* st, int current,
                                     const zr_adamw_hyper* h, float loss_scale, int64_t t, int32_t* overflow,
                                     void* stream) {
  zr::Range range("zr_step_noalloc");
  zr::clear_error();
  if (W < 1 || W > ZR_MAX_W) return fail(ZR_ERR_INVALID, "zr_step_noalloc: W=%d outside [1, %d]", W, ZR_MAX_W);
  if (A < 1 || (int64_t)W * A > ZR_MAX_REPLICAS)
    return fail(ZR_ERR_INVALID, "zr_step_noalloc: A=%d (W*A must be in [1, %d])", A, ZR_MAX_REPLICAS);
  if (dtype != ZR_F16 && dtype != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_step_noalloc: dtype must be F16 or BF16");
  if (nbuckets < 0 || (nbuckets > 0 && !buckets)) return fail(ZR_ERR_INVALID, "zr_step_noalloc: bad bucket table");
  if (!grads || !st || !h || !overflow) return fail(ZR_ERR_INVALID, "zr_step_noalloc: null argument");
  if (current != 0 && current != 1) return fail(ZR_ERR_INVALID, "zr_step_noalloc: current must be 0 or 1");
  if (t < 1) return fail(ZR_ERR_INVALID, "zr_step_noalloc: t must be >= 1");
  if (!zr::betas_ok(*h)) return fail(ZR_ERR_INVALID, "zr_step_noalloc: betas must lie in [0, 1)");
  if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
    return fail(ZR_ERR_INVALID, "zr_step_noalloc: loss_scale must be positive and finite");
  if (reinterpret_cast<uintptr_t>(overflow) & 3u) return fail(ZR_ERR_INVALID, "zr_step_noalloc: misaligned overflow");
  bool seen[ZR_MAX_W] = {};
  int ord[ZR_MAX_W];
  for (int p = 0; p < W; ++p) {
    const int w = order ? order[p] : p;
    if (w < 0 || w >= W || seen[w]) return fail(ZR_ERR_INVALID, "zr_step_noalloc: order is not a permutation");
    seen[w] = true;
    ord[p] = w;
  }
  // every bucket must follow the ring rule
  bool any = false;  // some bucket has elements (else the arrays are empty and may be null)
  for (int b = 0; b < nbuckets; ++b) {
    any = any || buckets[b].len > 0;
    const zr_bucket& bk = buckets[b];
    if (bk.start < 0 || bk.len < 0 || (bk.start % ZR_ALIGN) || (bk.len % ZR_ALIGN) ||
        bk.chunk != zr_chunk_size(bk.len, W, ZR_ALIGN))
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: bucket %d is not a ring bucket (start/len multiples of %d, "
                  "chunk = zr_chunk_size(len, W, %d))", b, ZR_ALIGN, ZR_ALIGN);
  }
  for (int r = 0; r < W * A && any; ++r)
    if (!grads[r] || !zr::aligned16(grads[r]))
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: grads[%d] null or misaligned", r);
  for (int k = 0; k < 2 && any; ++k)
    if (!st->master[k] || !st->m[k] || !st->v[k] || !st->param[k] || !zr::aligned16(st->master[k]) ||
        !zr::aligned16(st->m[k]) || !zr::aligned16(st->v[k]) || !zr::aligned16(st->param[k]))
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: state set %d null or misaligned", k);
  if (any && (st->master[0] == st->master[1] || st->m[0] == st->m[1] || st->v[0] == st->v[1] ||
              st->param[0] == st->param[1]))
    return fail(ZR_ERR_INVALID, "zr_step_noalloc: the two state sets must be distinct buffers");
  // the step kernel for (dtype, W, A) and the blocks of it that fit on the GPU at once
  KernelFn kern = dtype == ZR_F16 ? pick_kernel<zr::DT_F16, kPingPong>(W, A, false)
                                  : pick_kernel<zr::DT_BF16, kPingPong>(W, A, false);
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0);
  if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step_noalloc: %s", cudaGetErrorString(e));
  const int64_t full = (int64_t)(sms > 0 ? sms : 1) * (per_sm > 0 ? per_sm : 1);
  // tiles of kTileElems, halved (down to 2048) until every block that fits gets two
  int64_t tile = kTileElems, ntiles = count_tiles(buckets, nbuckets, W, tile);
  while (tile > 2048 && ntiles < 2 * full) {
    tile /= 2;
    ntiles = count_tiles(buckets, nbuckets, W, tile);
  }
  if (ntiles > ZR_NOALLOC_MAX_TILES)
    return fail(ZR_ERR_INVALID, "zr_step_noalloc: the buckets need more than %d tiles of %lld elements "
                "(the static scratch limit); use zr_plan_create/zr_step", ZR_NOALLOC_MAX_TILES, (long long)tile);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (ntiles == 0) {
    // nothing to reduce: the step is clean, and the flag says so
    e = cudaMemsetAsync(overflow, 0, sizeof(int32_t), cs);
    return e == cudaSuccess ? ZR_OK : fail(ZR_ERR_CUDA, "zr_step_noalloc: %s", cudaGetErrorString(e));
  }

  void* scratch = nullptr;
  zr_status s = scratch_address(&scratch);
  if (s != ZR_OK) return s;

  // the tile schedule and the control block: one set-up launch per group of kSetupBuckets buckets
  double prod1 = 1.0, prod2 = 1.0;  // beta^(t-1): the step kernel takes the t-th factor itself
  beta_powers(h->beta1, h->beta2, t - 1, &prod1, &prod2);
  int32_t first = 0;
  for (int b0 = 0; b0 < nbuckets; b0 += kSetupBuckets) {
    SetupArgs sa;
    std::memset(&sa, 0, sizeof sa);
    sa.nb = nbuckets - b0 < kSetupBuckets ? nbuckets - b0 : kSetupBuckets;
    sa.W = W;
    sa.tile = tile;
    sa.init_ctrl = b0 == 0;
    sa.current = current;
    sa.scale = loss_scale;
    sa.prod1 = prod1;
    sa.prod2 = prod2;
    sa.scratch = static_cast<unsigned char*>(scratch);
    for (int i = 0; i < sa.nb; ++i) {
      const zr_bucket& bk = buckets[b0 + i];
      sa.start[i] = bk.start;
      sa.len[i] = bk.len;
      sa.chunk[i] = bk.chunk;
      sa.first_tile[i] = first;
      first += (int32_t)count_tiles(&bk, 1, W, tile);
    }
    setup_tiles_kernel<<<sa.nb, 128, 0, cs>>>(sa);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step_noalloc: set-up launch failed: %s", cudaGetErrorString(e));
  }

  // the step: the kernel zr_step launches, over the scratch's tiles and control block
  FusedArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < W * A; ++r) a.grads[r] = grads[r];
  for (int p = 0; p < W; ++p) a.order[p] = ord[p];
  zr::Ctrl* ctrl = static_cast<zr::Ctrl*>(scratch);
  a.tiles = reinterpret_cast<const int4*>(static_cast<unsigned char*>(scratch) + kHeaderBytes);
  a.tile0 = 0;
  a.tile1 = ntiles;
  // The kernel zr_step would use: bulk-copy staging where zr::bulk_preferred says so (it
  // allocates nothing: its shared memory is an attribute of the kernel, set on this device
  // here), else register staging.
  BulkKernelFn bulk = nullptr;
  BulkCfg cfg{0, 0, 0u};
  int bulk_smem = 0;
  {
    int E = 0, NS = 0;
    zr::bulk_auto_shape(W * A, &E, &NS);
    const int smem = NS * bulk_stage_bytes(W * A, E);
    BulkKernelFn k = dtype == ZR_F16 ? pick_bulk_kernel<zr::DT_F16, false>(W, A)
                                     : pick_bulk_kernel<zr::DT_BF16, false>(W, A);
    int bps = 0;
    cudaError_t eb = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (eb == cudaSuccess) eb = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, k, bulk_threads(false), smem);
    if (eb != cudaSuccess) (void)cudaGetLastError();  // not fatal: register staging then
    else if (bps > 0 && zr::bulk_preferred(E, ntiles, (int64_t)sms * bps)) {
      bulk = k;
      cfg.E = E;
      cfg.NS = NS;
      bulk_smem = smem;
    }
  }
  const int grid = (int)(ntiles >= 4 * full ? ntiles : (ntiles < full ? ntiles : full));
  a.total_blocks = (unsigned)(bulk ? ntiles : grid);
  for (int k = 0; k < 2; ++k) {
    a.master[k] = st->master[k];
    a.m[k] = st->m[k];
    a.v[k] = st->v[k];
    a.param[k] = static_cast<uint16_t*>(st->param[k]);
  }
  a.ctrl = ctrl;
  a.lr = h->lr;
  a.beta1 = h->beta1;
  a.beta2 = h->beta2;
  a.eps = h->eps;
  a.weight_decay = h->weight_decay;
  a.W = W;
  a.A = A;
  a.stage = 1;
  if (bulk) bulk<<<(int)ntiles, bulk_threads(false), bulk_smem, cs>>>(a, cfg);
  else kern<<<grid, kThreads, 0, cs>>>(a);
  e = cudaGetLastError();
  // the step's flag, which its last block leaves in the control block, to the caller
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(overflow, &ctrl->last_overflow, sizeof(int32_t), cudaMemcpyDeviceToDevice, cs);
  return e == cudaSuccess ? ZR_OK : fail(ZR_ERR_CUDA, "zr_step_noalloc: launch failed: %s", cudaGetErrorString(e));
}
