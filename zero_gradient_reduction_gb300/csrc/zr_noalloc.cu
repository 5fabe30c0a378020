// zr_step_noalloc: the fused step for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: an embedding runtime that owns every byte of
// device memory through its own pool and forbids allocations behind its back, code
// running under a hard memory budget that was sized before the first step, or a
// caller on a path where an allocation would implicitly synchronise the device.
// zr_plan_create allocates a tile table and a control block, so such callers cannot
// use zr_step. This entry point runs the same fused arithmetic with its scratch (the
// tile schedule, the block ticket and the overflow accumulator) kept in one static
// device array of this file, sized at compile time. The caller passes every input
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

using zr::fail;

namespace zr {
float bias_correction_host(float beta, int64_t t);
}

namespace {

constexpr int kThreads = 256;
constexpr int kTileElems = 8192;
constexpr int kMaxDevices = 64;
constexpr int kSetupBuckets = 64;  // bucket descriptors carried by one set-up launch

// Scratch layout: [0, 256) header {ticket, flag}; then ZR_NOALLOC_MAX_TILES tiles of 16 bytes.
struct ScratchHeader {
  uint32_t ticket;
  int32_t flag;
};
constexpr size_t kHeaderBytes = 256;
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
  int clear_header;  // the first set-up launch of a call zeroes the ticket and the flag
  unsigned char* scratch;
};

// One block per bucket: writes the bucket's tiles (block by block, pieces of at most
// kTileElems) into the table, in the same order zr_plan_create uses.
__global__ void setup_tiles_kernel(const __grid_constant__ SetupArgs a) {
  if (a.clear_header && blockIdx.x == 0 && threadIdx.x == 0) {
    ScratchHeader* hdr = reinterpret_cast<ScratchHeader*>(a.scratch);
    hdr->ticket = 0;
    hdr->flag = 0;
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
    const int64_t pieces = (hi - lo + kTileElems - 1) / kTileElems;
    for (int64_t i = threadIdx.x; i < pieces; i += blockDim.x) {
      const int64_t x = lo + i * kTileElems;
      const int64_t ln = (hi - x) < kTileElems ? (hi - x) : kTileElems;
      table[tile + i] = make_int4((int)(uint32_t)(uint64_t)x, (int)(uint32_t)((uint64_t)x >> 32), (int)(ln / 8), c);
    }
    tile += (int32_t)pieces;
  }
}

struct StaticArgs {
  const uint16_t* grads[ZR_MAX_REPLICAS];
  int order[ZR_MAX_W];
  const float* master_in;
  const float* m_in;
  const float* v_in;
  float* master_out;
  float* m_out;
  float* v_out;
  uint16_t* param_out;
  unsigned char* scratch;
  int32_t* overflow;
  int64_t ntiles;
  float r;
  zr::AdamConsts k;
  int W, A;
};

template <int DT>
__global__ void __launch_bounds__(kThreads) fused_step_noalloc_kernel(const __grid_constant__ StaticArgs a) {
  __shared__ const uint16_t* s_ptr[ZR_MAX_REPLICAS];
  __shared__ int s_bad;
  __shared__ unsigned s_ticket;
  ScratchHeader* hdr = reinterpret_cast<ScratchHeader*>(a.scratch);
  const int4* table = reinterpret_cast<const int4*>(a.scratch + kHeaderBytes);
  if (threadIdx.x == 0) s_bad = 0;
  const int W = a.W, A = a.A;
  bool bad = false;
  for (int64_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    const int4 d = table[tile];
    const int64_t start = (int64_t)(((uint64_t)(uint32_t)d.y << 32) | (uint32_t)d.x);
    const int groups = d.z, c = d.w;
    __syncthreads();
    for (int i = threadIdx.x; i < W * A; i += blockDim.x) {
      const int h = i / A, q = i - h * A;
      int pos = c + h;
      pos -= pos >= W ? W : 0;
      s_ptr[i] = a.grads[a.order[pos] * A + q] + start;
    }
    __syncthreads();
    for (int g = threadIdx.x; g < groups; g += blockDim.x) {
      const int64_t off = (int64_t)g * 8;
      float s[8];
      for (int h = 0; h < W; ++h) {
        float wsum[8];
        zr::unpack8<DT>(zr::ld_once(s_ptr[h * A] + off), wsum);
        for (int q = 1; q < A; ++q) {
          float x[8];
          zr::unpack8<DT>(zr::ld_once(s_ptr[h * A + q] + off), x);
#pragma unroll
          for (int j = 0; j < 8; ++j) wsum[j] = __fadd_rn(wsum[j], x[j]);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j] = h == 0 ? wsum[j] : __fadd_rn(s[j], wsum[j]);
      }
      const int64_t e = start + off;
      const float4 p0 = zr::ld_once_f4(a.master_in + e), p1 = zr::ld_once_f4(a.master_in + e + 4);
      const float4 m0 = zr::ld_once_f4(a.m_in + e), m1 = zr::ld_once_f4(a.m_in + e + 4);
      const float4 v0 = zr::ld_once_f4(a.v_in + e), v1 = zr::ld_once_f4(a.v_in + e + 4);
      float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        bad |= zr::nonfinite(s[j]);
        zr::adamw_elem(__fmul_rn(s[j], a.r), p[j], m[j], v[j], a.k);
      }
      zr::st_once_f4(a.master_out + e, make_float4(p[0], p[1], p[2], p[3]));
      zr::st_once_f4(a.master_out + e + 4, make_float4(p[4], p[5], p[6], p[7]));
      zr::st_once_f4(a.m_out + e, make_float4(m[0], m[1], m[2], m[3]));
      zr::st_once_f4(a.m_out + e + 4, make_float4(m[4], m[5], m[6], m[7]));
      zr::st_once_f4(a.v_out + e, make_float4(v[0], v[1], v[2], v[3]));
      zr::st_once_f4(a.v_out + e + 4, make_float4(v[4], v[5], v[6], v[7]));
      zr::st_once(a.param_out + e, zr::pack8<DT>(p));
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) s_bad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s_bad) atomicOr(&hdr->flag, 1);
    __threadfence();
    s_ticket = atomicAdd(&hdr->ticket, 1u);
  }
  __syncthreads();
  if (s_ticket == gridDim.x - 1 && threadIdx.x == 0) {
    __threadfence();
    volatile ScratchHeader* vh = hdr;
    *a.overflow = vh->flag;
    vh->flag = 0;
    vh->ticket = 0;
    __threadfence();
  }
}

}  // namespace

extern "C" zr_status zr_step_noalloc(const zr_bucket* buckets, int nbuckets, int W, int A, zr_dtype dtype,
                                     const int* order, const void* const* grads, const zr_state* st, int current,
                                     const zr_adamw_hyper* h, float loss_scale, int64_t t, int32_t* overflow,
                                     void* stream) {
  zr::clear_error();
  if (W < 1 || W > ZR_MAX_W) return fail(ZR_ERR_INVALID, "zr_step_noalloc: W=%d outside [1, %d]", W, ZR_MAX_W);
  if (A < 1 || (int64_t)W * A > ZR_MAX_REPLICAS)
    return fail(ZR_ERR_INVALID, "zr_step_noalloc: A=%d (W*A must be in [1, %d])", A, ZR_MAX_REPLICAS);
  if (dtype != ZR_F16 && dtype != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_step_noalloc: dtype must be F16 or BF16");
  if (nbuckets < 0 || (nbuckets > 0 && !buckets)) return fail(ZR_ERR_INVALID, "zr_step_noalloc: bad bucket table");
  if (!grads || !st || !h || !overflow) return fail(ZR_ERR_INVALID, "zr_step_noalloc: null argument");
  if (current != 0 && current != 1) return fail(ZR_ERR_INVALID, "zr_step_noalloc: current must be 0 or 1");
  if (t < 1) return fail(ZR_ERR_INVALID, "zr_step_noalloc: t must be >= 1");
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
  for (int r = 0; r < W * A; ++r)
    if (!grads[r] || !zr::aligned16(grads[r]))
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: grads[%d] null or misaligned", r);
  for (int k = 0; k < 2; ++k)
    if (!st->master[k] || !st->m[k] || !st->v[k] || !st->param[k] || !zr::aligned16(st->master[k]) ||
        !zr::aligned16(st->m[k]) || !zr::aligned16(st->v[k]) || !zr::aligned16(st->param[k]))
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: state set %d null or misaligned", k);
  if (st->master[0] == st->master[1] || st->m[0] == st->m[1] || st->v[0] == st->v[1] || st->param[0] == st->param[1])
    return fail(ZR_ERR_INVALID, "zr_step_noalloc: the two state sets must be distinct buffers");
  // every bucket must follow the ring rule; count its tiles
  int64_t ntiles = 0;
  for (int b = 0; b < nbuckets; ++b) {
    const zr_bucket& bk = buckets[b];
    if (bk.start < 0 || bk.len < 0 || (bk.start % ZR_ALIGN) || (bk.len % ZR_ALIGN) ||
        bk.chunk != zr_chunk_size(bk.len, W, ZR_ALIGN))
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: bucket %d is not a ring bucket (start/len multiples of %d, "
                  "chunk = zr_chunk_size(len, W, %d))", b, ZR_ALIGN, ZR_ALIGN);
    for (int c = 0; c < W; ++c) {
      int64_t lo = (int64_t)c * bk.chunk, hi = lo + bk.chunk;
      if (lo > bk.len) lo = bk.len;
      if (hi > bk.len) hi = bk.len;
      ntiles += (hi - lo + kTileElems - 1) / kTileElems;
    }
    if (ntiles > ZR_NOALLOC_MAX_TILES)
      return fail(ZR_ERR_INVALID, "zr_step_noalloc: the buckets need more than %d tiles of %d elements "
                  "(the static scratch limit); use zr_plan_create/zr_step", ZR_NOALLOC_MAX_TILES, kTileElems);
  }
  if (ntiles == 0) return ZR_OK;

  void* scratch = nullptr;
  zr_status s = scratch_address(&scratch);
  if (s != ZR_OK) return s;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);

  // schedule: one set-up launch per group of kSetupBuckets buckets
  int32_t tile = 0;
  for (int b0 = 0; b0 < nbuckets; b0 += kSetupBuckets) {
    SetupArgs sa;
    std::memset(&sa, 0, sizeof sa);
    sa.nb = nbuckets - b0 < kSetupBuckets ? nbuckets - b0 : kSetupBuckets;
    sa.W = W;
    sa.clear_header = b0 == 0;
    sa.scratch = static_cast<unsigned char*>(scratch);
    for (int i = 0; i < sa.nb; ++i) {
      const zr_bucket& bk = buckets[b0 + i];
      sa.start[i] = bk.start;
      sa.len[i] = bk.len;
      sa.chunk[i] = bk.chunk;
      sa.first_tile[i] = tile;
      for (int c = 0; c < W; ++c) {
        int64_t lo = (int64_t)c * bk.chunk, hi = lo + bk.chunk;
        if (lo > bk.len) lo = bk.len;
        if (hi > bk.len) hi = bk.len;
        tile += (int32_t)((hi - lo + kTileElems - 1) / kTileElems);
      }
    }
    setup_tiles_kernel<<<sa.nb, 128, 0, cs>>>(sa);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step_noalloc: set-up launch failed: %s", cudaGetErrorString(e));
  }

  StaticArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < W * A; ++r) a.grads[r] = static_cast<const uint16_t*>(grads[r]);
  for (int p = 0; p < W; ++p) a.order[p] = ord[p];
  a.master_in = st->master[current];
  a.m_in = st->m[current];
  a.v_in = st->v[current];
  a.master_out = st->master[1 - current];
  a.m_out = st->m[1 - current];
  a.v_out = st->v[1 - current];
  a.param_out = static_cast<uint16_t*>(st->param[1 - current]);
  a.scratch = static_cast<unsigned char*>(scratch);
  a.overflow = overflow;
  a.ntiles = ntiles;
  a.r = (float)(1.0 / ((double)loss_scale * (double)W));
  a.k.b1 = h->beta1;
  a.k.b2 = h->beta2;
  a.k.omb1 = 1.0f - h->beta1;
  a.k.omb2 = 1.0f - h->beta2;
  a.k.lr = h->lr;
  a.k.eps = h->eps;
  const float lrwd = h->lr * h->weight_decay;
  a.k.decay = 1.0f - lrwd;
  a.k.bc1 = zr::bias_correction_host(h->beta1, t);
  a.k.bc2 = zr::bias_correction_host(h->beta2, t);
  a.W = W;
  a.A = A;

  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto kern = dtype == ZR_F16 ? fused_step_noalloc_kernel<zr::DT_F16> : fused_step_noalloc_kernel<zr::DT_BF16>;
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0);
  if (e != cudaSuccess) return fail(ZR_ERR_CUDA, "zr_step_noalloc: %s", cudaGetErrorString(e));
  if (per_sm < 1) per_sm = 1;
  const int64_t full = (int64_t)sms * per_sm;
  const int grid = (int)(ntiles < full ? ntiles : full);
  kern<<<grid, kThreads, 0, cs>>>(a);
  e = cudaGetLastError();
  return e == cudaSuccess ? ZR_OK : fail(ZR_ERR_CUDA, "zr_step_noalloc: launch failed: %s", cudaGetErrorString(e));
}
