// Host-only parts of libzr: error reporting, the reverse-order bucket builder,
// ring traffic and model-state accounting. Built with -ffp-contract=off.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "zr_internal.h"

namespace zr {

static thread_local char g_err[512] = "";

zr_status fail(zr_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  std::vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  // a failed CUDA runtime call also leaves its code in the runtime's per-thread last
  // error, where the caller's next unrelated check would find it: it is reported here
  if (s == ZR_ERR_CUDA || s == ZR_ERR_OOM) take_cuda_error();
  return s;
}

void clear_error() { g_err[0] = '\0'; }

}  // namespace zr

using zr::fail;

extern "C" const char* zr_last_error(void) { return zr::g_err; }

extern "C" const char* zr_status_str(zr_status s) {
  switch (s) {
    case ZR_OK: return "ok";
    case ZR_ERR_INVALID: return "invalid argument";
    case ZR_ERR_UNSUPPORTED: return "unsupported";
    case ZR_ERR_CUDA: return "CUDA error";
    case ZR_ERR_OOM: return "out of memory";
    case ZR_ERR_TIMEOUT: return "timeout";
  }
  return "unknown status";
}

extern "C" const char* zr_version(void) { return "zr 0.1 sm_103a"; }

// Blocks are whole multiples of `align` elements, as equal as that allows; the last
// ones take the remainder (possibly none).
extern "C" int64_t zr_chunk_size(int64_t n, int W, int align) {
  if (n <= 0 || W < 1 || align < 1) return 0;
  const int64_t per = (n + W - 1) / W;                 // ceil(n / W)
  return (per + align - 1) / align * align;            // rounded up to align
}

// Tensors walk from the last defined to the first (output side first), each placed at
// the next multiple of `align`; the open bucket closes when the next tensor would take
// its element count past the cap.
extern "C" zr_status zr_bucket_plan(const int64_t* numels, int ntensors, int64_t cap_elems, int W, int align,
                                    zr_bucket* out, int* nbuckets, int64_t* tensor_offsets) {
  zr::clear_error();
  if (!out || !nbuckets) return fail(ZR_ERR_INVALID, "zr_bucket_plan: null output");
  if (ntensors < 0 || (ntensors > 0 && !numels)) return fail(ZR_ERR_INVALID, "zr_bucket_plan: bad tensor list");
  if (cap_elems < 1) return fail(ZR_ERR_INVALID, "zr_bucket_plan: cap must be >= 1");
  if (W < 1 || W > ZR_MAX_W) return fail(ZR_ERR_INVALID, "zr_bucket_plan: W=%d outside [1, %d]", W, ZR_MAX_W);
  if (align < 1) return fail(ZR_ERR_INVALID, "zr_bucket_plan: align must be >= 1");
  for (int t = 0; t < ntensors; ++t)
    if (numels[t] < 0) return fail(ZR_ERR_INVALID, "zr_bucket_plan: numel[%d] < 0", t);
  int nb = 0;
  int64_t next = 0, open_at = 0, open_len = 0;
  auto close = [&]() {
    out[nb].start = open_at;
    out[nb].len = open_len;
    out[nb].chunk = zr_chunk_size(open_len, W, align);
    ++nb;
  };
  for (int t = ntensors - 1; t >= 0; --t) {
    if (open_len > 0 && open_len + numels[t] > cap_elems) {
      close();
      open_at = next;
      open_len = 0;
    }
    const int64_t padded = (numels[t] + align - 1) / align * align;
    if (tensor_offsets) tensor_offsets[t] = next;
    next += padded;
    open_len += padded;
  }
  if (open_len > 0) close();
  *nbuckets = nb;
  return ZR_OK;
}

extern "C" int64_t zr_model_state_bytes(int stage, int64_t n, int W) {
  if (n < 0 || W < 1) return -1;
  // 2 B fp16 param + 2 B fp16 grad + 12 B fp32 master/m/v per parameter; ZeRO shards the
  // optimizer states (stage 1), then the gradients (2), then the parameters (3) over W.
  const int64_t param = 2 * n, grad = 2 * n, opt = 12 * n;
  switch (stage) {
    case 0: return param + grad + opt;
    case 1: return param + grad + opt / W;
    case 2: return param + (grad + opt) / W;
    case 3: return (param + grad + opt) / W;
    default: return -1;
  }
}

extern "C" zr_status zr_ring_traffic(int64_t n, int W, int align, int64_t* rs_sent, int64_t* rs_recv,
                                     int64_t* ag_sent, int64_t* ag_recv) {
  zr::clear_error();
  if (n < 0 || W < 1 || W > ZR_MAX_W || align < 1) return fail(ZR_ERR_INVALID, "zr_ring_traffic: bad n/W/align");
  const int64_t C = zr_chunk_size(n, W, align);
  auto block = [&](int c) -> int64_t {
    int64_t lo = (int64_t)c * C, hi = lo + C;
    if (lo > n) lo = n;
    if (hi > n) hi = n;
    return hi - lo;
  };
  for (int p = 0; p < W; ++p) {
    // with one worker nothing moves
    const int64_t all = W > 1 ? n : 0;
    if (rs_sent) rs_sent[p] = W > 1 ? all - block((p + 1) % W) : 0;
    if (rs_recv) rs_recv[p] = W > 1 ? all - block(p) : 0;
    if (ag_sent) ag_sent[p] = W > 1 ? all - block((p + 2) % W) : 0;
    if (ag_recv) ag_recv[p] = W > 1 ? all - block((p + 1) % W) : 0;
  }
  return ZR_OK;
}
