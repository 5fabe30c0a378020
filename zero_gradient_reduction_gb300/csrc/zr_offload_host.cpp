// ZeRO-Offload's optimizer half on the host CPU: the owner-side AdamW update of fp32
// master/m/v kept in host memory and the 16-bit cast of the result, run by a team of
// threads over contiguous slices. Same arithmetic and op order as the GPU kernels
// (each fp32 operation rounded once; built with -ffp-contract=off), so the result is
// bit-identical to zr_adamw_shard_step + zr_all_gather.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "zr_internal.h"

using zr::fail;

namespace {

uint32_t f32_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return u;
}

// Round-to-nearest-even fp32 -> bfloat16 / binary16 bit patterns, written without branches
// so that the loops vectorise; a NaN becomes the canonical quiet NaN of its sign.
inline uint16_t to_bf16(float f) {
  const uint32_t x = f32_bits(f);
  const uint16_t nan = (uint16_t)(((x >> 16) & 0x8000u) | 0x7FC0u);
  const uint16_t r = (uint16_t)((x + 0x7FFFu + ((x >> 16) & 1u)) >> 16);
  return (x & 0x7FFFFFFFu) > 0x7F800000u ? nan : r;
}

// binary16 through the compiler's _Float16 conversion (one IEEE round-to-nearest-even: a
// hardware conversion on Arm, exact software rounding elsewhere); NaNs made canonical.
inline uint16_t to_f16(float f) {
  const _Float16 h = (_Float16)f;
  uint16_t u;
  std::memcpy(&u, &h, 2);
  const uint32_t x = f32_bits(f);
  const uint16_t nan = (uint16_t)(((x >> 16) & 0x8000u) | 0x7E00u);
  return (x & 0x7FFFFFFFu) > 0x7F800000u ? nan : u;
}

using Consts = zr::OffloadConsts;

// AdamW over elements [lo, hi), with the bf16 cast (CAST = 1) taking each new master value
// as it is computed: every operation is branch-free, so the loop vectorises and host memory
// is passed over once. The fp16 cast inside the same loop is slower on the Grace cores (86
// against 70 ms for 4e8 params), so fp16 casts in a pass of its own over each chunk.
template <int CAST>
void update_range(const float* __restrict__ sums, float* __restrict__ p, float* __restrict__ m,
                  float* __restrict__ v, uint16_t* __restrict__ out, int64_t lo, int64_t hi, const Consts& k) {
  for (int64_t i = lo; i < hi; ++i) {
    const float g = sums[i] * k.r;
    const float mi = k.b1 * m[i] + k.omb1 * g;
    const float vi = k.b2 * v[i] + k.omb2 * (g * g);
    const float mhat = mi / k.bc1;
    const float vhat = vi / k.bc2;
    const float den = std::sqrt(vhat) + k.eps;
    const float u = mhat / den;
    const float pi = p[i] * k.decay - k.lr * u;
    m[i] = mi;
    v[i] = vi;
    p[i] = pi;
    if constexpr (CAST == 1) out[i] = to_bf16(pi);
  }
}

void update_slice(const float* sums, float* p, float* m, float* v, uint16_t* out, int64_t lo, int64_t hi,
                  const Consts& k, bool bf16) {
  if (!out) {
    update_range<0>(sums, p, m, v, out, lo, hi, k);
  } else if (bf16) {
    update_range<1>(sums, p, m, v, out, lo, hi, k);
  } else {
    // chunks small enough that the cast reads the chunk's new master values from cache
    constexpr int64_t kChunk = 4096;
    for (int64_t c = lo; c < hi; c += kChunk) {
      const int64_t e = c + kChunk < hi ? c + kChunk : hi;
      update_range<0>(sums, p, m, v, out, c, e, k);
      for (int64_t i = c; i < e; ++i) out[i] = to_f16(p[i]);
    }
  }
}

// Any +-inf or NaN in x[lo, hi): an all-ones exponent. The test is OR-ed into a 32-bit word, which the
// compiler vectorises (a bool accumulator it does not: 12.6 against 7.9 ms for 4e8 values on 16 Grace cores).
bool any_nonfinite(const float* x, int64_t lo, int64_t hi) {
  uint32_t acc = 0;
  for (int64_t i = lo; i < hi; ++i) acc |= (uint32_t)((f32_bits(x[i]) & 0x7F800000u) == 0x7F800000u);
  return acc != 0;
}

template <typename F>
void parallel_for(int64_t n, int nthreads, F fn) {
  if (nthreads <= 1 || n < (1 << 16)) {
    fn(0, n, 0);
    return;
  }
  std::vector<std::thread> team;
  const int64_t per = (n + nthreads - 1) / nthreads;
  for (int t = 0; t < nthreads; ++t) {
    const int64_t lo = t * per, hi = lo + per < n ? lo + per : n;
    if (lo >= hi) break;
    team.emplace_back(fn, lo, hi, t);
  }
  for (auto& th : team) th.join();
}

}  // namespace

namespace zr {

OffloadConsts offload_consts(const zr_adamw_hyper& h, float loss_scale, int W, int64_t t) {
  OffloadConsts k;
  k.b1 = h.beta1;
  k.b2 = h.beta2;
  k.omb1 = 1.0f - h.beta1;
  k.omb2 = 1.0f - h.beta2;
  k.lr = h.lr;
  k.eps = h.eps;
  const float lrwd = h.lr * h.weight_decay;
  k.decay = 1.0f - lrwd;
  k.bc1 = bias_correction_host(h.beta1, t);
  k.bc2 = bias_correction_host(h.beta2, t);
  k.r = (float)(1.0 / ((double)loss_scale * (double)W));
  return k;
}

void offload_update(const float* sums, float* master, float* m, float* v, void* param16, zr_dtype dt, int64_t lo,
                    int64_t hi, const OffloadConsts& k) {
  update_slice(sums, master, m, v, static_cast<uint16_t*>(param16), lo, hi, k, dt == ZR_BF16);
}
}  // namespace zr

extern "C" zr_status zr_offload_adamw(const float* sums, float* master, float* m, float* v, void* param16,
                                      zr_dtype dt, int64_t n, const zr_adamw_hyper* h, float loss_scale, int W,
                                      int64_t t, int nthreads, int32_t* overflow) {
  zr::clear_error();
  if (n < 0 || W < 1 || t < 1 || !h || !overflow) return fail(ZR_ERR_INVALID, "zr_offload_adamw: bad n/W/t or null");
  if (!zr::betas_ok(*h)) return fail(ZR_ERR_INVALID, "zr_offload_adamw: betas must lie in [0, 1)");
  if (dt != ZR_F16 && dt != ZR_BF16) return fail(ZR_ERR_INVALID, "zr_offload_adamw: dtype must be F16 or BF16");
  if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
    return fail(ZR_ERR_INVALID, "zr_offload_adamw: loss_scale must be positive and finite");
  if (n > 0 && (!sums || !master || !m || !v)) return fail(ZR_ERR_INVALID, "zr_offload_adamw: null array");
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  std::vector<char> bad(nthreads, 0);
  parallel_for(n, nthreads, [&](int64_t lo, int64_t hi, int tid) { bad[tid] = any_nonfinite(sums, lo, hi); });
  for (char b : bad)
    if (b) {
      *overflow = 1;
      return ZR_OK;  // skipped: nothing written
    }
  *overflow = 0;
  const Consts k = zr::offload_consts(*h, loss_scale, W, t);
  uint16_t* out = static_cast<uint16_t*>(param16);
  const bool bf16 = dt == ZR_BF16;
  parallel_for(n, nthreads, [&](int64_t lo, int64_t hi, int) { update_slice(sums, master, m, v, out, lo, hi, k, bf16); });
  return ZR_OK;
}
