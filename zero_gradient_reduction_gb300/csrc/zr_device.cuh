// Device helpers shared by the libzr kernels: streaming vector loads/stores,
// exact 16-bit <-> fp32 conversions for groups of 8 elements, and the
// non-finite test. Every fp32 operation in the kernels uses an explicit
// round-to-nearest intrinsic so that no multiply-add is ever contracted.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace zr {

enum { DT_F16 = 0, DT_BF16 = 1, DT_F32 = 2 };

// 16-byte load of data read exactly once: non-coherent path, no L1 allocation,
// 256-byte L2 prefetch granule. Not volatile, so the compiler may batch loads.
__device__ __forceinline__ uint4 ld_once(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 16-byte store of data not read again in this kernel (streaming, evict-first).
// No compiler memory clobber: the kernels never read what they store through these
// (inputs and outputs are distinct buffers, or a thread reads an element before it
// overwrites it), so later independent loads may be scheduled ahead of the store.
__device__ __forceinline__ void st_once(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
}

__device__ __forceinline__ float4 ld_once_f4(const float* p) {
  uint4 u = ld_once(p);
  return make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
}

// As ld_once, on the coherent path: for data the same kernel later overwrites in place
// (the non-coherent path is only defined for data that stays read-only for the launch).
__device__ __forceinline__ float4 ld_rw_f4(const float* p) {
  uint4 r;
  asm("ld.global.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return make_float4(__uint_as_float(r.x), __uint_as_float(r.y), __uint_as_float(r.z), __uint_as_float(r.w));
}

__device__ __forceinline__ void st_once_f4(float* p, float4 v) {
  st_once(p, make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w)));
}

// 8 consecutive 16-bit values (one 16-byte word) -> 8 fp32, exact.
template <int DT>
__device__ __forceinline__ void unpack8(const uint4 v, float f[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (DT == DT_BF16) {
      f[2 * j] = __uint_as_float(w[j] << 16);
      f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[j]);
      float2 t = __half22float2(h);
      f[2 * j] = t.x;
      f[2 * j + 1] = t.y;
    }
  }
}

// 8 fp32 -> 8 round-to-nearest-even 16-bit values packed in one 16-byte word.
template <int DT>
__device__ __forceinline__ uint4 pack8(const float f[8]) {
  uint32_t w[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (DT == DT_BF16) {
      __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&b);
    } else {
      __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <int DT>
__device__ __forceinline__ float to_f32(uint16_t b) {
  if (DT == DT_BF16) return __uint_as_float(static_cast<uint32_t>(b) << 16);
  return __half2float(__ushort_as_half(b));
}

template <int DT>
__device__ __forceinline__ uint16_t from_f32(float x) {
  if (DT == DT_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  return __half_as_ushort(__float2half_rn(x));
}

// Elements e .. e+7 of an array of type DT (fp16, bf16 or fp32) as 8 fp32 values, exact.
template <int DT>
__device__ __forceinline__ void load8(const void* base, int64_t e, float f[8]) {
  if (DT == DT_F32) {
    const float* p = static_cast<const float*>(base) + e;
    const float4 a = ld_once_f4(p), b = ld_once_f4(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  } else {
    unpack8<DT>(ld_once(static_cast<const uint16_t*>(base) + e), f);
  }
}

template <int DT>
__device__ __forceinline__ float load1(const void* base, int64_t i) {
  if (DT == DT_F32) return static_cast<const float*>(base)[i];
  return to_f32<DT>(static_cast<const uint16_t*>(base)[i]);
}

__device__ __forceinline__ bool nonfinite(float x) {
  return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// Per-element AdamW with decoupled weight decay, every op rounded once:
//   m = b1*m + (1-b1)*g ; v = b2*v + (1-b2)*(g*g)
//   u = (m/bc1) / (sqrt(v/bc2) + eps) ; p = p*(1-lr*wd) - lr*u
struct AdamConsts {
  float b1, b2, omb1, omb2, lr, eps, decay, bc1, bc2;
};

__device__ __forceinline__ void adamw_elem(float g, float& p, float& m, float& v, const AdamConsts& k) {
  const float mi = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, g));
  const float vi = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(g, g)));
  const float mhat = __fdiv_rn(mi, k.bc1);
  const float vhat = __fdiv_rn(vi, k.bc2);
  const float den = __fadd_rn(__fsqrt_rn(vhat), k.eps);
  const float u = __fdiv_rn(mhat, den);
  p = __fsub_rn(__fmul_rn(p, k.decay), __fmul_rn(k.lr, u));
  m = mi;
  v = vi;
}

}  // namespace zr
