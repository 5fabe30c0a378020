// Device side of the synthetic input generator: the same values as
// zrgen_fill_normal_host (see zrgen.h), written straight into HBM so that
// multi-GB inputs take milliseconds. Inputs only; none of the step's arithmetic.
#include "zrgen.h"
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

namespace {

__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    uint32_t hi0 = __umulhi(0xD2511F53u, c[0]), lo0 = 0xD2511F53u * c[0];
    uint32_t hi1 = __umulhi(0xCD9E8D57u, c[2]), lo1 = 0xCD9E8D57u * c[2];
    uint32_t n0 = hi1 ^ c[1] ^ k0;
    uint32_t n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0; c[1] = lo1; c[2] = n2; c[3] = lo0;
  }
}

template <int DT>
__global__ void fill_normal_kernel(void* __restrict__ out, uint64_t n, uint64_t seed, uint64_t stream,
                                   uint64_t first, float scale, const float* __restrict__ table) {
  // One thread per Philox block (8 consecutive element indices).
  const uint64_t first_block = first >> 3;
  const uint64_t last_block = (first + n - 1) >> 3;
  const uint64_t nblocks = last_block - first_block + 1;
  for (uint64_t t = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; t < nblocks;
       t += (uint64_t)gridDim.x * blockDim.x) {
    uint64_t blk = first_block + t;
    uint32_t c[4] = {(uint32_t)blk, (uint32_t)(blk >> 32), (uint32_t)stream, (uint32_t)(stream >> 32)};
    philox4x32_10(c, (uint32_t)seed, (uint32_t)(seed >> 32));
#pragma unroll
    for (int lane = 0; lane < 8; ++lane) {
      uint64_t idx = blk * 8 + lane;
      if (idx < first || idx >= first + n) continue;
      uint32_t w = c[lane >> 1];
      uint32_t u = (lane & 1) ? (w >> 16) : (w & 0xFFFFu);
      float v = __fmul_rn(__ldg(table + u), scale);
      uint64_t j = idx - first;
      if (DT == ZRGEN_F32) static_cast<float*>(out)[j] = v;
      else if (DT == ZRGEN_F16) static_cast<__half*>(out)[j] = __float2half_rn(v);
      else static_cast<__nv_bfloat16*>(out)[j] = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace

extern "C" int zrgen_fill_normal_dev(void* out, int dtype, uint64_t n, uint64_t seed, uint64_t stream,
                                     uint64_t first, float scale, const float* table_dev,
                                     void* stream_handle) {
  if (n == 0) return 0;
  if (!out || !table_dev) return -1;
  cudaStream_t s = static_cast<cudaStream_t>(stream_handle);
  const uint64_t nblocks = ((first + n - 1) >> 3) - (first >> 3) + 1;
  const int threads = 256;
  uint64_t want = (nblocks + threads - 1) / threads;
  int grid = (int)(want < 152ull * 32ull ? want : 152ull * 32ull);
  switch (dtype) {
    case ZRGEN_F16: fill_normal_kernel<ZRGEN_F16><<<grid, threads, 0, s>>>(out, n, seed, stream, first, scale, table_dev); break;
    case ZRGEN_BF16: fill_normal_kernel<ZRGEN_BF16><<<grid, threads, 0, s>>>(out, n, seed, stream, first, scale, table_dev); break;
    case ZRGEN_F32: fill_normal_kernel<ZRGEN_F32><<<grid, threads, 0, s>>>(out, n, seed, stream, first, scale, table_dev); break;
    default: return -1;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
