// The fused step with bulk-copy staging for plans with more than kChunkSlices replica
// slices per element (W * A > 8; included by zr_step.cu after zr_step_bulk.cuh). One stage
// of fused_bulk_kernel holds every slice of its elements, so many slices shrink its stages
// until most consumer threads have no group to work on. Here the slices of one range of
// E elements are spread over ceil(W * A / 8) consecutive stages of 8 slices each; a
// consumer thread keeps its group's running ring sum and its worker's running micro-batch
// sum in registers from one stage to the next, so the fold is the same sequence of fp32
// additions in the same order (workers in ring order starting at position c, each
// worker's micro-batches in order). The range's master/m/v arrive with its last stage,
// where the update, cast and stores run as in fused_bulk_kernel. Producer, mbarriers,
// bounded waits, flag, ticket and epilogue are those of fused_bulk_kernel.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kChunkSlices = 8;    // replica slices per stage
constexpr int kChunkMaxElems = 2048;  // elements per stage: at most one 8-element group per consumer thread

// Stage layout: kChunkSlices slices of E 16-bit values, then E fp32 master, m and v values
// (filled on a range's last stage only).
__host__ __device__ inline int chunked_stage_bytes(int E) { return kChunkSlices * E * 2 + 12 * E; }

struct ChunkHdr {
  int64_t start;  // flat index of the range's first element
  int count;      // elements in the range (0 marks the end of the block's work)
  int c;          // ring block index of the tile
  int r0, nr;     // the stage holds slices [r0, r0 + nr) of the ring-ordered sequence
  int last;       // the range's last stage: master/m/v are in it
};

template <int DT, int AT>
__global__ void __launch_bounds__(bulk_threads(false), 2) fused_bulk_chunked_kernel(const __grid_constant__ FusedArgs a,
                                                                                 const BulkCfg cfg) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kBulkMaxStages], empty[kBulkMaxStages];
  __shared__ ChunkHdr hdr[kBulkMaxStages];
  __shared__ StepConsts s_k;
  __shared__ int s_bad, s_err;
  __shared__ unsigned s_ticket;
  const int W = a.W;
  const int A = AT > 0 ? AT : a.A;
  const int R = W * A;  // slices per element, in ring order: worker h's micro-batches at h*A .. h*A + A-1
  const int E = cfg.E, NS = cfg.NS;
  const int slot16 = E * 2, stage_bytes = chunked_stage_bytes(E);
  const int nsub = (R + kChunkSlices - 1) / kChunkSlices;  // stages per range
  if (threadIdx.x == 0) {
    read_consts(a, s_k);
    s_bad = 0;
    s_err = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kBulkConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const StepConsts K = s_k;
  const int in = K.cur, out = 1 - K.cur;
  bool bad = false;

  if (warp == 0) {
    if (lane == 0) {
      int64_t it = 0;
      bool ok = true;
      for (int64_t tile = a.tile0 + blockIdx.x; tile < a.tile1 && ok; tile += gridDim.x) {
        const int4 d = a.tiles[tile];
        const int64_t start = (int64_t)(((uint64_t)(uint32_t)d.y << 32) | (uint32_t)d.x);
        const int n = d.z * 8, c = d.w;
        for (int off = 0; off < n && ok; off += E) {
          const int cnt = n - off < E ? n - off : E;
          const int64_t e0 = start + off;
          for (int j = 0; j < nsub; ++j, ++it) {
            const int s = (int)(it % NS);
            if (it >= NS && !mbar_wait(&empty[s], (uint32_t)(((it / NS) - 1) & 1))) {
              ok = false;
              break;
            }
            const int r0 = j * kChunkSlices, nr = R - r0 < kChunkSlices ? R - r0 : kChunkSlices;
            const bool last = j == nsub - 1;
            hdr[s].start = e0;
            hdr[s].count = cnt;
            hdr[s].c = c;
            hdr[s].r0 = r0;
            hdr[s].nr = nr;
            hdr[s].last = last ? 1 : 0;
            mbar_arrive_tx(&full[s], (uint32_t)(nr * cnt * 2 + (last ? 12 * cnt : 0)) + cfg.stall_tx);
            unsigned char* base = smem + (size_t)s * stage_bytes;
            for (int k = 0; k < nr; ++k) {
              const int r = r0 + k, h = r / A, q = r - h * A;
              int pos = c + h;  // c < W and h < W
              pos -= pos >= W ? W : 0;
              const void* src = a.grads[a.order[pos] * A + q];
              bulk_load(base + k * slot16, static_cast<const uint16_t*>(src) + e0, cnt * 2, &full[s]);
            }
            if (last) {
              bulk_load(base + kChunkSlices * slot16, a.master[in] + e0, cnt * 4, &full[s]);
              bulk_load(base + kChunkSlices * slot16 + 4 * E, a.m[in] + e0, cnt * 4, &full[s]);
              bulk_load(base + kChunkSlices * slot16 + 8 * E, a.v[in] + e0, cnt * 4, &full[s]);
            }
          }
        }
      }
      if (ok) {
        // end marker: a stage with no elements, once the consumers have released its slot
        const int s = (int)(it % NS);
        if (it >= NS && !mbar_wait(&empty[s], (uint32_t)(((it / NS) - 1) & 1))) {
          ok = false;
        } else {
          hdr[s].count = 0;
          mbar_arrive(&full[s]);
        }
      }
      if (!ok) {
        // the consumers stopped releasing stages: let the copies already issued land before
        // the block (and its shared memory) goes away, then report
        s_err = 1;
        for (int64_t j = it - NS > 0 ? it - NS : 0; j < it; ++j)
          mbar_wait(&full[(int)(j % NS)], (uint32_t)((j / NS) & 1));
      }
    }
  } else {
    const int g = threadIdx.x - 32;  // this thread's 8-element group of every range (E <= 8 * 256)
    float sum[8], w8[8];             // carried from one stage of a range to the next
    for (int64_t it = 0;; ++it) {
      const int s = (int)(it % NS);
      if (!mbar_wait(&full[s], (uint32_t)((it / NS) & 1))) {
        if (lane == 0) s_err = 1;
        break;
      }
      const ChunkHdr H = hdr[s];
      if (H.count == 0) break;
      const unsigned char* base = smem + (size_t)s * stage_bytes;
      if (g < H.count / 8) {
        for (int k = 0; k < H.nr; ++k) {
          const int r = H.r0 + k, h = r / A, q = r - h * A;
          float x[8];
          zr::unpack8<DT>(*reinterpret_cast<const uint4*>(base + k * slot16 + g * 16), x);
          if (q == 0) {
#pragma unroll
            for (int e = 0; e < 8; ++e) w8[e] = x[e];
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) w8[e] = __fadd_rn(w8[e], x[e]);
          }
          if (q == A - 1) {
            if (h == 0) {
#pragma unroll
              for (int e = 0; e < 8; ++e) sum[e] = w8[e];
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) sum[e] = __fadd_rn(sum[e], w8[e]);
            }
          }
        }
        if (H.last) {
          const float4* ps = reinterpret_cast<const float4*>(base + kChunkSlices * slot16) + 2 * g;
          const float4* ms = reinterpret_cast<const float4*>(base + kChunkSlices * slot16 + 4 * E) + 2 * g;
          const float4* vs = reinterpret_cast<const float4*>(base + kChunkSlices * slot16 + 8 * E) + 2 * g;
          bad |= update_group<DT>(a, K, out, H.start + (int64_t)g * 8, sum, ps[0], ps[1], ms[0], ms[1], vs[0],
                                  vs[1]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
  }

  // Block flag -> control block, then the ticket: the last block to arrive decides. A
  // block whose waits gave up marks the step as failed; its last block then skips it.
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) s_bad = 1;
  __syncthreads();
  if (threadIdx.x == 0) {
    if (s_bad) atomicOr(&a.ctrl->overflow, 1);
    if (s_err) atomicOr(&a.ctrl->error, 1);
    __threadfence();
    s_ticket = atomicAdd(&a.ctrl->ticket, 1u);
  }
  __syncthreads();
  if (s_ticket == a.total_blocks - 1 && threadIdx.x == 0) {
    __threadfence();
    if (*static_cast<volatile int32_t*>(&a.ctrl->error)) atomicOr(&a.ctrl->overflow, 1);
    __threadfence();
    finish_step<kPingPong>(a);
  }
}

template <int DT>
BulkKernelFn pick_chunked_kernel(int A) {
  return A == 1 ? fused_bulk_chunked_kernel<DT, 1> : A == 4 ? fused_bulk_chunked_kernel<DT, 4> : fused_bulk_chunked_kernel<DT, 0>;
}

}  // namespace
