// The fused step with its loads staged by bulk copies (included by zr_step.cu after
// zr_step_kernel.cuh): the same arithmetic, ring order, flag, ticket and epilogue as
// fused_step_kernel in kPingPong mode, but the W replica slices and the master/m/v slices
// of each stage of a tile reach shared memory through one-dimensional cp.async.bulk copies
// (this GPU's own memory, no multicast, no cluster), so no register holds a load in flight.
//
// A block is one producer warp and kBulkConsumerWarps consumer warps (plus a storer warp
// when the results leave by bulk copies too). The producer walks the block's tiles in
// stages of E elements and keeps a ring of NS stages filled: it waits until a stage has
// been released (the stage's `empty` barrier), announces the stage's bytes on its `full`
// barrier and issues W + 3 bulk copies that complete on it. The consumers wait for a
// stage's `full` barrier, fold the W replicas in ring order, update the 8-element groups
// and store the results straight to global memory, then release the stage; or, with the
// storer, write the results back into the stage's slots and signal the storer (`done`),
// which copies them out and releases the stage once its copies have read it. No block
// barrier is taken inside the loop. Every wait gives up after kBulkWaitNs and records an
// error in the control block; the step is then skipped and zr_plan_report returns
// ZR_ERR_TIMEOUT.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr int kBulkConsumerWarps = 8;
// threads of a block: the producer warp, the storer warp when stores are bulk too, consumers
__host__ __device__ constexpr int bulk_threads(bool store_bulk) {
  return (kBulkConsumerWarps + (store_bulk ? 2 : 1)) * 32;
}
constexpr int kBulkMaxStages = 4;
constexpr uint64_t kBulkWaitNs = 2000000000ull;  // 2 s for one stage is a fault, not a slow step

struct BulkCfg {
  int E;             // elements per stage (a multiple of 8)
  int NS;            // stages in the ring (<= kBulkMaxStages)
  uint32_t stall_tx; // test hook: bytes announced on every stage beyond those copied (0 in use)
};

struct StageHdr {
  int64_t start;  // flat index of the stage's first element
  int count;      // elements in the stage (0 marks the end of the block's work)
  int c;          // ring block index of the tile
};

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// One arrival that also announces `bytes` of bulk-copy traffic the phase must wait for.
__device__ __forceinline__ void mbar_arrive_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with parity `parity` to complete, for at most kBulkWaitNs.
__device__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = now_ns();
  while (!mbar_try(bar, parity))
    if (now_ns() - t0 > kBulkWaitNs) return false;
  return true;
}

// `bytes` (a multiple of 16, both addresses 16-byte aligned) from global to this block's
// shared memory; completion is counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// `bytes` (a multiple of 16, both addresses 16-byte aligned) from this block's shared memory
// to global memory, in the executing thread's current bulk group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until the executing thread's bulk groups have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Waits until the executing thread's bulk groups have completed their writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's earlier shared-memory writes before later bulk copies that read them.
__device__ __forceinline__ void fence_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Stage layout in shared memory: R = W*A replica slices of E 16-bit values (ring position
// order, each worker's A micro-batches together), then E fp32 master, m and v values.
__host__ __device__ inline int bulk_stage_bytes(int R, int E) { return R * E * 2 + 12 * E; }

// SB (store bulk): the consumers write a stage's results back into its shared-memory slots
// (the new master/m/v over the old ones, the 16-bit parameter over the first replica slice)
// and a storer warp (warp 1) copies them out with bulk copies; the stage's slot is released
// to the producer once those copies have read it. Without SB the consumers store to global
// memory directly and release the slot themselves.
template <int DT, int WT, int AT, bool SB>
__global__ void __launch_bounds__(bulk_threads(SB), 2) fused_bulk_kernel(const __grid_constant__ FusedArgs a,
                                                                         const BulkCfg cfg) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[kBulkMaxStages], empty[kBulkMaxStages], done[kBulkMaxStages];
  __shared__ StageHdr hdr[kBulkMaxStages];
  __shared__ StepConsts s_k;
  __shared__ int s_bad, s_err;
  __shared__ unsigned s_ticket;
  const int W = WT > 0 ? WT : a.W;
  const int A = AT > 0 ? AT : a.A;
  const int R = W * A;  // replica slices per stage
  const int E = cfg.E, NS = cfg.NS;
  const int slot16 = E * 2, stage_bytes = bulk_stage_bytes(R, E);
  if (threadIdx.x == 0) {
    read_consts(a, s_k);
    s_bad = 0;
    s_err = 0;
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], SB ? 1 : kBulkConsumerWarps);
      mbar_init(&done[s], kBulkConsumerWarps);
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
        for (int off = 0; off < n; off += E, ++it) {
          const int s = (int)(it % NS);
          if (it >= NS && !mbar_wait(&empty[s], (uint32_t)(((it / NS) - 1) & 1))) {
            ok = false;
            break;
          }
          const int cnt = n - off < E ? n - off : E;
          const int64_t e0 = start + off;
          hdr[s].start = e0;
          hdr[s].count = cnt;
          hdr[s].c = c;
          mbar_arrive_tx(&full[s], (uint32_t)bulk_stage_bytes(R, cnt) + cfg.stall_tx);
          unsigned char* base = smem + (size_t)s * stage_bytes;
          for (int h = 0; h < W; ++h) {
            int pos = c + h;  // c < W and h < W
            pos -= pos >= W ? W : 0;
            const void* const* rep = a.grads + a.order[pos] * A;  // that worker's A micro-batches
            for (int q = 0; q < A; ++q)
              bulk_load(base + (h * A + q) * slot16, static_cast<const uint16_t*>(rep[q]) + e0, cnt * 2, &full[s]);
          }
          bulk_load(base + R * slot16, a.master[in] + e0, cnt * 4, &full[s]);
          bulk_load(base + R * slot16 + 4 * E, a.m[in] + e0, cnt * 4, &full[s]);
          bulk_load(base + R * slot16 + 8 * E, a.v[in] + e0, cnt * 4, &full[s]);
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
  } else if (SB && warp == 1) {
    if (lane == 0) {
      // storer: once the consumers are done with a stage, copy its results out and release
      // the slot when the copies have read it
      for (int64_t it = 0;; ++it) {
        const int s = (int)(it % NS);
        if (!mbar_wait(&done[s], (uint32_t)((it / NS) & 1))) {
          s_err = 1;
          break;
        }
        const StageHdr H = hdr[s];
        if (H.count == 0) break;
        unsigned char* base = smem + (size_t)s * stage_bytes;
        const int64_t e0 = H.start;
        bulk_store(a.master[out] + e0, base + R * slot16, H.count * 4);
        bulk_store(a.m[out] + e0, base + R * slot16 + 4 * E, H.count * 4);
        bulk_store(a.v[out] + e0, base + R * slot16 + 8 * E, H.count * 4);
        bulk_store(a.param[out] + e0, base, H.count * 2);
        bulk_commit();
        bulk_wait_read();
        mbar_arrive(&empty[s]);
      }
      bulk_wait_all();
    }
  } else {
    const int ct = threadIdx.x - (SB ? 64 : 32);
    for (int64_t it = 0;; ++it) {
      const int s = (int)(it % NS);
      if (!mbar_wait(&full[s], (uint32_t)((it / NS) & 1))) {
        if (lane == 0) s_err = 1;
        break;
      }
      const StageHdr H = hdr[s];
      if (H.count == 0) {
        if (SB) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&done[s]);  // tells the storer the block's work is over
        }
        break;
      }
      unsigned char* base = smem + (size_t)s * stage_bytes;
      const int groups = H.count / 8;
      for (int g = ct; g < groups; g += kBulkConsumerWarps * 32) {
        float sum[8];
        if constexpr (WT > 0 && AT == 1) {
          zr::unpack8<DT>(*reinterpret_cast<const uint4*>(base + g * 16), sum);
#pragma unroll
          for (int h = 1; h < WT; ++h) {
            float x[8];
            zr::unpack8<DT>(*reinterpret_cast<const uint4*>(base + h * slot16 + g * 16), x);
#pragma unroll
            for (int j = 0; j < 8; ++j) sum[j] = __fadd_rn(sum[j], x[j]);
          }
        } else {
          // each worker's micro-batches summed in order, then the workers in ring order
          for (int h = 0; h < W; ++h) {
            float w8[8];
            zr::unpack8<DT>(*reinterpret_cast<const uint4*>(base + (h * A) * slot16 + g * 16), w8);
            for (int q = 1; q < A; ++q) {
              float x[8];
              zr::unpack8<DT>(*reinterpret_cast<const uint4*>(base + (h * A + q) * slot16 + g * 16), x);
#pragma unroll
              for (int j = 0; j < 8; ++j) w8[j] = __fadd_rn(w8[j], x[j]);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) sum[j] = h == 0 ? w8[j] : __fadd_rn(sum[j], w8[j]);
          }
        }
        float4* ps = reinterpret_cast<float4*>(base + R * slot16) + 2 * g;
        float4* ms = reinterpret_cast<float4*>(base + R * slot16 + 4 * E) + 2 * g;
        float4* vs = reinterpret_cast<float4*>(base + R * slot16 + 8 * E) + 2 * g;
        if constexpr (SB) {
          const float4 p0 = ps[0], p1 = ps[1], m0 = ms[0], m1 = ms[1], v0 = vs[0], v1 = vs[1];
          float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
          float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            bad |= zr::nonfinite(sum[j]);
            zr::adamw_elem(__fmul_rn(sum[j], K.r), p[j], m[j], v[j], K.k);
          }
          ps[0] = make_float4(p[0], p[1], p[2], p[3]);
          ps[1] = make_float4(p[4], p[5], p[6], p[7]);
          ms[0] = make_float4(m[0], m[1], m[2], m[3]);
          ms[1] = make_float4(m[4], m[5], m[6], m[7]);
          vs[0] = make_float4(v[0], v[1], v[2], v[3]);
          vs[1] = make_float4(v[4], v[5], v[6], v[7]);
          *reinterpret_cast<uint4*>(base + g * 16) = zr::pack8<DT>(p);  // over this group's first replica values
        } else {
          bad |= update_group<DT>(a, K, out, H.start + (int64_t)g * 8, sum, ps[0], ps[1], ms[0], ms[1], vs[0],
                                  vs[1]);
        }
      }
      if constexpr (SB) {
        fence_to_async();  // the results written above, before the storer's bulk copies read them
        __syncwarp();
        if (lane == 0) mbar_arrive(&done[s]);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      }
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

using BulkKernelFn = void (*)(FusedArgs, BulkCfg);

template <int DT, bool SB>
BulkKernelFn pick_bulk_kernel(int W, int A) {
  if (A == 1 && W == 2) return fused_bulk_kernel<DT, 2, 1, SB>;
  if (A == 1 && W == 8) return fused_bulk_kernel<DT, 8, 1, SB>;
  return fused_bulk_kernel<DT, 0, 0, SB>;
}

}  // namespace
