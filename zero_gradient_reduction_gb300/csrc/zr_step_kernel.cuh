// Device side of the fused post-backward step (included by zr_step.cu and zr_inplace.cu):
// the kernel arguments, the per-step constants read from the control block, the
// last-block epilogue and fused_step_kernel itself, in three modes:
//   kPingPong  reads state set k, writes set 1-k; the last block decides and flips k;
//   kFlagPass  only forms the ring sums and ORs their non-finite flag (no state traffic);
//   kInPlace   after a kFlagPass launch: skips everything if the flag is set, else
//              updates one state set in place; the last block applies the scaler rule.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "zr_device.cuh"
#include "zr_internal.h"
#include "zr_plan.h"

namespace {

constexpr int kThreads = 256;
constexpr int kTileElems = 32768;  // elements per tile (a multiple of 8 * kThreads)

enum : int { kPingPong = 0, kFlagPass = 1, kInPlace = 2 };

struct FusedArgs {
  const void* grads[ZR_MAX_REPLICAS];      // replica w*A + a (16-bit of the param type, or fp32)
  int order[ZR_MAX_W];                     // ring position -> worker
  const int4* tiles;                       // {start lo, start hi, groups, block index c}
  int64_t tile0, tile1;                    // this launch's tiles: [tile0, tile1)
  unsigned total_blocks;                   // blocks over all launches of the step (one, or one per bucket)
  float* master[2];
  float* m[2];
  float* v[2];
  uint16_t* param[2];
  zr::Ctrl* ctrl;
  float lr, beta1, beta2, eps, weight_decay;
  int W, A, stage;
};

// Per-block view of the control block, read once at the start of the step.
struct StepConsts {
  zr::AdamConsts k;
  float r;  // fp32(1/(S*W))
  int cur;  // live state set
};

__device__ void read_consts(const FusedArgs& a, StepConsts& out) {
  const volatile zr::Ctrl* c = a.ctrl;
  const double S = (double)c->scale;
  const double p1 = c->prod1, p2 = c->prod2;
  out.cur = c->k;
  out.r = (float)__ddiv_rn(1.0, __dmul_rn(S, (double)a.W));
  out.k.b1 = a.beta1;
  out.k.b2 = a.beta2;
  out.k.omb1 = __fsub_rn(1.0f, a.beta1);
  out.k.omb2 = __fsub_rn(1.0f, a.beta2);
  out.k.lr = a.lr;
  out.k.eps = a.eps;
  out.k.decay = __fsub_rn(1.0f, __fmul_rn(a.lr, a.weight_decay));
  out.k.bc1 = (float)__dsub_rn(1.0, __dmul_rn(p1, (double)a.beta1));
  out.k.bc2 = (float)__dsub_rn(1.0, __dmul_rn(p2, (double)a.beta2));
}

// The loss-scale rule and commit, run by one thread of the last block. Every other block
// is done with the control block by then, so it is read in one round trip of 16-byte
// loads from L2, updated in registers and written back the same way (a chain of single
// volatile accesses cost several microseconds on small plans). In place there is one
// state set, so a clean step does not flip k.
template <int MODE>
__device__ void finish_step(const FusedArgs& a) {
  constexpr int kWords = sizeof(zr::Ctrl) / 16;
  union {
    zr::Ctrl c;
    uint4 w[kWords];
  } u;
  const uint4* src = reinterpret_cast<const uint4*>(a.ctrl);
#pragma unroll
  for (int i = 0; i < kWords; ++i) u.w[i] = __ldcg(src + i);
  zr::Ctrl& c = u.c;
  const int of = c.overflow;
  float scale = c.scale;
  c.last_overflow = of;
  c.scale_used = scale;
  c.stage = a.stage;
  c.steps = c.steps + 1;
  if (of) {
    c.skipped = c.skipped + 1;
    if (c.dynamic) {
      const float s2 = __fmul_rn(scale, c.backoff);
      scale = s2 > c.min_scale ? s2 : c.min_scale;
      c.good = 0;
    }
  } else {
    c.t = c.t + 1;
    c.prod1 = __dmul_rn(c.prod1, (double)a.beta1);
    c.prod2 = __dmul_rn(c.prod2, (double)a.beta2);
    if (MODE == kPingPong) c.k = 1 - c.k;
    c.good = c.good + 1;
    if (c.dynamic && c.good >= c.interval) {
      scale = __fmul_rn(scale, c.growth);
      c.good = 0;
    }
  }
  c.scale = scale;
  c.overflow = 0;
  c.ticket = 0;
  uint4* dst = reinterpret_cast<uint4*>(a.ctrl);
#pragma unroll
  for (int i = 0; i < kWords; ++i) __stcg(dst + i, u.w[i]);
  __threadfence();
}

// AdamW on one 8-element group whose ring sums are s[0..7] and whose state (read by
// the caller) is p/m/v; writes state set `out` at flat element e and returns whether
// any sum was not finite.
template <int DT>
__device__ __forceinline__ bool update_group(const FusedArgs& a, const StepConsts& K, int out, int64_t e,
                                             const float s[8], float4 p0, float4 p1, float4 m0, float4 m1, float4 v0,
                                             float4 v1) {
  float p[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
  float m[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float v[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  bool bad = false;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    bad |= zr::nonfinite(s[j]);
    zr::adamw_elem(__fmul_rn(s[j], K.r), p[j], m[j], v[j], K.k);
  }
  zr::st_once_f4(a.master[out] + e, make_float4(p[0], p[1], p[2], p[3]));
  zr::st_once_f4(a.master[out] + e + 4, make_float4(p[4], p[5], p[6], p[7]));
  zr::st_once_f4(a.m[out] + e, make_float4(m[0], m[1], m[2], m[3]));
  zr::st_once_f4(a.m[out] + e + 4, make_float4(m[4], m[5], m[6], m[7]));
  zr::st_once_f4(a.v[out] + e, make_float4(v[0], v[1], v[2], v[3]));
  zr::st_once_f4(a.v[out] + e + 4, make_float4(v[4], v[5], v[6], v[7]));
  zr::st_once(a.param[out] + e, zr::pack8<DT>(p));
  return bad;
}

// State loads: the non-coherent path for a set the launch does not write, the coherent
// one for the set an in-place launch overwrites.
template <int MODE>
__device__ __forceinline__ float4 ld_state(const float* p) {
  if constexpr (MODE == kInPlace) return zr::ld_rw_f4(p);
  else return zr::ld_once_f4(p);
}

// Ring-position pointers are computed per tile from the grid constants (block index c
// is uniform over the tile), so tiles need no shared table and no block barrier. For
// A = 1 with a compile-time W all W gradient loads and the six state loads of a group
// are issued before any arithmetic. The three modes share the ring-sum code, so a
// kFlagPass launch and the kInPlace launch after it fold every sum in the same order.
// Blocks per SM an instantiation is built for: two (up to 128 registers, so that a thread
// keeps a group's replica and state loads in flight), except W = 8 with A = 4, whose 32
// micro-batch streams are consumed as they arrive: there four blocks (64 registers, no
// spill) measured 3.9 % faster (16.90 against 17.58 ms on the 1.3B shapes). Four blocks
// made the W > 8 and the other A = 4 paths spill, and slowed W > 8 down.
template <int WT, int AT>
constexpr int step_min_blocks() { return (WT == 8 && AT == 4) ? 4 : 2; }

template <int DT, int WT, int AT, int GT, int MODE>
__global__ void __launch_bounds__(kThreads, step_min_blocks<WT, AT>())
    fused_step_kernel(const __grid_constant__ FusedArgs a) {
  constexpr bool kState = MODE != kFlagPass;  // reads and writes optimizer state
  __shared__ StepConsts s_k;
  __shared__ int s_bad, s_skip;
  __shared__ unsigned s_ticket;
  if (threadIdx.x == 0) {
    read_consts(a, s_k);
    s_bad = 0;
    // In place, the flag pass before this launch has already decided the step.
    s_skip = MODE == kInPlace ? static_cast<const volatile zr::Ctrl*>(a.ctrl)->overflow : 0;
  }
  __syncthreads();
  const StepConsts K = s_k;
  const bool skip = MODE == kInPlace && s_skip != 0;
  const int W = WT > 0 ? WT : a.W;
  const int A = AT > 0 ? AT : a.A;
  // In place the single state set is passed as set 0 and read and written there.
  const int in = MODE == kInPlace ? 0 : K.cur;
  const int out = MODE == kInPlace ? 0 : 1 - K.cur;
  const float* mst_in = a.master[in];
  const float* m_in = a.m[in];
  const float* v_in = a.v[in];
  bool bad = false;

  for (int64_t tile = a.tile0 + blockIdx.x; tile < a.tile1 && !skip; tile += gridDim.x) {
    const int4 d = a.tiles[tile];
    const int64_t start = (int64_t)(((uint64_t)(uint32_t)d.y << 32) | (uint32_t)d.x);
    const int groups = d.z, c = d.w;
    if (WT != 0 && AT == 1 && GT == DT) {
      // WT > 0: W known at compile time; WT < 0: any W <= 8, the missing replicas' loads
      // and additions predicated off (W is uniform, so no lane diverges).
      constexpr int WN = WT > 0 ? WT : 8;
      const uint16_t* gp[WN];
#pragma unroll
      for (int h = 0; h < WN; ++h) {
        if (WT > 0 || h < W) {
          int pos = c + h;  // c < W and h < W
          pos -= pos >= W ? W : 0;
          gp[h] = static_cast<const uint16_t*>(a.grads[a.order[pos]]) + start;
        } else {
          gp[h] = nullptr;
        }
      }
      // U groups per thread and iteration, all of their loads issued before any arithmetic:
      // with few replicas one group holds too few bytes in flight to cover HBM latency. The
      // flag pass has no state loads and registers to spare: 8/W groups (128 bytes in flight).
      constexpr int UN = WT < 0 ? 1 : MODE == kFlagPass ? (WN >= 8 ? 1 : 8 / WN) : (WN <= 3 ? 2 : 1);
      for (int g0 = threadIdx.x; g0 < groups; g0 += UN * blockDim.x) {
        uint4 raw[UN][WN];
        float4 st[UN][6];
#pragma unroll
        for (int u = 0; u < UN; ++u) {
          const int g = g0 + u * (int)blockDim.x;
          if (g < groups) {
            const int64_t off = (int64_t)g * 8, e = start + off;
#pragma unroll
            for (int h = 0; h < WN; ++h)
              if (WT > 0 || h < W) raw[u][h] = zr::ld_once(gp[h] + off);
            if constexpr (kState) {
              st[u][0] = ld_state<MODE>(mst_in + e);
              st[u][1] = ld_state<MODE>(mst_in + e + 4);
              st[u][2] = ld_state<MODE>(m_in + e);
              st[u][3] = ld_state<MODE>(m_in + e + 4);
              st[u][4] = ld_state<MODE>(v_in + e);
              st[u][5] = ld_state<MODE>(v_in + e + 4);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < UN; ++u) {
          const int g = g0 + u * (int)blockDim.x;
          if (g < groups) {
            float s[8];
            zr::unpack8<DT>(raw[u][0], s);
#pragma unroll
            for (int h = 1; h < WN; ++h) {
              if (WT > 0 || h < W) {
                float x[8];
                zr::unpack8<DT>(raw[u][h], x);
#pragma unroll
                for (int j = 0; j < 8; ++j) s[j] = __fadd_rn(s[j], x[j]);
              }
            }
            if constexpr (kState) {
              bad |= update_group<DT>(a, K, out, start + (int64_t)g * 8, s, st[u][0], st[u][1], st[u][2], st[u][3],
                                      st[u][4], st[u][5]);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) bad |= zr::nonfinite(s[j]);
            }
          }
        }
      }
    } else if (WT == 0 && AT == 1 && GT == DT) {
      // W > 8: the group's state loads, then the replicas in batches of kBatch, double
      // buffered: the next batch's loads are in flight while the current one is added in
      // ring order, so a thread never waits on fewer than kBatch replica loads.
      constexpr int kBatch = 8;
      for (int g = threadIdx.x; g < groups; g += blockDim.x) {
        const int64_t e = start + (int64_t)g * 8;
        float4 st[6];
        if constexpr (kState) {
          st[0] = ld_state<MODE>(mst_in + e);
          st[1] = ld_state<MODE>(mst_in + e + 4);
          st[2] = ld_state<MODE>(m_in + e);
          st[3] = ld_state<MODE>(m_in + e + 4);
          st[4] = ld_state<MODE>(v_in + e);
          st[5] = ld_state<MODE>(v_in + e + 4);
        }
        auto load_batch = [&](uint4(&raw)[kBatch], int h0) {
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            if (h0 + j < W) {
              int pos = c + h0 + j;  // c < W and h0 + j < W
              pos -= pos >= W ? W : 0;
              raw[j] = zr::ld_once(static_cast<const uint16_t*>(a.grads[a.order[pos]]) + e);
            }
          }
        };
        float s[8];
        auto add_batch = [&](const uint4(&raw)[kBatch], int h0) {
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            if (h0 + j < W) {
              float x[8];
              zr::unpack8<DT>(raw[j], x);
#pragma unroll
              for (int k = 0; k < 8; ++k) s[k] = h0 + j == 0 ? x[k] : __fadd_rn(s[k], x[k]);
            }
          }
        };
        uint4 ra[kBatch], rb[kBatch];
        load_batch(ra, 0);
        for (int h0 = 0; h0 < W; h0 += 2 * kBatch) {
          if (h0 + kBatch < W) load_batch(rb, h0 + kBatch);
          add_batch(ra, h0);
          if (h0 + 2 * kBatch < W) load_batch(ra, h0 + 2 * kBatch);
          if (h0 + kBatch < W) add_batch(rb, h0 + kBatch);
        }
        if constexpr (kState) {
          bad |= update_group<DT>(a, K, out, e, s, st[0], st[1], st[2], st[3], st[4], st[5]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) bad |= zr::nonfinite(s[j]);
        }
      }
    } else {
      for (int g = threadIdx.x; g < groups; g += blockDim.x) {
        const int64_t off = (int64_t)g * 8, e = start + off;
        float s[8];
        for (int h = 0; h < W; ++h) {
          int pos = c + h;
          pos -= pos >= W ? W : 0;
          const void* const* rep = a.grads + a.order[pos] * A;  // worker's A micro-batches
          float w8[8];
          zr::load8<GT>(rep[0], e, w8);
          for (int q = 1; q < A; ++q) {
            float x[8];
            zr::load8<GT>(rep[q], e, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) w8[j] = __fadd_rn(w8[j], x[j]);
          }
#pragma unroll
          for (int j = 0; j < 8; ++j) s[j] = h == 0 ? w8[j] : __fadd_rn(s[j], w8[j]);
        }
        if constexpr (kState) {
          const float4 p0 = ld_state<MODE>(mst_in + e), p1 = ld_state<MODE>(mst_in + e + 4);
          const float4 m0 = ld_state<MODE>(m_in + e), m1 = ld_state<MODE>(m_in + e + 4);
          const float4 v0 = ld_state<MODE>(v_in + e), v1 = ld_state<MODE>(v_in + e + 4);
          bad |= update_group<DT>(a, K, out, e, s, p0, p1, m0, m1, v0, v1);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) bad |= zr::nonfinite(s[j]);
        }
      }
    }
  }

  // Block flag -> control block. A flag pass stops there; otherwise the ticket: the last
  // block to arrive, over all launches of the step, decides (in place: only the scaler
  // rule, the flag pass having decided the skip).
  if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0) s_bad = 1;
  __syncthreads();
  if (MODE == kFlagPass) {
    if (threadIdx.x == 0 && s_bad) atomicOr(&a.ctrl->overflow, 1);
    return;
  }
  if (threadIdx.x == 0) {
    if (s_bad) atomicOr(&a.ctrl->overflow, 1);
    __threadfence();
    s_ticket = atomicAdd(&a.ctrl->ticket, 1u);
  }
  __syncthreads();
  if (s_ticket == a.total_blocks - 1 && threadIdx.x == 0) {
    __threadfence();
    finish_step<MODE>(a);
  }
}

using KernelFn = void (*)(FusedArgs);

// Host: the arguments of one launch over plan p's tiles [tile0, tile1), the step's
// launches adding up to `total` blocks. State set k is (master[k], m[k], v[k], param[k]).
inline FusedArgs make_args(const zr_plan* p, int stage, const void* const* grads, float* const master[2],
                           float* const m[2], float* const v[2], void* const param[2], const zr_adamw_hyper* h,
                           int64_t tile0, int64_t tile1, unsigned total) {
  FusedArgs a;
  std::memset(&a, 0, sizeof a);
  for (int r = 0; r < p->W * p->A; ++r) a.grads[r] = grads[r];
  for (int i = 0; i < p->W; ++i) a.order[i] = p->order[i];
  a.tiles = p->tiles_dev;
  a.tile0 = tile0;
  a.tile1 = tile1;
  a.total_blocks = total;
  for (int k = 0; k < 2; ++k) {
    a.master[k] = master[k];
    a.m[k] = m[k];
    a.v[k] = v[k];
    a.param[k] = static_cast<uint16_t*>(param[k]);
  }
  a.ctrl = p->ctrl_dev;
  a.lr = h->lr;
  a.beta1 = h->beta1;
  a.beta2 = h->beta2;
  a.eps = h->eps;
  a.weight_decay = h->weight_decay;
  a.W = p->W;
  a.A = p->A;
  a.stage = stage;
  return a;
}

// GT: the gradients' type (the param type DT, or fp32 accumulators).
template <int DT, int MODE>
KernelFn pick_kernel(int W, int A, bool fp32_grads) {
  constexpr int F = zr::DT_F32;
  if (fp32_grads) return A == 1 ? fused_step_kernel<DT, 0, 1, F, MODE> : fused_step_kernel<DT, 0, 0, F, MODE>;
  if (A == 1) {
    switch (W) {
      case 1: return fused_step_kernel<DT, 1, 1, DT, MODE>;
      case 2: return fused_step_kernel<DT, 2, 1, DT, MODE>;
      case 3: return fused_step_kernel<DT, 3, 1, DT, MODE>;
      case 4: return fused_step_kernel<DT, 4, 1, DT, MODE>;
      case 8: return fused_step_kernel<DT, 8, 1, DT, MODE>;
      default: return W < 8 ? fused_step_kernel<DT, -1, 1, DT, MODE> : fused_step_kernel<DT, 0, 1, DT, MODE>;
    }
  }
  if (A == 4) {
    switch (W) {
      case 2: return fused_step_kernel<DT, 2, 4, DT, MODE>;
      case 4: return fused_step_kernel<DT, 4, 4, DT, MODE>;
      case 8: return fused_step_kernel<DT, 8, 4, DT, MODE>;
      default: return fused_step_kernel<DT, 0, 4, DT, MODE>;
    }
  }
  return fused_step_kernel<DT, 0, 0, DT, MODE>;
}

}  // namespace
