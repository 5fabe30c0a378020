// Internal declarations shared by the libzr translation units (host side).
#pragma once
#include <cstdint>
#include <string>

#include "zr.h"

namespace zr {

// Thread-local last-error message; returns `s` for tail calls. For ZR_ERR_CUDA and
// ZR_ERR_OOM it also clears the CUDA runtime's last error (take_cuda_error).
zr_status fail(zr_status s, const char* fmt, ...);
void take_cuda_error();
void clear_error();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Control block of a plan, resident in device memory. Written by the last block of
// each fused step; read at the start of every block of the next one.
struct Ctrl {
  int32_t k;              // live state set
  int32_t overflow;       // OR of this step's block flags (0 between steps)
  uint32_t ticket;        // blocks finished in this step (0 between steps)
  int32_t last_overflow;  // flag of the last finished step
  float scale;            // loss scale for the next step
  float scale_used;       // loss scale of the last finished step
  int32_t dynamic;
  int32_t interval;
  float backoff, growth, min_scale;
  int32_t stage;          // stage of the last step
  int64_t good, t, steps, skipped;
  double prod1, prod2;    // beta1^t, beta2^t (running products)
  int32_t offload_flag;   // overflow flag of the reduce-scatter in zr_offload_step
  int32_t error;          // a bulk-staged step gave up a wait (the step was skipped); cleared by a reset
  int32_t pad[2];         // to a multiple of 16 bytes: the step's epilogue moves it as 16-byte words
};
static_assert(sizeof(Ctrl) % 16 == 0, "Ctrl is read and written as 16-byte words");

// beta^n as the running product the fused step keeps in its control block (one double
// multiplication per clean step, from 1.0), continued from p = beta^k (k <= n). The walk
// stops once the product no longer changes: for 0 <= beta < 1 it settles at zero or at a
// subnormal fixed point (after about 745 / (1 - beta) factors), so any n costs at most that.
double beta_power_from(double p, int64_t k, float beta, int64_t n);
// fp32(1 - beta^t), the bias correction of update t.
float bias_correction_host(float beta, int64_t t);
// 0 <= beta < 1 for both betas (what the host-side powers above need to terminate early).
bool betas_ok(const zr_adamw_hyper& h);

// The host AdamW of ZeRO-Offload (zr_offload_host.cpp): its constants for one step, and
// the update plus 16-bit cast of elements [lo, hi), for callers that run their own threads.
struct OffloadConsts {
  float b1, b2, omb1, omb2, lr, eps, decay, bc1, bc2, r;
};
OffloadConsts offload_consts(const zr_adamw_hyper& h, float loss_scale, int W, int64_t t);
void offload_update(const float* sums, float* master, float* m, float* v, void* param16, zr_dtype dt, int64_t lo,
                    int64_t hi, const OffloadConsts& k);

}  // namespace zr
