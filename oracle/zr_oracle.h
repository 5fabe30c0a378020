/*
 * zr_oracle — TEST INFRASTRUCTURE. The plain, slow, single-threaded CPU oracle of
 * the data-parallel step that runs after backward (ring reduce-scatter of W
 * gradient replicas, loss-unscale, overflow check, mixed-precision AdamW on each
 * worker's fp32 shard, cast, ring all-gather of the 16-bit params).
 *
 * It shares no code with the CUDA path and is used only by the tests, by the
 * smoke check and by the benchmark's CPU-baseline leg. The product never calls it.
 *
 * Sources (the pages, cited by title and section):
 *  [P1] "DP / DDP / ZeRO-1 / ZeRO-2 & ZeRO-3" article (gitcode.csdn.net), section 二 (DDP):
 *       the three-GPU A/B/C ring walk-through (scatter reduce, then all-gather),
 *       the per-GPU traffic (N-1)*phi/N per phase; section 三 (ZeRO-1): owner
 *       averages its shard, converts to FP32, scales, updates m, v, then the FP32
 *       master, then the FP16 params, which are broadcast; "2+2+K" memory count.
 *  [P2] "DeepSpeed introduction" (nanhubrain.csdn.net), 核心技术 (1)-(3): mixed
 *       precision with dynamic loss scaling, BF16 vs FP16; (11)-(13) ZeRO stages.
 *  [P3] "CS336 lecture 7: Parallelism" (cs336.sjfarm.cc): the 16N memory table,
 *       the data-parallel mean equivalence, Ring AllReduce = ReduceScatter +
 *       AllGather with traffic M(W-1)/W per phase, ZeRO stage memory formulas,
 *       torch.optim.AdamW in the DDP loop, gradient accumulation.
 *
 * Readings where the pages leave a step open (each one is stated at its function):
 *  - all stages use ReduceScatter for the gradients; the reduction accumulates in
 *    fp32 starting from the chunk-origin worker's value, in ring order;
 *  - chunk size C = align * ceil(n / (align * W)); the last chunks may be short
 *    or empty (equivalent to zero padding to W*C);
 *  - position p owns chunk (p+1) mod W after reduce-scatter ([P1] 二: GPU0 ends
 *    with B, GPU1 with C, GPU2 with A);
 *  - the mean's 1/W is folded with 1/S into r = fp32(1/(S*W)) computed in double;
 *  - decoupled AdamW (Loshchilov & Hutter) in the op order of zro_adamw;
 *  - loss scaler: skip on any non-finite reduced value; dynamic: S <- max(S*backoff,
 *    min_scale) on skip, S <- S*growth after `interval` clean steps.
 *
 * Parity pins: every function here is pinned by a test in tests/test_oracle_*.py
 * except the exact fp32 rounding order of the AdamW update, which the pages do not
 * print; it is pinned by closed forms and by torch.optim.AdamW within 2 ulp, not
 * bit for bit (parity unpinned at the last-ulp level).
 */
#ifndef ZR_ORACLE_H
#define ZR_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZRO_MAX_W 64

enum { ZRO_F16 = 0, ZRO_BF16 = 1 };

typedef struct {
    int64_t start; /* flat offset of the bucket */
    int64_t len;   /* elements in the bucket */
    int64_t chunk; /* C: elements per ring chunk (the last ones may be short) */
} zro_bucket;

typedef struct { float lr, beta1, beta2, eps, weight_decay; } zro_hyper;

typedef struct {
    float scale;        /* current loss scale S */
    int64_t good;       /* clean steps since the last scale change */
    int64_t t;          /* committed AdamW steps */
    double prod1, prod2;/* running products beta1^t, beta2^t */
    float backoff, growth, min_scale;
    int64_t interval;
    int dynamic;
} zro_scaler;

typedef struct {
    int overflow;       /* OR over all reduced values of !isfinite */
    int skipped;        /* update skipped (== overflow) */
    float scale_used;   /* S of this step */
    float scale_next;   /* S after the scaler rule */
    int64_t t_after;
    int64_t rs_sent[ZRO_MAX_W], rs_recv[ZRO_MAX_W]; /* elements, per worker id */
    int64_t ag_sent[ZRO_MAX_W], ag_recv[ZRO_MAX_W];
} zro_report;

/* ---- layout ---- */
int64_t zro_chunk_size(int64_t n, int W, int align);
int zro_bucket_plan(const int64_t* numels, int ntensors, int64_t cap, int W, int align,
                    zro_bucket* buckets, int* nbuckets, int64_t* tensor_offset);

/* ---- number formats ---- */
float zro_f16_to_f32(uint16_t h);
float zro_bf16_to_f32(uint16_t h);
uint16_t zro_f32_to_f16(float x);
uint16_t zro_f32_to_bf16(float x);
void zro_decode(int dtype, const uint16_t* in, float* out, int64_t n);
void zro_encode(int dtype, const float* in, uint16_t* out, int64_t n);
void zro_accumulate(int dtype, const uint16_t* g, float* acc, int64_t n, int first);

/* ---- ring collectives over one bucket, by ring position ---- */
void zro_ring_reduce_scatter(int W, int64_t n, int64_t C, float* const* work, float* msg,
                             int64_t* sent, int64_t* recv);
void zro_ring_reduce_scatter_hops(int W, int64_t n, int64_t C, float* const* work, float* msg,
                                  int64_t* sent, int64_t* recv, int s0, int s1);
void zro_ring_all_gather_hops(int W, int64_t n, int64_t C, uint16_t* const* rep, uint16_t* msg,
                              int64_t* sent, int64_t* recv, int s0, int s1);
void zro_ring_all_gather(int W, int64_t n, int64_t C, uint16_t* const* rep, uint16_t* msg,
                         int64_t* sent, int64_t* recv);
void zro_ring_all_reduce(int W, int64_t n, int64_t C, float* const* work, float* msg,
                         int64_t* sent, int64_t* recv);
void zro_ring_traffic(int64_t n, int W, int align, int64_t* sent_per_pos, int64_t* recv_per_pos);

/* ---- ZeRO-3 parameter shards and the all-gather before forward/backward ---- */
void zro_shard_params(int W, const int* order, int nbuckets, const zro_bucket* buckets, const uint16_t* replica,
                      uint16_t* const* shards);
int zro_param_all_gather(int W, const int* order, int nbuckets, const zro_bucket* buckets, int b_lo, int b_hi,
                         const uint16_t* const* shards, uint16_t* replica);

/* ---- per-shard arithmetic ---- */
float zro_unscale_factor(float scale, int W);
float zro_bias_correction(float beta, int64_t t);
void zro_adamw(int64_t len, const float* g, float* p, float* m, float* v,
               const zro_hyper* h, float bc1, float bc2);

/* ---- one whole step ---- */
int zro_step(int W, int A, int dtype, const int* order, int nbuckets, const zro_bucket* buckets,
             const uint16_t* const* grads, float* master, float* m, float* v, uint16_t* param,
             const zro_hyper* h, zro_scaler* sc, int flag_override, float* sums_out, zro_report* rep);

/* ---- memory accounting ---- */
int64_t zro_model_state_bytes(int stage, int64_t n, int W);

#ifdef __cplusplus
}
#endif
#endif
