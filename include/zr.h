/*
 * zr.h — C ABI of libzr: the data-parallel step that runs after backward, on one GB300.
 *
 * W data-parallel workers are emulated as W gradient replicas resident in one GPU's
 * HBM. The step ring-reduce-scatters their gradient buckets, removes the loss scale
 * and takes the mean, checks for overflow, runs a mixed-precision AdamW update of
 * each owner's fp32 master/m/v shard, casts the shard to fp16/bf16 and all-gathers
 * it into the full parameter replica.
 *
 * Pages the operations follow (cited by title and section):
 *  [P1] "DP / DDP / DeepSpeed ZeRO-1/2/3" (gitcode.csdn.net): 二 DDP — ring
 *       all-reduce walk-through (scatter reduce, then all-gather), reverse-order
 *       buckets, per-GPU traffic; 三 ZeRO-1 — owners average, convert to FP32,
 *       scale, update m, v, master, then the FP16 params, and broadcast them;
 *       四 ZeRO-2/3 — gradient and parameter sharding.
 *  [P2] "并行训练框架DeepSpeed介绍" (nanhubrain.csdn.net): 核心技术 (1)-(3) mixed
 *       precision, BF16/FP16, dynamic loss scaling; (11)-(13) ZeRO-1/2/3 flows.
 *  [P3] "第 7 讲：Parallelism（上）" (CS336 lecture 7): memory table (16 bytes per
 *       parameter), Ring AllReduce = ReduceScatter + AllGather, ZeRO stage memory
 *       formulas, gradient accumulation, torch.optim.AdamW in the DDP loop.
 *
 * Conventions for every call:
 *  - Device pointers point into memory the caller owns (allocated with
 *    cudaMalloc, torch, ...) on the current device. They must be 16-byte aligned.
 *    Host arrays of device pointers (grads, replicas) are read during the call only.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *    stream-ordered and asynchronous unless a report is requested.
 *  - The steps of one plan (zr_step, zr_step_bucket, zr_step_inplace, zr_step_from_host,
 *    zr_offload_step) share its device control block: order them on one stream, or with
 *    events. Plans are independent of each other. Host calls on one plan from several
 *    threads at once are not supported.
 *  - Errors are returned as zr_status; no exception crosses the ABI. A failed call
 *    launches nothing. zr_last_error() returns a thread-local message for the last
 *    failure on the calling thread. An asynchronous CUDA error from an earlier
 *    launch surfaces as ZR_ERR_CUDA on a later call that synchronises.
 *  - Overflow (a non-finite reduced gradient) is not an error: it is reported
 *    through the overflow flag / step report, and the update is skipped.
 *  - 16-bit formats are IEEE binary16 (ZR_F16) and bfloat16 (ZR_BF16); fp32
 *    arithmetic is round-to-nearest-even with no fused multiply-add, in the op
 *    order documented at each call.
 */
#ifndef ZR_H
#define ZR_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ZR_OK = 0,
    ZR_ERR_INVALID = 1,     /* bad argument: null/misaligned pointer, size, W, stage, dtype */
    ZR_ERR_UNSUPPORTED = 2, /* valid request the library does not handle */
    ZR_ERR_CUDA = 3,        /* a CUDA runtime call failed */
    ZR_ERR_OOM = 4,         /* the library could not allocate its own small buffers */
    ZR_ERR_TIMEOUT = 5      /* reserved: no call waits on the device without a bound */
} zr_status;

typedef enum { ZR_F16 = 0, ZR_BF16 = 1, ZR_F32 = 2 } zr_dtype;

#define ZR_MAX_W 64         /* workers per ring */
#define ZR_MAX_REPLICAS 256 /* W * A gradient replicas per fused step */
#define ZR_ALIGN 8          /* elements; every block and tensor starts on a multiple */

/* AdamW hyperparameters (fp32 values; see zr_adamw_shard_step for the formula). */
typedef struct { float lr, beta1, beta2, eps, weight_decay; } zr_adamw_hyper;

/* Dynamic loss scaling ([P2] 核心技术 (1),(3) name it; the rule is this library's
 * reading): a step with any non-finite reduced gradient is skipped; if `dynamic`,
 * the scale becomes max(scale*backoff, min_scale) on a skip and scale*growth after
 * growth_interval consecutive clean steps. With dynamic = 0 the scale never changes. */
typedef struct {
    float init_scale, backoff, growth, min_scale;
    int32_t growth_interval;
    int32_t dynamic;
} zr_scaler_cfg;

/* One gradient bucket in the flat buffer: elements [start, start+len), cut into W
 * blocks of `chunk` elements (the last blocks may be short or empty). */
typedef struct { int64_t start, len, chunk; } zr_bucket;

/* ------------------------------------------------------------------------- */
/* Layout                                                                     */
/* ------------------------------------------------------------------------- */

/* Elements per ring block of an n-element bucket: align * ceil(n / (align * W))
 * ([P1] 二: each of the N blocks holds phi/N; [P3] Ring AllReduce, 阶段一). */
int64_t zr_chunk_size(int64_t n, int W, int align);

/* Reverse-order bucket builder ([P1] 二: parameters in reverse definition order,
 * output layer first, synchronised a full bucket at a time; [P3] DDP 核心实现细节).
 * numels[ntensors]: tensor sizes in definition order (host). Tensors are placed from
 * the last defined to the first, each at a multiple of `align` elements; a tensor is
 * never split; a non-empty bucket closes before a tensor that would take it past
 * cap_elems, so a tensor larger than the cap sits alone. Buckets are contiguous.
 * out: caller array of at least ntensors entries (host); *nbuckets: count written;
 * tensor_offsets[ntensors]: flat offset of each tensor (host, may be NULL). The gaps
 * that align tensors are elements of the flat arrays like any other: the ring sums,
 * the overflow flag and the update cover them, so a caller keeps them finite in its
 * gradient buffers (zero, as a zero-initialised buffer leaves them).
 * Errors: ZR_ERR_INVALID for null out/nbuckets, ntensors < 0, a negative numel,
 * cap_elems < 1, W outside [1, ZR_MAX_W], align < 1. */
zr_status zr_bucket_plan(const int64_t* numels, int ntensors, int64_t cap_elems, int W, int align,
                         zr_bucket* out, int* nbuckets, int64_t* tensor_offsets);

/* ------------------------------------------------------------------------- */
/* Standalone collectives and optimizer (the unfused chain)                    */
/* ------------------------------------------------------------------------- */

/* Ring reduce-scatter of one n-element bucket over W workers ([P1] 二 scatter reduce,
 * GPU0/GPU1/GPU2 example; [P3] Ring AllReduce 阶段一).
 * grads[W]: host array of device pointers, worker w's n gradients of type dt (F16,
 * BF16, or F32 for micro-batch sums from zr_accumulate). order[W]: host array,
 * order[p] = worker at ring position p (NULL = identity).
 * With C = zr_chunk_size(n, W, ZR_ALIGN), block c = [c*C, min((c+1)*C, n)) starts at
 * position c and travels the ring; the result is
 *     sums[i] = (((x_{order[c]}[i] + x_{order[c+1]}[i]) + ...) + x_{order[c+W-1]}[i])
 * (positions mod W, each value converted exactly to fp32, fp32 adds left to right),
 * which ring position (c-1) mod W owns. sums: device, n fp32 (the owners' shards in
 * place). overflow: device int32, set to 1 (never cleared) if any sum is not finite.
 * Errors: ZR_ERR_INVALID for n < 0, W outside [1, ZR_MAX_W], a bad order
 * permutation, null or misaligned pointers, dt not F16/BF16/F32. n == 0 is a no-op. */
zr_status zr_reduce_scatter(const void* const* grads, zr_dtype dt, int64_t n, int W, const int* order,
                            float* sums, int32_t* overflow, void* stream);

/* Ring all-reduce of one n-element bucket over W workers, as DDP runs it on the
 * gradients ([P1] 二: the scatter reduce, then the all-gather phase, after which every
 * GPU holds every reduced block; [P3] Ring AllReduce = ReduceScatter + AllGather). Every
 * worker ends with the sums zr_reduce_scatter defines, so the W copies are identical:
 * out[R] is a host array of R device fp32[n] outputs (the workers' copies; R in
 * [1, ZR_MAX_REPLICAS], typically 1..W), each written in full. The all-gather hops add
 * nothing: their traffic is zr_ring_traffic's second phase, counted, not moved.
 * grads, dt, n, W, order, overflow: as zr_reduce_scatter.
 * Errors: as zr_reduce_scatter, plus R outside [1, ZR_MAX_REPLICAS] and null or
 * misaligned outputs. n == 0 is a no-op. */
zr_status zr_all_reduce(const void* const* grads, zr_dtype dt, int64_t n, int W, const int* order,
                        float* const* out, int R, int32_t* overflow, void* stream);

/* One micro-batch of gradient accumulation on one worker ([P3] Gradient Accumulation:
 * micro-batch gradients add up locally, with the synchronisation skipped, before the
 * one reduction of the step): acc[i] = fp32(grad[i]) if `first`, else
 * acc[i] = acc[i] + fp32(grad[i]) (one fp32 add, round to nearest even).
 * grad: device, n values of type dt (F16 or BF16); acc: device fp32[n].
 * Calling it for micro-batches 0..A-1 in order and then zr_reduce_scatter / zr_step
 * on the fp32 accumulators gives the same bits as the fused A-way step.
 * Errors: ZR_ERR_INVALID for n < 0, dt not F16/BF16, null or misaligned pointers. */
zr_status zr_accumulate(const void* grad, zr_dtype dt, float* acc, int64_t n, int first, void* stream);

/* Owner-side update of one shard ([P1] 三: average, convert to FP32 and scale, update
 * m and v, then the FP32 master; [P3] memory table: master, m, v in FP32).
 * Runs two kernels: a pass that sets *overflow to 1 if any shard_sums value is not
 * finite, then, only if *overflow is 0 (read on the device), the AdamW update in place:
 *   g = sums * r,  r = fp32(1 / (loss_scale * W)) formed in double
 *   m = b1*m + (1-b1)*g ;  v = b2*v + (1-b2)*(g*g)
 *   u = (m / bc1) / (sqrt(v / bc2) + eps),  bc_i = fp32(1 - beta_i^t), beta_i^t a
 *       running product of t double multiplications (walked on the host only until it
 *       stops changing, which for 0 <= beta < 1 it does within about 745/(1-beta) steps)
 *   master = master*(1 - lr*wd) - lr*u     (1-b1, 1-b2, 1-lr*wd formed in fp32)
 * t: the 1-based index of this update. All arrays: device fp32, len elements.
 * Errors: ZR_ERR_INVALID for len < 0, t < 1, W < 1, loss_scale <= 0 or not finite,
 * betas outside [0, 1), null h, null or misaligned pointers. len == 0 only runs nothing. */
zr_status zr_adamw_shard_step(const float* shard_sums, float* m, float* v, float* master, int64_t len,
                              const zr_adamw_hyper* h, float loss_scale, int W, int64_t t,
                              int32_t* overflow, void* stream);

/* All-gather of the updated parameters ([P1] 二 all-gather phase and 三 parameter
 * broadcast; [P3] ZeRO stage 1 step 4): every worker ends with every block, so each of
 * the n_replicas outputs receives round-to-nearest-even out_dt(master[i]) for all i.
 * master: device fp32[n]; replicas: host array of n_replicas device pointers of n
 * out_dt values. The ring hop schedule is traffic only (zr_ring_traffic).
 * Errors: ZR_ERR_INVALID for n < 0, n_replicas outside [1, ZR_MAX_REPLICAS],
 * out_dt not F16/BF16, null or misaligned pointers. */
zr_status zr_all_gather(const float* master, int64_t n, zr_dtype out_dt, void* const* replicas, int n_replicas,
                        void* stream);

/* ------------------------------------------------------------------------- */
/* The fused step                                                              */
/* ------------------------------------------------------------------------- */

typedef struct zr_plan zr_plan;

typedef struct {
    int32_t W;                /* workers, 1..ZR_MAX_W */
    int32_t A;                /* micro-batches per worker, W*A <= ZR_MAX_REPLICAS */
    zr_dtype dtype;           /* gradient and parameter type: ZR_F16 or ZR_BF16 */
    int32_t stage;            /* 0 = DDP, or ZeRO stage 1, 2 or 3 (memory plan; same arithmetic) */
    int32_t align;            /* tensor alignment in elements; must be ZR_ALIGN */
    int64_t cap;              /* bucket cap in elements */
    int32_t ntensors;
    const int64_t* numels;    /* host, definition order */
    const int32_t* order;     /* host [W] ring order, NULL = identity */
    zr_scaler_cfg scaler;
    int32_t fp32_grads;       /* 1: the gradient replicas are fp32 (e.g. micro-batch sums built with
                                 zr_accumulate, [P3] Gradient Accumulation); 0: they have `dtype` */
} zr_plan_desc;

/* Optimizer state and parameter replica, two sets (ping-pong), in the flat layout of
 * zr_plan_numel elements. Set k (k = the plan's current index, 0 after create/reset)
 * holds the live values; a step reads set k and writes set 1-k, and the index flips
 * only if the step was clean, so a skipped step leaves set k bit-unchanged.
 * All device pointers; param is of the plan's dtype. */
typedef struct {
    float* master[2];
    float* m[2];
    float* v[2];
    void* param[2];
} zr_state;

typedef struct {
    int32_t overflow;      /* the last step saw a non-finite reduced gradient */
    int32_t skipped;       /* ... and was therefore skipped */
    int32_t current;       /* index of the live state set after the last step */
    int32_t stage;
    float scale_used;      /* loss scale of the last step */
    float scale;           /* loss scale for the next step */
    int64_t t;             /* committed AdamW updates */
    int64_t steps;         /* steps run, skipped included */
    int64_t skipped_total;
    int64_t good;          /* clean steps since the last scale change */
    int64_t n_real;        /* parameters (sum of numels) */
    int64_t bytes_alg;     /* algorithmic HBM bytes of one zr_step: (2*W*A + 26) * n_real
                              (16-bit gradients; zr_step_inplace adds 2*W*A * n_real) */
} zr_step_report;

/* Builds the bucket table, the tile schedule and the device control block.
 * *out receives the plan (free with zr_plan_destroy). The control block starts with
 * k = 0, t = 0, scale = scaler.init_scale.
 * Errors: ZR_ERR_INVALID (see zr_plan_desc), ZR_ERR_OOM, ZR_ERR_CUDA. */
zr_status zr_plan_create(const zr_plan_desc* d, zr_plan** out);
zr_status zr_plan_destroy(zr_plan* p);
int64_t zr_plan_numel(const zr_plan* p);          /* flat elements per replica and state array */
int32_t zr_plan_nbuckets(const zr_plan* p);
/* Copies the bucket table (nbuckets entries) and tensor offsets (ntensors) to host arrays. */
zr_status zr_plan_buckets(const zr_plan* p, zr_bucket* buckets, int64_t* tensor_offsets);
/* Resets the control block (k = 0, t = 0, scale) on `stream`. */
zr_status zr_plan_reset(zr_plan* p, void* stream);

/* One fused step, one kernel launch: for every element of every bucket, the ring-order
 * fp32 sum of the W workers' values, each worker's value being the fp32 sum of its A
 * micro-batch gradients in micro-batch order ([P3] Gradient Accumulation); then the
 * unscale and mean, the overflow flag, AdamW and the 16-bit cast exactly as
 * zr_reduce_scatter + zr_adamw_shard_step + zr_all_gather, reading state set k and
 * writing set 1-k. The last block to finish ORs all flags and applies the loss-scale
 * rule; on a clean step it sets t += 1 and k = 1-k ([P2] 核心技术 (3) dynamic scaling).
 * stage is 0, 1, 2 or 3 ([P3] ZeRO stages; [P2] (11)-(13)): stage 0 is DDP ([P1] 二:
 * the gradients are ring-all-reduced and every worker runs the same update on the full
 * gradient and keeps everything), stages 1-3 shard the optimizer state, the gradients
 * and the parameters. They share this arithmetic (every worker's update of an element
 * gives the owner's bits) and differ in what a real worker keeps resident.
 * grads[W*A]: host array of device pointers; replica w*A + a is worker w's micro-batch
 * a, zr_plan_numel elements of the plan's dtype. rep: NULL for a fully asynchronous
 * call; otherwise the call synchronises `stream` and fills *rep. A plan whose tensors
 * are all empty (zr_plan_numel 0) reduces nothing: its step is clean (one block runs the
 * rule above), and its array pointers may be null; the same holds for zr_step_inplace,
 * the from-host variants and zr_offload_step, and for zr_step_noalloc over buckets with
 * no elements.
 * Errors: ZR_ERR_INVALID for a null plan/state/hyper, stage outside 0..3, null or
 * misaligned pointers, aliasing of the two state sets; ZR_ERR_CUDA. */
zr_status zr_step(zr_plan* p, int stage, const void* const* grads, const zr_state* st,
                  const zr_adamw_hyper* h, void* stream, zr_step_report* rep);

/* As zr_step, with the gradients in HOST memory, and the report read back (rep is
 * required). If every host_grads[r] is page-locked memory the device can address
 * (cudaHostAlloc, cudaHostRegister; torch's pin_memory), the step kernel reads it in
 * place over the host link, so each gradient byte crosses the link once while the HBM
 * half of the step overlaps the transfer; dev_grads is then not used (may hold NULLs).
 * Otherwise each host_grads[r] is copied into the device buffer dev_grads[r] with one
 * cudaMemcpyAsync per replica and bucket, in bucket order, before the step. */
zr_status zr_step_from_host(zr_plan* p, int stage, const void* const* host_grads, void* const* dev_grads,
                            const zr_state* st, const zr_adamw_hyper* h, void* stream, zr_step_report* rep);

/* One bucket of a step, for overlap with backward ([P1] 二: a bucket is synchronised as
 * soon as all its gradients exist, while the GPU keeps computing the others; [P3] DDP
 * Gradient Bucketing and Overlap). Call it once for every bucket b = 0 .. nbuckets-1,
 * in that order (bucket 0 holds the output-side layers, whose gradients come first),
 * each launch ordered after the one before (one stream, or events), typically as bucket
 * b's gradients become ready. The launches together compute exactly what one zr_step
 * computes: the last block of the last launch takes the overflow decision for the whole
 * step and commits. A step must launch every bucket exactly once; after an incomplete
 * step, call zr_plan_reset. Same arguments and errors as zr_step, plus ZR_ERR_INVALID
 * for a bucket index outside [0, nbuckets). */
zr_status zr_step_bucket(zr_plan* p, int stage, int bucket, const void* const* grads, const zr_state* st,
                         const zr_adamw_hyper* h, void* stream);

/* How many thread blocks each zr_step_bucket launch of plan p may take, so that buckets
 * stepped while backward is still running leave the other SMs to it (the pages' overlap
 * moves gradients over links driven by a few SMs while the rest compute: [P1] 二, [P3]
 * Overlap). max_blocks = 0, the default, gives each launch one block per tile (every
 * block that fits at once for a small bucket); max_blocks > 0 caps each launch at that
 * many blocks, which then stride over the bucket's tiles. The results are the same bytes
 * for every value; only the launch shape changes. Call it between steps, never while a
 * step's bucket launches are in flight (the step's last block is found by counting the
 * blocks of all its launches). Errors: ZR_ERR_INVALID for a null plan or max_blocks < 0. */
zr_status zr_plan_set_bucket_blocks(zr_plan* p, int max_blocks);

/* How zr_step moves a tile's inputs into the SMs (a launch setting; the pages have no
 * counterpart: their step runs in NCCL and the optimizer). ZR_STAGING_REGISTERS: every thread
 * issues its 16-byte loads of the W replicas and of master/m/v into registers before any
 * arithmetic. ZR_STAGING_BULK: a producer warp per block copies each stage of a tile
 * (stage_elems elements of the W replicas and of master/m/v) into shared memory with
 * one-dimensional bulk copies (cp.async.bulk, this GPU's memory only) completed on mbarriers,
 * keeping `stages` stages in flight, and eight consumer warps compute from shared memory.
 * Both give the same bytes; only speed differs. Bulk staging covers zr_step (and its CUDA
 * graph capture) for plans with 16-bit gradients and any W and A: with W*A <= 8 a stage
 * holds all W*A replica slices of its elements; with more, the slices of a range of
 * elements follow one another in stages of 8 slices (at most 2048 elements each), the
 * consumers carrying their running sums from one stage to the next in the same order.
 * It is what zr_plan_create chooses when the automatic shape keeps stages of 2048
 * elements with all slices in one stage (W*A <= 8) and the plan has at least four waves
 * of tiles (a plan that streams from HBM); other plans, and the other calls, use register
 * staging (with W*A > 8 it measured as fast or faster).
 * stage_elems = 0 and stages = 0 choose a shape that lets two blocks share an SM. Call it
 * between steps; a CUDA graph captured earlier keeps the kernel it captured.
 * Every wait of a bulk-staged step is bounded (2 s); one that gives up skips the step and
 * makes zr_plan_report (and zr_step with a report) return ZR_ERR_TIMEOUT until
 * zr_plan_reset. Errors: ZR_ERR_INVALID (null plan, unknown staging, stage_elems not 0 or a
 * multiple of 8 up to 65536, or up to 2048 for ZR_STAGING_BULK with W*A > 8, stages above
 * 4), ZR_ERR_UNSUPPORTED (fp32 gradients, a shape that does not fit an SM's shared memory),
 * ZR_ERR_CUDA.
 * ZR_STAGING_BULK_IO: as ZR_STAGING_BULK (every slice of its elements in one stage, for any
 * W*A), and the results go out the same way: the consumers write each stage's new
 * master/m/v and 16-bit parameter back into its shared-memory slots and a storer warp
 * copies them to state set 1-k with bulk copies (shared to global). */
typedef enum { ZR_STAGING_REGISTERS = 0, ZR_STAGING_BULK = 1, ZR_STAGING_BULK_IO = 2 } zr_staging;
zr_status zr_plan_set_staging(zr_plan* p, int staging, int stage_elems, int stages);
/* The staging zr_step uses for plan p (a zr_staging value); -1 for a null plan. */
int zr_plan_staging(const zr_plan* p);

/* Test hook for the bounded waits of bulk staging; never needed in use. While on != 0,
 * every stage of a bulk-staged zr_step announces 16 bytes more on its mbarrier than its
 * copies deliver, so no stage completes: every wait runs out after its 2 s limit (no fault,
 * no trap, no endless wait; the copies themselves land), the step is skipped with the state
 * unchanged and zr_plan_report returns ZR_ERR_TIMEOUT until zr_plan_reset. Lets a test check
 * that a timed-out step reports its error and leaves the CUDA context usable. Errors:
 * ZR_ERR_INVALID for a null plan. */
zr_status zr_plan_stall_bulk_waits(zr_plan* p, int on);

/* The optimizer state and the parameter replica as ONE set (zr_step_inplace). Device
 * pointers, zr_plan_numel elements each; param is of the plan's dtype. */
typedef struct {
    float* master;
    float* m;
    float* v;
    void* param;
} zr_state1;

/* The fused step on one state set, updated in place, for runs whose HBM has no room for
 * zr_state's second set: it saves 14 bytes per parameter (12 of fp32 master/m/v, 2 of the
 * 16-bit replica), e.g. 98 GB for a 7B-parameter model. Same arithmetic, overflow rule
 * and loss-scale rule as zr_step ([P1] 三 ZeRO-1; [P2] 核心技术 (3) dynamic scaling).
 * The skip decision covers the whole step and must be known before any state is
 * overwritten, so the call makes two launches on `stream`:
 *   1. a flag pass over every bucket: the same ring-order fp32 sums as the update, kept
 *      only for their non-finite flag (reads 2*W*A bytes per parameter; 4*W*A for fp32
 *      gradients);
 *   2. the update: if the flag is set nothing is written, so the set stays bit-unchanged;
 *      otherwise master/m/v/param are read and rewritten in place. Its last block applies
 *      the loss-scale rule and counts the step.
 * Algorithmic bytes per parameter: 4*W*A + 26 for 16-bit gradients. The control block's
 * current index is neither used nor changed (after ping-pong steps on the same plan,
 * pass the live set). Both launches can be captured in a CUDA graph. There is no
 * bucket-by-bucket form (zr_step_bucket): no bucket may be updated before the flag of
 * the last one is known.
 * rep: NULL for an asynchronous call, else the call synchronises `stream` and fills it.
 * Errors: ZR_ERR_INVALID for a null plan/state/hyper/grads, stage outside 0..3, a null or
 * misaligned array; ZR_ERR_CUDA. */
zr_status zr_step_inplace(zr_plan* p, int stage, const void* const* grads, const zr_state1* st,
                          const zr_adamw_hyper* h, void* stream, zr_step_report* rep);

/* As zr_step_inplace, with the gradients in HOST memory, and the report read back (rep
 * is required): each host_grads[r] is copied into the device buffer dev_grads[r]
 * (zr_plan_numel elements of the gradient type) with one cudaMemcpyAsync per replica and
 * bucket, in bucket order, on `stream`, then the in-place step runs on dev_grads. The
 * gradients always go through device memory here: the step reads them twice (flag pass,
 * then update), so reading page-locked host memory in place would cross the host link
 * twice. Errors: as zr_step_inplace, plus null host or device gradient pointers. */
zr_status zr_step_inplace_from_host(zr_plan* p, int stage, const void* const* host_grads, void* const* dev_grads,
                                    const zr_state1* st, const zr_adamw_hyper* h, void* stream,
                                    zr_step_report* rep);

/* Synchronises `stream` and reads the control block into *rep. */
zr_status zr_plan_report(zr_plan* p, void* stream, zr_step_report* rep);

/* Checkpoint / resume of a plan's step state (the pages name checkpoints among the
 * runtime's duties, [P2] 2 (1) ②, without a mechanism). The optimizer state and the
 * replica live in caller buffers, which the caller saves itself (the live set is
 * `current`); this record holds what the control block adds. Restoring it into a plan
 * with the same layout and continuing gives the same bytes as never stopping. */
typedef struct {
    int32_t current;       /* live state set */
    float scale;           /* loss scale for the next step */
    int64_t good, t, steps, skipped;
    double beta1_pow, beta2_pow; /* beta1^t, beta2^t as running products */
} zr_checkpoint;

/* Synchronises `stream` and copies the control block into *out. */
zr_status zr_plan_checkpoint(zr_plan* p, void* stream, zr_checkpoint* out);
/* Writes *in into the control block on `stream` and synchronises it.
 * Errors: ZR_ERR_INVALID for a null argument, current not 0/1, a scale that is not
 * positive and finite, negative counters, beta powers outside [0, 1]. */
zr_status zr_plan_restore(zr_plan* p, const zr_checkpoint* in, void* stream);

/* ------------------------------------------------------------------------- */
/* ZeRO-3 parameter shards and the all-gather before forward / backward        */
/* ------------------------------------------------------------------------- */

/* Under ZeRO-3 a worker keeps only its share of the 16-bit parameters and all-gathers
 * a layer's parameters from the others right before the layer's forward and again
 * before its backward, dropping them after use ([P1] 四 ZeRO-3: the missing
 * parameters are broadcast for forward and again for backward, then discarded;
 * [P2] (13) ②③; [P3] ZeRO Stage 3). Here worker w's shard is the packed
 * concatenation, in bucket order, of the block it owns in every bucket (the worker at
 * ring position p owns block (p+1) mod W), zr_plan_shard_numel(w) elements of the
 * plan's dtype. */
int64_t zr_plan_shard_numel(const zr_plan* p, int worker);
/* Where bucket `bucket`'s block starts in worker `worker`'s shard. */
zr_status zr_plan_shard_offset(const zr_plan* p, int bucket, int worker, int64_t* offset);

/* Copies each worker's owned blocks of the full replica (zr_plan_numel elements of the
 * plan's dtype, device) into its packed shard: what a ZeRO-3 worker keeps after the
 * step. shards[W]: host array of device pointers indexed by worker id.
 * Errors: ZR_ERR_INVALID for null or misaligned pointers; ZR_ERR_CUDA. */
zr_status zr_shard_params(zr_plan* p, const void* replica, void* const* shards, void* stream);

/* The ZeRO-3 parameter all-gather for buckets [bucket_lo, bucket_hi): every block of
 * those buckets is copied from its owner's shard into the (transient) replica at its
 * flat position; the rest of the replica is not touched. Moves 2 bytes in and 2 out
 * per parameter. Errors: ZR_ERR_INVALID for a bad range, null or misaligned
 * pointers; ZR_ERR_CUDA. */
zr_status zr_gather_params(zr_plan* p, int bucket_lo, int bucket_hi, const void* const* shards, void* replica,
                           void* stream);

/* ------------------------------------------------------------------------- */
/* ZeRO-Offload: the optimizer on the host CPU                                */
/* ------------------------------------------------------------------------- */

/* The owner-side update of zr_adamw_shard_step followed by the cast of zr_all_gather,
 * run on the host CPU over host memory ([P2] (16) ZeRO-Offload: the update, which
 * needs little compute, and the optimizer states move to the CPU, forward and
 * backward stay on the GPU; [P2] 总结: offloaded to the CPU side). Same arithmetic and
 * op order, so the same bits. sums, master, m, v: host fp32[n]; param16: host, n
 * values of dt (may be NULL to skip the cast); nthreads worker threads (1..256).
 * If any sums value is not finite, *overflow = 1 and nothing is written; otherwise
 * *overflow = 0. Errors: ZR_ERR_INVALID for bad sizes, null pointers, dt, t < 1,
 * W < 1, a bad loss_scale, betas outside [0, 1). */
zr_status zr_offload_adamw(const float* sums, float* master, float* m, float* v, void* param16, zr_dtype dt,
                           int64_t n, const zr_adamw_hyper* h, float loss_scale, int W, int64_t t, int nthreads,
                           int32_t* overflow);

/* One ZeRO-Offload step over a plan (A = 1; 16-bit or fp32 gradients): the ring
 * reduce-scatter of every bucket on the GPU into sums_dev (device fp32, plan numel),
 * the global overflow flag read back first (a skip writes nothing), then bucket by
 * bucket: the sums copied into sums_host (pinned host fp32), the update on the CPU of
 * the host-resident master/m/v (host fp32) into param_host (pinned host, plan dtype),
 * and the parameters copied into param_dev (device replica). The host update of bucket
 * b overlaps the copies of the other buckets. "Pinned" means page-locked: allocated by
 * cudaHostAlloc or registered with cudaHostRegister. The last parameter copies are
 * still queued on `stream` at return: synchronise it before reading param_dev or
 * reusing param_host. The caller applies its loss-scale rule from *overflow (host int32).
 * Errors: ZR_ERR_INVALID for null or misaligned buffers, stage, t < 1, betas outside
 * [0, 1); ZR_ERR_UNSUPPORTED for A > 1; ZR_ERR_CUDA. */
zr_status zr_offload_step(zr_plan* p, int stage, const void* const* grads, float* sums_dev, float* sums_host,
                          float* master, float* m, float* v, void* param_host, void* param_dev,
                          const zr_adamw_hyper* h, float loss_scale, int64_t t, int nthreads, void* stream,
                          int32_t* overflow);

/* ------------------------------------------------------------------------- */
/* Fused step without device allocation                                        */
/* ------------------------------------------------------------------------- */

/* Tile capacity of the static scratch used by zr_step_noalloc: 16 bytes per tile of at
 * most 32768 elements, i.e. 1 MiB of device memory per GPU, enough for about 2e9
 * elements when the ring blocks are long. */
#define ZR_NOALLOC_MAX_TILES 65536

/* The pages have no counterpart to this call; it exists for callers that cannot
 * allocate device memory. zr_plan_create allocates a tile table and a control block,
 * which a caller cannot accept if its runtime owns all device memory through its own
 * pool, if its memory budget was fixed before the first step, or if an allocation
 * would synchronise the device on its path. zr_step_noalloc computes exactly what
 * zr_step computes for one step, with the kernel zr_step would choose for these buckets
 * (bulk-copy staging, whose shared memory is a kernel attribute set on the current
 * device, or register staging), allocating nothing (no cudaMalloc, no cudaFree, no
 * allocating library routine): its scratch is one static device array of this library
 * (ZR_NOALLOC_MAX_TILES tiles plus a 256-byte control block), present on every GPU that loads
 * the library until the process exits.
 *
 * buckets[nbuckets]: host bucket table, e.g. from zr_bucket_plan (starts and lengths
 * multiples of ZR_ALIGN, chunk = zr_chunk_size(len, W, ZR_ALIGN)). grads[W*A]: host
 * array of device pointers, replica w*A + a, each covering every bucket. order: ring
 * order (NULL = identity). st/current: reads state set `current`, writes set
 * 1-current in full. loss_scale and t (1-based index of this update) as in
 * zr_adamw_shard_step; the bias corrections come from the same running products of the
 * betas that zr_step keeps (fp32(1 - beta^t), beta^t as t double multiplications), which
 * the library caches between calls, so stepping t = 1, 2, 3, ... costs one multiplication
 * per call and any t costs at most the walk to the products' fixed point. overflow:
 * device int32, set to 1 if any reduced gradient is not finite, else 0 (also 0 for an
 * empty bucket table); when it is 1 the written set must be discarded (keep `current`),
 * and the caller applies its own loss-scale rule. Under bulk-copy staging a wait that
 * gave up (each is bounded at 2 s; zr_step reports that as ZR_ERR_TIMEOUT) also sets
 * it to 1: nothing is lost, but this call cannot tell it from an overflow.
 * The caller carries the live-set index, the scale and t between calls.
 *
 * Every call on a device reuses the same scratch and leaves its last contents there;
 * the call rebuilds the tile schedule and clears the ticket and flag itself. Calls
 * whose kernels overlap on the GPU race on the scratch: order them on one stream (or
 * otherwise serialise them). The first call on a device looks up the scratch's device
 * address (cudaGetSymbolAddress); make it before any stream capture.
 * Errors: ZR_ERR_INVALID for the cases of zr_step, a bucket that breaks the ring rule,
 * current not 0/1, t < 1, a bad loss_scale, betas outside [0, 1), or buckets needing more than
 * ZR_NOALLOC_MAX_TILES tiles (use zr_plan_create/zr_step for those); ZR_ERR_CUDA. */
zr_status zr_step_noalloc(const zr_bucket* buckets, int nbuckets, int W, int A, zr_dtype dtype, const int* order,
                          const void* const* grads, const zr_state* st, int current, const zr_adamw_hyper* h,
                          float loss_scale, int64_t t, int32_t* overflow, void* stream);

/* ------------------------------------------------------------------------- */
/* Accounting                                                                 */
/* ------------------------------------------------------------------------- */

/* Model-state bytes per worker under mixed precision + Adam ([P3] memory table and
 * ZeRO formulas; [P1] 三/四 "2+2+K", K = 12): stage 0 (DDP) 16n; stage 1
 * 4n + 12n/W; stage 2 2n + 14n/W; stage 3 16n/W (integer division). -1 on bad input. */
int64_t zr_model_state_bytes(int stage, int64_t n, int W);

/* Elements each ring position sends and receives in one phase over an n-element
 * bucket ([P1] 二 traffic: (N-1) * phi / N per phase when N divides phi; [P3]
 * 通信量分析). Position p sends every block but (p+1) mod W in reduce-scatter and
 * every block but (p+2) mod W in all-gather; it receives every block but p, resp.
 * (p+1) mod W. Arrays are host [W]; any may be NULL. */
zr_status zr_ring_traffic(int64_t n, int W, int align, int64_t* rs_sent, int64_t* rs_recv, int64_t* ag_sent,
                          int64_t* ag_recv);

const char* zr_status_str(zr_status s);
const char* zr_last_error(void);
/* Library version string. */
const char* zr_version(void);

#ifdef __cplusplus
}
#endif
#endif
