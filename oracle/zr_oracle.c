/*
 * zr_oracle.c — TEST INFRASTRUCTURE: the CPU oracle of the post-backward ZeRO step.
 * Plain C99, single-threaded, built with -O2 -ffp-contract=off (no FMA contraction,
 * no fast-math) so that every float operation below is one IEEE-754 binary32
 * operation rounded to nearest even. See zr_oracle.h for sources and readings.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use it.
 */
#include "zr_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Layout                                                                     */
/* ------------------------------------------------------------------------- */

/* Elements per ring chunk of an n-element bucket. The ring splits a bucket into
 * W blocks ([P1] 二: each block holds phi/N of the parameters; [P3] Ring
 * AllReduce, 阶段一: the gradient vector is cut into W blocks). Reading: blocks are whole multiples of
 * `align` elements so that every block starts on a 16-byte boundary; the last
 * blocks take what is left (possibly nothing). */
int64_t zro_chunk_size(int64_t n, int W, int align) {
    if (n <= 0) return 0;
    int64_t unit = (int64_t)align * W;
    return ((n + unit - 1) / unit) * align;
}

static int64_t round_up(int64_t x, int64_t a) { return ((x + a - 1) / a) * a; }

/* Reverse-order bucketing ([P1] 二, DDP internals: parameters are arranged in the
 * reverse of their definition order, output layer first, and a bucket is
 * synchronised once it is full; [P3] DDP "Bucket 的构建顺序": buckets follow the
 * reverse of the backward computation order).
 * Reading: walk tensors from the last defined to the first; a tensor never
 * splits; a non-empty bucket closes before a tensor that would take it past
 * `cap` elements; a tensor larger than `cap` therefore sits alone. Each tensor
 * starts at a multiple of `align` elements (the gap, if any, belongs to the
 * bucket). Buckets are contiguous in the flat buffer, in creation order. */
int zro_bucket_plan(const int64_t* numels, int ntensors, int64_t cap, int W, int align,
                    zro_bucket* buckets, int* nbuckets, int64_t* tensor_offset) {
    if (ntensors < 0 || W < 1 || align < 1 || cap < 1) return -1;
    int nb = 0;
    int64_t flat = 0;       /* next free flat offset */
    int64_t cur_start = 0;  /* start of the open bucket */
    int64_t cur_len = 0;    /* aligned length of the open bucket */
    for (int t = ntensors - 1; t >= 0; --t) {
        if (numels[t] < 0) return -1;
        int64_t sz = round_up(numels[t], align);
        if (cur_len > 0 && cur_len + numels[t] > cap) {
            buckets[nb].start = cur_start;
            buckets[nb].len = cur_len;
            buckets[nb].chunk = zro_chunk_size(cur_len, W, align);
            ++nb;
            cur_start = flat;
            cur_len = 0;
        }
        tensor_offset[t] = flat;
        flat += sz;
        cur_len += sz;
    }
    if (cur_len > 0) {
        buckets[nb].start = cur_start;
        buckets[nb].len = cur_len;
        buckets[nb].chunk = zro_chunk_size(cur_len, W, align);
        ++nb;
    }
    *nbuckets = nb;
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Number formats ([P2] 核心技术 (2): FP16 has a 5-bit exponent and 10-bit      */
/* mantissa, BF16 the FP32 exponent range with 7 mantissa bits). Written from   */
/* the IEEE-754 definitions: value = (-1)^s * 2^(e - bias) * (1.f), or the      */
/* subnormal form; conversion from fp32 rounds to the nearest representable     */
/* value, ties to an even last bit.                                             */
/* ------------------------------------------------------------------------- */

static float decode16(uint16_t h, int ebits, int mbits) {
    int bias = (1 << (ebits - 1)) - 1;
    int s = (h >> 15) & 1;
    int e = (h >> mbits) & ((1 << ebits) - 1);
    int f = h & ((1 << mbits) - 1);
    float mag;
    if (e == (1 << ebits) - 1) {
        mag = f ? NAN : INFINITY;
    } else if (e == 0) {
        mag = ldexpf((float)f, 1 - bias - mbits);           /* subnormal */
    } else {
        mag = ldexpf((float)((1 << mbits) | f), e - bias - mbits);
    }
    return s ? -mag : mag;
}

/* Round |x| to the format's grid: the representable values near |x| are the
 * multiples of the quantum 2^q, q = max(exp(|x|) - mbits, emin - mbits), with
 * exp(|x|) = floor(log2|x|). nearbyint rounds ties to even in the default mode.
 * Then encode the rounded magnitude. */
static uint16_t encode16(float x, int ebits, int mbits) {
    int bias = (1 << (ebits - 1)) - 1;
    int emax = bias;            /* largest unbiased exponent of a finite value */
    int emin = 1 - bias;        /* smallest normal exponent */
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    uint16_t inf = (uint16_t)(((1 << ebits) - 1) << mbits);
    if (isnan(x)) return (uint16_t)(sign | inf | (1 << (mbits - 1)));
    double a = fabs((double)x);
    if (isinf(x)) return (uint16_t)(sign | inf);
    if (a == 0.0) return sign;
    int ex;
    frexp(a, &ex);                              /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                             /* floor(log2 a) */
    int q = (e > emin ? e : emin) - mbits;
    double k = nearbyint(ldexp(a, -q));         /* integer multiple of 2^q, ties to even */
    double r = ldexp(k, q);                     /* rounded magnitude */
    double maxfin = ldexp((double)((1 << (mbits + 1)) - 1), emax - mbits);
    if (r > maxfin) return (uint16_t)(sign | inf);
    if (r == 0.0) return sign;                  /* rounded down to a signed zero */
    /* encode r */
    int rex;
    frexp(r, &rex);
    int re = rex - 1;
    if (re < emin) {                            /* subnormal: r = f * 2^(emin - mbits) */
        int f = (int)ldexp(r, -(emin - mbits));
        return (uint16_t)(sign | f);
    }
    int f = (int)(ldexp(r, -(re - mbits)) - (double)(1 << mbits));
    return (uint16_t)(sign | ((re + bias) << mbits) | f);
}

float zro_f16_to_f32(uint16_t h) { return decode16(h, 5, 10); }
float zro_bf16_to_f32(uint16_t h) { return decode16(h, 8, 7); }
uint16_t zro_f32_to_f16(float x) { return encode16(x, 5, 10); }
uint16_t zro_f32_to_bf16(float x) { return encode16(x, 8, 7); }

void zro_decode(int dtype, const uint16_t* in, float* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = dtype == ZRO_F16 ? zro_f16_to_f32(in[i]) : zro_bf16_to_f32(in[i]);
}

void zro_encode(int dtype, const float* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = dtype == ZRO_F16 ? zro_f32_to_f16(in[i]) : zro_f32_to_bf16(in[i]);
}

/* One micro-batch of gradient accumulation on one worker ([P3] Gradient
 * Accumulation: the micro-batch gradients are summed locally, the synchronisation
 * skipped, before the one reduction): acc = fp32(g) for the first micro-batch, then
 * acc = acc + fp32(g), in micro-batch order. zro_step's S1 is this, A times. */
void zro_accumulate(int dtype, const uint16_t* g, float* acc, int64_t n, int first) {
    for (int64_t i = 0; i < n; ++i) {
        float x = dtype == ZRO_F16 ? zro_f16_to_f32(g[i]) : zro_bf16_to_f32(g[i]);
        acc[i] = first ? x : acc[i] + x;
    }
}

/* ------------------------------------------------------------------------- */
/* Ring collectives                                                           */
/* ------------------------------------------------------------------------- */

static int64_t chunk_lo(int64_t n, int64_t C, int c) { int64_t lo = (int64_t)c * C; return lo < n ? lo : n; }
static int64_t chunk_hi(int64_t n, int64_t C, int c) { int64_t hi = ((int64_t)c + 1) * C; return hi < n ? hi : n; }
static int mod(int a, int W) { int r = a % W; return r < 0 ? r + W : r; }

/* Ring reduce-scatter ("scatter reduce"), hop by hop ([P1] 二, the A/B/C
 * walk-through; [P3] Ring AllReduce, 阶段一). work[p] is ring position p's copy
 * of the bucket. In hop s = 0..W-2 every position p sends block (p - s) mod W to
 * its successor p+1, which adds the message to its own copy of that block. All
 * positions send at once, so the messages are taken before anyone adds. After
 * W-1 hops position p holds the full sum of block (p + 1) mod W, accumulated as
 * x_c + x_{c+1} + ... + x_{c+W-1} (positions mod W, left to right).
 * msg: scratch of W*C floats. sent/recv: per-position element counters.
 * The _hops form runs hops s0 .. s1-1 only, to look at the state between hops. */
void zro_ring_reduce_scatter_hops(int W, int64_t n, int64_t C, float* const* work, float* msg,
                                  int64_t* sent, int64_t* recv, int s0, int s1) {
    for (int s = s0; s < s1 && s <= W - 2; ++s) {
        for (int p = 0; p < W; ++p) {                     /* everyone sends */
            int c = mod(p - s, W);
            int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            memcpy(msg + (int64_t)p * C, work[p] + lo, (size_t)(hi - lo) * sizeof(float));
            sent[p] += hi - lo;
        }
        for (int p = 0; p < W; ++p) {                     /* successor adds */
            int dst = mod(p + 1, W);
            int c = mod(p - s, W);
            int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            const float* in = msg + (int64_t)p * C;
            float* own = work[dst] + lo;
            for (int64_t i = 0; i < hi - lo; ++i) own[i] = in[i] + own[i];
            recv[dst] += hi - lo;
        }
    }
}

void zro_ring_reduce_scatter(int W, int64_t n, int64_t C, float* const* work, float* msg,
                             int64_t* sent, int64_t* recv) {
    zro_ring_reduce_scatter_hops(W, n, C, work, msg, sent, recv, 0, W - 1);
}

/* Ring all-gather ([P1] 二, second phase: GPU0 first sends B, GPU1 C, GPU2 A,
 * then A, B, C; [P3] Ring AllReduce, 阶段二). rep[p] is position p's replica,
 * in which only block (p + 1) mod W is filled on entry. In hop s = 0..W-2
 * position p forwards block (p + 1 - s) mod W to p+1, which stores it. */
void zro_ring_all_gather_hops(int W, int64_t n, int64_t C, uint16_t* const* rep, uint16_t* msg,
                              int64_t* sent, int64_t* recv, int s0, int s1) {
    for (int s = s0; s < s1 && s <= W - 2; ++s) {
        for (int p = 0; p < W; ++p) {
            int c = mod(p + 1 - s, W);
            int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            memcpy(msg + (int64_t)p * C, rep[p] + lo, (size_t)(hi - lo) * sizeof(uint16_t));
            sent[p] += hi - lo;
        }
        for (int p = 0; p < W; ++p) {
            int dst = mod(p + 1, W);
            int c = mod(p + 1 - s, W);
            int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            memcpy(rep[dst] + lo, msg + (int64_t)p * C, (size_t)(hi - lo) * sizeof(uint16_t));
            recv[dst] += hi - lo;
        }
    }
}

void zro_ring_all_gather(int W, int64_t n, int64_t C, uint16_t* const* rep, uint16_t* msg,
                         int64_t* sent, int64_t* recv) {
    zro_ring_all_gather_hops(W, n, C, rep, msg, sent, recv, 0, W - 1);
}

/* Ring all-reduce, as DDP runs it on the gradients ([P1] 二: after the scatter-reduce
 * hops comes the all-gather phase, at the end of which every GPU holds every reduced
 * block; [P3] Ring AllReduce = ReduceScatter + AllGather). work[p] as in
 * zro_ring_reduce_scatter; the reduce-scatter hops run first, then in all-gather hop
 * s = 0..W-2 every position p sends its copy of block (p + 1 - s) mod W, already fully
 * reduced, to p+1, which stores it. Afterwards every work[p] holds every block's sum.
 * msg: scratch of W*C floats; sent/recv count both phases. */
void zro_ring_all_reduce(int W, int64_t n, int64_t C, float* const* work, float* msg,
                         int64_t* sent, int64_t* recv) {
    zro_ring_reduce_scatter_hops(W, n, C, work, msg, sent, recv, 0, W - 1);
    for (int s = 0; s <= W - 2; ++s) {
        for (int p = 0; p < W; ++p) {
            int c = mod(p + 1 - s, W);
            int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            memcpy(msg + (int64_t)p * C, work[p] + lo, (size_t)(hi - lo) * sizeof(float));
            sent[p] += hi - lo;
        }
        for (int p = 0; p < W; ++p) {
            int dst = mod(p + 1, W);
            int c = mod(p + 1 - s, W);
            int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            memcpy(work[dst] + lo, msg + (int64_t)p * C, (size_t)(hi - lo) * sizeof(float));
            recv[dst] += hi - lo;
        }
    }
}

/* ZeRO-3 keeps on each worker only its share of the 16-bit parameters ([P1] 四:
 * parameters are partitioned too; [P3] ZeRO Stage 3: each GPU stores 1/W of them).
 * Reading: the worker at ring position p keeps the block it owns after the
 * reduce-scatter, (p+1) mod W, of every bucket, packed in bucket order.
 * shards[w] is indexed by worker id. */
void zro_shard_params(int W, const int* order, int nbuckets, const zro_bucket* buckets, const uint16_t* replica,
                      uint16_t* const* shards) {
    int64_t fill[ZRO_MAX_W] = {0};
    for (int b = 0; b < nbuckets; ++b) {
        const int64_t st = buckets[b].start, n = buckets[b].len, C = buckets[b].chunk;
        for (int p = 0; p < W; ++p) {
            const int w = order ? order[p] : p;
            const int c = mod(p + 1, W);
            const int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            memcpy(shards[w] + fill[w], replica + st + lo, (size_t)(hi - lo) * sizeof(uint16_t));
            fill[w] += hi - lo;
        }
    }
}

/* The parameter all-gather that ZeRO-3 runs before a layer's forward and again before
 * its backward ([P1] 四; [P2] (13) ②③): for each bucket in [b_lo, b_hi), every
 * position starts with its own block taken from its shard, the W-1 ring all-gather
 * hops run, all W replicas must agree, and the result is written to `replica` at the
 * bucket's flat position. Returns 0, -2 on allocation failure, -3 on disagreement. */
int zro_param_all_gather(int W, const int* order, int nbuckets, const zro_bucket* buckets, int b_lo, int b_hi,
                         const uint16_t* const* shards, uint16_t* replica) {
    int64_t maxlen = 0, maxC = 0;
    for (int b = 0; b < nbuckets; ++b) {
        if (buckets[b].len > maxlen) maxlen = buckets[b].len;
        if (buckets[b].chunk > maxC) maxC = buckets[b].chunk;
    }
    uint16_t* rep[ZRO_MAX_W];
    uint16_t* msg = (uint16_t*)malloc((size_t)(W * (maxC ? maxC : 1)) * sizeof(uint16_t));
    int rc = msg ? 0 : -2;
    for (int p = 0; p < W; ++p) {
        rep[p] = (uint16_t*)calloc((size_t)(maxlen ? maxlen : 1), sizeof(uint16_t));
        if (!rep[p]) rc = -2;
    }
    int64_t off[ZRO_MAX_W] = {0};  /* running offset of each worker's shard, by worker id */
    for (int b = 0; b < nbuckets && rc == 0; ++b) {
        const int64_t st = buckets[b].start, n = buckets[b].len, C = buckets[b].chunk;
        for (int p = 0; p < W; ++p) {
            const int w = order ? order[p] : p;
            const int c = mod(p + 1, W);
            const int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            if (b >= b_lo && b < b_hi) {
                memset(rep[p], 0, (size_t)n * sizeof(uint16_t));
                memcpy(rep[p] + lo, shards[w] + off[w], (size_t)(hi - lo) * sizeof(uint16_t));
            }
            off[w] += hi - lo;
        }
        if (b < b_lo || b >= b_hi) continue;
        int64_t sent[ZRO_MAX_W] = {0}, recv[ZRO_MAX_W] = {0};
        zro_ring_all_gather(W, n, C, rep, msg, sent, recv);
        for (int p = 1; p < W; ++p)
            if (memcmp(rep[p], rep[0], (size_t)n * sizeof(uint16_t)) != 0) rc = -3;
        memcpy(replica + st, rep[0], (size_t)n * sizeof(uint16_t));
    }
    for (int p = 0; p < W; ++p) free(rep[p]);
    free(msg);
    return rc;
}

/* Per-position traffic of one ring phase over an n-element bucket, by running
 * the hop schedule on block sizes only. */
void zro_ring_traffic(int64_t n, int W, int align, int64_t* sent_per_pos, int64_t* recv_per_pos) {
    int64_t C = zro_chunk_size(n, W, align);
    for (int p = 0; p < W; ++p) { sent_per_pos[p] = 0; recv_per_pos[p] = 0; }
    for (int s = 0; s <= W - 2; ++s)
        for (int p = 0; p < W; ++p) {
            int c = mod(p - s, W);
            int64_t k = chunk_hi(n, C, c) - chunk_lo(n, C, c);
            sent_per_pos[p] += k;
            recv_per_pos[mod(p + 1, W)] += k;
        }
}

/* ------------------------------------------------------------------------- */
/* Unscale and AdamW                                                          */
/* ------------------------------------------------------------------------- */

/* The reduced value is a sum over W workers of gradients scaled by S. The update
 * uses their mean ([P1] 三: the owner computes the mean of the gradients;
 * [P3] 数学等价性: g = (1/W) sum g_k) with the loss scale removed ([P1] 三: the
 * owner's gradients go to FP32 and are scaled before m and v). Reading: one fp32 factor 1/(S*W), formed in
 * double and rounded once. */
float zro_unscale_factor(float scale, int W) { return (float)(1.0 / ((double)scale * (double)W)); }

/* fp32(1 - beta^t), beta^t as a running product of t double multiplications. */
float zro_bias_correction(float beta, int64_t t) {
    double prod = 1.0;
    for (int64_t i = 0; i < t; ++i) prod *= (double)beta;
    return (float)(1.0 - prod);
}

/* AdamW with decoupled weight decay (Loshchilov & Hutter, "Decoupled Weight
 * Decay Regularization"), the optimizer the pages run (torch.optim.AdamW in
 * [P3]'s DDP loop) on fp32 master, m and v ([P1] 三: update m and v, then the
 * FP32 master; [P3] memory table: master, m, v in FP32). Reading of the op order
 * (every operation one fp32 rounding):
 *   m <- b1*m + (1-b1)*g ;  v <- b2*v + (1-b2)*(g*g)
 *   u <- (m / bc1) / (sqrt(v / bc2) + eps)
 *   p <- p*(1 - lr*wd) - lr*u                                              */
void zro_adamw(int64_t len, const float* g, float* p, float* m, float* v,
               const zro_hyper* h, float bc1, float bc2) {
    const float b1 = h->beta1, b2 = h->beta2, lr = h->lr, eps = h->eps;
    const float omb1 = 1.0f - b1;
    const float omb2 = 1.0f - b2;
    const float lrwd = lr * h->weight_decay;
    const float decay = 1.0f - lrwd;
    for (int64_t i = 0; i < len; ++i) {
        float gi = g[i];
        float t1 = b1 * m[i];
        float t2 = omb1 * gi;
        float mi = t1 + t2;
        float gg = gi * gi;
        float t3 = b2 * v[i];
        float t4 = omb2 * gg;
        float vi = t3 + t4;
        float mhat = mi / bc1;
        float vhat = vi / bc2;
        float den = sqrtf(vhat) + eps;
        float u = mhat / den;
        float pd = p[i] * decay;
        float step = lr * u;
        m[i] = mi;
        v[i] = vi;
        p[i] = pd - step;
    }
}

/* ------------------------------------------------------------------------- */
/* One step                                                                   */
/* ------------------------------------------------------------------------- */

/* One post-backward step over every bucket:
 *  S1  per worker, fp32 sum of its A micro-batch gradients in micro-batch order
 *      ([P3] Gradient Accumulation: micro-batch gradients add up before the one
 *      synchronisation);
 *  S2  ring reduce-scatter, hop by hop, per bucket;
 *  S3  r = fp32(1/(S*W)); g = s*r on each owner's shard;
 *  S4  overflow flag = OR of !isfinite over all reduced values of all buckets; the
 *      step is skipped if it is set ([P2] 核心技术 (1),(3): dynamic loss scaling);
 *  S5  AdamW on each owner's shard (t+1), unless skipped;
 *  S6  cast the shard to the 16-bit format and ring all-gather it into W
 *      replicas, which must agree; the full replica is written to `param`.
 * Stage 1/2/3 change what each worker keeps resident, not these numbers
 * ([P3] ZeRO stages; [P2] (11)-(13)), so the stage is not an argument.
 *
 * grads[w*A + a]: flat 16-bit gradients of worker w, micro-batch a. order[p]:
 * worker at ring position p (NULL = identity). master/m/v/param: flat arrays,
 * updated only on the owners' shards and only when the step is not skipped.
 * flag_override: -1 computes the flag from these buckets; 0/1 imposes a global
 * flag computed elsewhere (for runs over a sample of the buckets), OR-ed with
 * the local one. sums_out (nullable): the reduced fp32 sums, flat.
 * With no buckets (a model without parameters) nothing is summed or flagged, so the
 * step is clean: t, the beta products and the good-step count advance as for any
 * clean step (the plain reading; the pages never meet this case).
 * Returns 0, or -1 on bad arguments, -2 on allocation failure, -3 if the
 * all-gathered replicas disagree. */
int zro_step(int W, int A, int dtype, const int* order, int nbuckets, const zro_bucket* buckets,
             const uint16_t* const* grads, float* master, float* m, float* v, uint16_t* param,
             const zro_hyper* h, zro_scaler* sc, int flag_override, float* sums_out, zro_report* rep) {
    if (W < 1 || W > ZRO_MAX_W || A < 1 || nbuckets < 0) return -1;
    int ord[ZRO_MAX_W];
    for (int p = 0; p < W; ++p) ord[p] = order ? order[p] : p;

    int64_t total = 0, maxlen = 0, maxC = 0;
    for (int b = 0; b < nbuckets; ++b) {
        int64_t end = buckets[b].start + buckets[b].len;
        if (end > total) total = end;
        if (buckets[b].len > maxlen) maxlen = buckets[b].len;
        if (buckets[b].chunk > maxC) maxC = buckets[b].chunk;
    }
    zro_report r;
    memset(&r, 0, sizeof r);
    r.scale_used = sc->scale;

    float* sums = sums_out ? sums_out : (float*)calloc((size_t)(total ? total : 1), sizeof(float));
    float** work = (float**)calloc((size_t)W, sizeof(float*));
    float* msg = (float*)malloc((size_t)(W * (maxC ? maxC : 1)) * sizeof(float));
    float* tmp = (float*)malloc((size_t)(maxlen ? maxlen : 1) * sizeof(float));
    int rc = 0;
    if (!sums || !work || !msg || !tmp) { rc = -2; goto done; }
    for (int p = 0; p < W; ++p) {
        work[p] = (float*)malloc((size_t)(maxlen ? maxlen : 1) * sizeof(float));
        if (!work[p]) { rc = -2; goto done; }
    }

    /* S1 + S2 per bucket; S4 flag */
    int flag = 0;
    for (int b = 0; b < nbuckets; ++b) {
        const int64_t st = buckets[b].start, n = buckets[b].len, C = buckets[b].chunk;
        int64_t sent[ZRO_MAX_W] = {0}, recv[ZRO_MAX_W] = {0};
        for (int p = 0; p < W; ++p) {
            const int w = ord[p];
            zro_decode(dtype, grads[(int64_t)w * A] + st, work[p], n);
            for (int a = 1; a < A; ++a) {
                zro_decode(dtype, grads[(int64_t)w * A + a] + st, tmp, n);
                for (int64_t i = 0; i < n; ++i) work[p][i] = work[p][i] + tmp[i];
            }
        }
        zro_ring_reduce_scatter(W, n, C, work, msg, sent, recv);
        for (int p = 0; p < W; ++p) {
            r.rs_sent[ord[p]] += sent[p];
            r.rs_recv[ord[p]] += recv[p];
            const int c = mod(p + 1, W);            /* owned block */
            const int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
            for (int64_t i = lo; i < hi; ++i) {
                sums[st + i] = work[p][i];
                if (!isfinite(work[p][i])) flag = 1;
            }
        }
    }
    if (flag_override >= 0) flag = flag || flag_override;
    r.overflow = flag;
    r.skipped = flag;

    if (!flag) {
        /* S3 + S5 + S6 */
        const float rr = zro_unscale_factor(sc->scale, W);
        const float bc1 = (float)(1.0 - sc->prod1 * (double)h->beta1);
        const float bc2 = (float)(1.0 - sc->prod2 * (double)h->beta2);
        uint16_t** rep16 = (uint16_t**)calloc((size_t)W, sizeof(uint16_t*));
        uint16_t* msg16 = (uint16_t*)malloc((size_t)(W * (maxC ? maxC : 1)) * sizeof(uint16_t));
        if (!rep16 || !msg16) { free(rep16); free(msg16); rc = -2; goto done; }
        for (int p = 0; p < W && rc == 0; ++p) {
            rep16[p] = (uint16_t*)calloc((size_t)(maxlen ? maxlen : 1), sizeof(uint16_t));
            if (!rep16[p]) rc = -2;
        }
        for (int b = 0; b < nbuckets && rc == 0; ++b) {
            const int64_t st = buckets[b].start, n = buckets[b].len, C = buckets[b].chunk;
            int64_t sent[ZRO_MAX_W] = {0}, recv[ZRO_MAX_W] = {0};
            for (int p = 0; p < W; ++p) {
                const int c = mod(p + 1, W);
                const int64_t lo = chunk_lo(n, C, c), hi = chunk_hi(n, C, c);
                for (int64_t i = lo; i < hi; ++i) tmp[i - lo] = sums[st + i] * rr;
                zro_adamw(hi - lo, tmp, master + st + lo, m + st + lo, v + st + lo, h, bc1, bc2);
                zro_encode(dtype, master + st + lo, rep16[p] + lo, hi - lo);
            }
            zro_ring_all_gather(W, n, C, rep16, msg16, sent, recv);
            for (int p = 0; p < W; ++p) {
                r.ag_sent[ord[p]] += sent[p];
                r.ag_recv[ord[p]] += recv[p];
                if (memcmp(rep16[p], rep16[0], (size_t)n * sizeof(uint16_t)) != 0) rc = -3;
            }
            memcpy(param + st, rep16[0], (size_t)n * sizeof(uint16_t));
        }
        for (int p = 0; p < W; ++p) free(rep16[p]);
        free(rep16);
        free(msg16);
        if (rc) goto done;
        sc->t += 1;
        sc->prod1 *= (double)h->beta1;
        sc->prod2 *= (double)h->beta2;
        sc->good += 1;
        if (sc->dynamic && sc->good >= sc->interval) { sc->scale = sc->scale * sc->growth; sc->good = 0; }
    } else if (sc->dynamic) {
        float s2 = sc->scale * sc->backoff;
        sc->scale = s2 > sc->min_scale ? s2 : sc->min_scale;
        sc->good = 0;
    }
    r.scale_next = sc->scale;
    r.t_after = sc->t;
    if (rep) *rep = r;

done:
    if (work) for (int p = 0; p < W; ++p) free(work[p]);
    free(work);
    free(msg);
    free(tmp);
    if (!sums_out) free(sums);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Memory accounting ([P3] memory table: 2+2+4+4+4 = 16 bytes per parameter;  */
/* ZeRO stage 1: 4N + 12N/W, stage 2: 2N + 14N/W, stage 3: 16N/W; [P1] 三, 四:  */
/* "2+2+K" with K = 12 for Adam). stage 0 = DDP (no sharding).                 */
/* ------------------------------------------------------------------------- */
int64_t zro_model_state_bytes(int stage, int64_t n, int W) {
    if (W < 1 || n < 0) return -1;
    switch (stage) {
        case 0: return 16 * n;
        case 1: return 4 * n + (12 * n) / W;
        case 2: return 2 * n + (14 * n) / W;
        case 3: return (16 * n) / W;
        default: return -1;
    }
}
