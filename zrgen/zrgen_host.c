/* Host side of the synthetic input generator. Plain C99; see zrgen.h for the
 * definition of every value produced here. Built with -ffp-contract=off. */
#include "zrgen.h"
#include <math.h>
#include <string.h>

/* Philox4x32 multipliers and Weyl key increments (Salmon et al., SC'11, Table 2). */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void zrgen_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += PHILOX_W0; k1 += PHILOX_W1; }
        uint64_t p0 = (uint64_t)PHILOX_M0 * c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static void block_of(uint64_t seed, uint64_t stream, uint64_t block, uint32_t out[4]) {
    uint32_t ctr[4] = {(uint32_t)block, (uint32_t)(block >> 32), (uint32_t)stream, (uint32_t)(stream >> 32)};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    zrgen_philox4x32_10(ctr, key, out);
}

uint16_t zrgen_u16(uint64_t seed, uint64_t stream, uint64_t index) {
    uint32_t b[4];
    block_of(seed, stream, index >> 3, b);
    unsigned lane = (unsigned)(index & 7u);
    uint32_t w = b[lane >> 1];
    return (uint16_t)((lane & 1u) ? (w >> 16) : (w & 0xFFFFu));
}

double zrgen_uniform(uint64_t seed, uint64_t stream, uint64_t block, int word) {
    uint32_t b[4];
    block_of(seed, stream, block, b);
    return (double)b[word & 3] * (1.0 / 4294967296.0);
}

/* Standard normal CDF in double. */
static double phi(double x) { return 0.5 * erfc(-x / sqrt(2.0)); }

void zrgen_normal_table(float* table) {
    for (int k = 0; k < ZRGEN_TABLE_SIZE / 2; ++k) {
        double p = ((double)k + 0.5) / (double)ZRGEN_TABLE_SIZE;
        double lo = -12.0, hi = 0.0; /* p < 0.5, so the quantile is negative */
        for (int it = 0; it < 200 && hi - lo > 0.0; ++it) {
            double mid = 0.5 * (lo + hi);
            if (mid <= lo || mid >= hi) break;
            if (phi(mid) < p) lo = mid; else hi = mid;
        }
        float q = (float)(0.5 * (lo + hi));
        table[k] = q;
        table[ZRGEN_TABLE_SIZE - 1 - k] = -q;
    }
}

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

uint16_t zrgen_f32_to_bf16(float f) {
    uint32_t x = f32_bits(f);
    if ((x & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)(((x >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t lsb = (x >> 16) & 1u;
    x += 0x7FFFu + lsb;
    return (uint16_t)(x >> 16);
}

uint16_t zrgen_f32_to_f16(float f) {
    uint32_t x = f32_bits(f);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t a = x & 0x7FFFFFFFu;
    if (a > 0x7F800000u) return (uint16_t)(sign | 0x7E00u);   /* NaN */
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);  /* >= 65520 rounds to inf */
    if (a < 0x38800000u) {                                    /* below 2^-14: subnormal or zero */
        if (a < 0x33000000u) return (uint16_t)sign;           /* below 2^-25 */
        uint32_t e = a >> 23;
        uint32_t mant = (a & 0x7FFFFFu) | 0x800000u;
        uint32_t sh = 126u - e;                               /* 14..24 */
        uint32_t m = mant >> sh;
        uint32_t rem = mant & ((1u << sh) - 1u);
        uint32_t half = 1u << (sh - 1u);
        if (rem > half || (rem == half && (m & 1u))) m += 1u;
        return (uint16_t)(sign | m);
    }
    uint32_t h = (a - 0x38000000u) >> 13;
    uint32_t rem = a & 0x1FFFu;
    if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
    return (uint16_t)(sign | h);
}

int zrgen_fill_normal_host(void* out, int dtype, uint64_t n, uint64_t seed, uint64_t stream,
                           uint64_t first, float scale, const float* table) {
    if (dtype != ZRGEN_F16 && dtype != ZRGEN_BF16 && dtype != ZRGEN_F32) return -1;
    uint64_t j = 0;
    while (j < n) {
        uint64_t idx = first + j;
        uint32_t b[4];
        block_of(seed, stream, idx >> 3, b);
        for (unsigned lane = (unsigned)(idx & 7u); lane < 8u && j < n; ++lane, ++j) {
            uint32_t w = b[lane >> 1];
            uint16_t u = (uint16_t)((lane & 1u) ? (w >> 16) : (w & 0xFFFFu));
            volatile float val = table[u] * scale;  /* one fp32 multiply */
            if (dtype == ZRGEN_F32) ((float*)out)[j] = val;
            else if (dtype == ZRGEN_F16) ((uint16_t*)out)[j] = zrgen_f32_to_f16(val);
            else ((uint16_t*)out)[j] = zrgen_f32_to_bf16(val);
        }
    }
    return 0;
}
