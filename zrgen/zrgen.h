/*
 * zrgen — seeded synthetic inputs for the ZeRO post-backward step.
 *
 * This module produces inputs only. It holds none of the step's arithmetic
 * (no reduction, no optimizer, no scaling rule): both the oracle's tests and the
 * CUDA path take their gradients, masters and per-tensor sigmas from here, so
 * that the two sides see the same bytes.
 *
 * Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11), a counter-based RNG. Element i of a
 * stream takes 16 bits of one Philox block:
 *     block  = Philox(ctr = {i/8 lo, i/8 hi, stream lo, stream hi},
 *                     key = {seed lo, seed hi})
 *     u16(i) = 16-bit lane (i mod 8) of block, lane 2j = low half of word j,
 *              lane 2j+1 = high half of word j.
 * A normal draw is table[u16(i)], where table[k] = Phi^-1((k + 0.5) / 65536)
 * rounded once to fp32 (built in double by bisection on erfc, mirrored so that
 * table[65535-k] = -table[k]). A scaled value is one fp32 multiply
 * table[u] * scale, rounded to the destination type with round-to-nearest-even.
 * Because every step is exactly rounded, the host and device fills give equal
 * bytes; a test checks that.
 *
 * Host functions live in zrgen_host.c (plain C); device fills in zrgen_dev.cu.
 */
#ifndef ZRGEN_H
#define ZRGEN_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ZRGEN_F16 = 0, ZRGEN_BF16 = 1, ZRGEN_F32 = 2 };
#define ZRGEN_TABLE_SIZE 65536

/* ---- host (libzrgen_host.so) ---- */

/* One Philox4x32-10 block. ctr[4], key[2] in; out[4] out. */
void zrgen_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* Fill table[65536] with the inverse-normal quantile table described above. */
void zrgen_normal_table(float* table);

/* u16 draw of element `index` of (seed, stream). */
uint16_t zrgen_u16(uint64_t seed, uint64_t stream, uint64_t index);

/* Uniform double in [0,1) from the 32-bit word `word` (0..3) of block `block`. */
double zrgen_uniform(uint64_t seed, uint64_t stream, uint64_t block, int word);

/* out[j] = round_dt(table[u16(first + j)] * scale), j in [0, n). dtype: ZRGEN_*.
   out is host memory of n elements of that dtype. Returns 0, or -1 on a bad dtype. */
int zrgen_fill_normal_host(void* out, int dtype, uint64_t n, uint64_t seed, uint64_t stream,
                           uint64_t first, float scale, const float* table);

/* Round-to-nearest-even fp32 -> fp16 / bf16 bit patterns (used to produce inputs). */
uint16_t zrgen_f32_to_f16(float f);
uint16_t zrgen_f32_to_bf16(float f);

/* ---- device (libzrgen_dev.so) ---- */
/* Same values as zrgen_fill_normal_host, written to device memory `out` on `stream_handle`
   (a cudaStream_t; NULL = legacy default stream). table_dev: device copy of the table.
   Returns 0, -1 on a bad argument, or -2 if the launch failed. */
int zrgen_fill_normal_dev(void* out, int dtype, uint64_t n, uint64_t seed, uint64_t stream,
                          uint64_t first, float scale, const float* table_dev, void* stream_handle);

#ifdef __cplusplus
}
#endif
#endif
