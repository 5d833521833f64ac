/*
 * Philox4x32-10 counter-based generator, written from its published
 * definition: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11, section 4
 * (the Philox-4x32 S-box: two 32x32->64 multiplies per round, Weyl key
 * schedule, 10 rounds).
 *
 * This header belongs to the seeded input generator only. It holds none of
 * the MoE layer's arithmetic; it is shared by the host and device halves of
 * the generator so that both emit byte-identical synthetic inputs.
 */
#ifndef SYNTH_PHILOX_H
#define SYNTH_PHILOX_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SYNTH_PHILOX_M0 0xD2511F53u
#define SYNTH_PHILOX_M1 0xCD9E8D57u
#define SYNTH_PHILOX_W0 0x9E3779B9u /* golden ratio */
#define SYNTH_PHILOX_W1 0xBB67AE85u /* sqrt(3) - 1 */

typedef struct { uint32_t v[4]; } synth_u32x4;

SYNTH_HD void synth_mulhilo32(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

/* One call: 10 rounds over the 128-bit counter under the 64-bit key. */
SYNTH_HD synth_u32x4 synth_philox4x32_10(synth_u32x4 c, uint32_t k0, uint32_t k1) {
    for (int r = 0; r < 10; ++r) {
        if (r > 0) { k0 += SYNTH_PHILOX_W0; k1 += SYNTH_PHILOX_W1; }
        uint32_t hi0, lo0, hi1, lo1;
        synth_mulhilo32(SYNTH_PHILOX_M0, c.v[0], &hi0, &lo0);
        synth_mulhilo32(SYNTH_PHILOX_M1, c.v[2], &hi1, &lo1);
        synth_u32x4 n;
        n.v[0] = hi1 ^ c.v[1] ^ k0;
        n.v[1] = lo1;
        n.v[2] = hi0 ^ c.v[3] ^ k1;
        n.v[3] = lo0;
        c = n;
    }
    return c;
}

/*
 * Stream addressing used by every synthetic tensor:
 *   key     = { low 32 bits of seed, tensor id }
 *   counter = { block index along the row, row, expert (or 0), high 32 bits of seed }
 * One call yields 16 bytes (4 little-endian words).
 */
SYNTH_HD synth_u32x4 synth_block(uint64_t seed, uint32_t tensor, uint32_t expert,
                                 uint32_t row, uint32_t blk) {
    synth_u32x4 c;
    c.v[0] = blk; c.v[1] = row; c.v[2] = expert; c.v[3] = (uint32_t)(seed >> 32);
    return synth_philox4x32_10(c, (uint32_t)seed, tensor);
}

/* Uniform draw over n consecutive integers starting at lo, from one word
 * (multiply-shift: floor(w * n / 2^32)). */
SYNTH_HD uint32_t synth_uniform_int(uint32_t w, uint32_t lo, uint32_t n) {
    return lo + (uint32_t)(((uint64_t)w * (uint64_t)n) >> 32);
}

/* Second code distribution ("peaked"): E2M1 codes shaped like those of
 * block-scaled normal weights rather than uniform, so that the bytes carry the
 * redundancy a trained layer's do. Magnitude codes 0..7 are drawn from a fixed
 * table (parts of 2^15: 3260, 6318, 5757, 4928, 5580, 4299, 2218, 408; close
 * to a standard normal binned at 0.125, 0.375, 0.625, 0.875, 1.25, 1.75, 2.5)
 * and the sign bit uniformly, so half of the zero codes are negative zeros.
 * One 16-bit draw per code: bit 0 the sign, bits 1..15 the magnitude. */
SYNTH_HD uint32_t synth_peaked_code(uint32_t h16) {
    const uint32_t u = (h16 >> 1) & 0x7FFFu;
    uint32_t m = 0;
    m += u >= 3260u;
    m += u >= 9578u;
    m += u >= 15335u;
    m += u >= 20263u;
    m += u >= 25843u;
    m += u >= 30142u;
    m += u >= 32360u;
    return ((h16 & 1u) << 3) | m;
}

/* 16 bytes (32 codes) of row `row`, block `blk` under the peaked distribution:
 * four Philox calls (blocks 4 blk .. 4 blk + 3), code n from the 16-bit half
 * n % 2 of word n / 2; byte j holds code 2j in its low nibble. */
SYNTH_HD void synth_peaked_block(uint64_t seed, uint32_t tensor, uint32_t expert, uint32_t row,
                                 uint32_t blk, uint8_t out[16]) {
    for (int q = 0; q < 4; ++q) {
        synth_u32x4 w = synth_block(seed, tensor, expert, row, 4u * blk + (uint32_t)q);
        for (int i = 0; i < 4; ++i) {  /* word i of call q: codes 8q + 2i, 8q + 2i + 1 */
            const uint32_t lo = synth_peaked_code(w.v[i] & 0xFFFFu);
            const uint32_t hi = synth_peaked_code(w.v[i] >> 16);
            out[4 * q + i] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* FP8 expert weights (E4M3FN lane): one byte per weight from one random
 * byte b: the sign from bit 7 and the magnitude code 0x20 + (b & 0x3F), i.e.
 * exponent fields 4..11 with every mantissa, values 2^-3 .. 30 spread
 * log-uniformly over eight binades; never a NaN code. */
SYNTH_HD uint32_t synth_fp8_code(uint32_t b) {
    return (b & 0x80u) | (0x20u + (b & 0x3Fu));
}

/* fp32 bits of an FP8 block scale from one word w: 2^-7 * (1 + m 2^-23) with
 * the 23 mantissa bits m = w >> 9 (every mantissa occurs; values in
 * [2^-7, 2^-6)). */
SYNTH_HD uint32_t synth_fp8_scale_bits(uint32_t w) {
    return ((uint32_t)(127 - 7) << 23) | (w >> 9);
}

/* Tensor ids (the Philox key's second word). */
enum {
    SYNTH_T_GATE_Q = 1, SYNTH_T_UP_Q = 2, SYNTH_T_DOWN_Q = 3,
    SYNTH_T_GATE_S = 4, SYNTH_T_UP_S = 5, SYNTH_T_DOWN_S = 6,
    SYNTH_T_X = 7, SYNTH_T_LOGITS = 8, SYNTH_T_WR = 9, SYNTH_T_ZIPF = 10,
    SYNTH_T_SH_GATE = 11, SYNTH_T_SH_UP = 12, SYNTH_T_SH_DOWN = 13,
    SYNTH_T_F8_GATE_Q = 14, SYNTH_T_F8_UP_Q = 15, SYNTH_T_F8_DOWN_Q = 16,
    SYNTH_T_F8_GATE_S = 17, SYNTH_T_F8_UP_S = 18, SYNTH_T_F8_DOWN_S = 19
};

#endif
