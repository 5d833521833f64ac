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

/* Tensor ids (the Philox key's second word). */
enum {
    SYNTH_T_GATE_Q = 1, SYNTH_T_UP_Q = 2, SYNTH_T_DOWN_Q = 3,
    SYNTH_T_GATE_S = 4, SYNTH_T_UP_S = 5, SYNTH_T_DOWN_S = 6,
    SYNTH_T_X = 7, SYNTH_T_LOGITS = 8, SYNTH_T_WR = 9, SYNTH_T_ZIPF = 10,
    SYNTH_T_SH_GATE = 11, SYNTH_T_SH_UP = 12, SYNTH_T_SH_DOWN = 13
};

#endif
