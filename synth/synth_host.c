/*
 * Host half of the seeded synthetic-input generator.
 *
 * Produces the workloads' inputs (MXFP4 expert weights, bf16 activations,
 * fp32 router logits and router weights) from Philox4x32-10 streams. It holds
 * none of the MoE layer's arithmetic: weights come out as raw E2M1 codes and
 * E8M0 bytes, never as decoded values. The device half (synth_dev.cu) emits
 * the same bytes for the expert weights, so the 15.7 GB layer can be made on
 * the GPU while any expert the CPU checker needs is made here.
 *
 * Distributions (one reading of the workloads described for the Kimi-K3
 * routed layer): E2M1 codes uniform over all 16 codes (a random byte holds two
 * independent uniform codes); E8M0 scale bytes uniform over {lo..lo+n-1};
 * normals by the Box-Muller transform in double precision, rounded to fp32
 * (and then to bf16 with round-to-nearest-even where asked).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include "philox.h"

#define SYNTH_API __attribute__((visibility("default")))

SYNTH_API void synth_philox(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    synth_u32x4 c;
    for (int i = 0; i < 4; ++i) c.v[i] = ctr[i];
    synth_u32x4 r = synth_philox4x32_10(c, key[0], key[1]);
    for (int i = 0; i < 4; ++i) out[i] = r.v[i];
}

/* Packed E2M1 codes: rows x (K/2) bytes for expert e; K must be a multiple of 32. */
SYNTH_API int synth_mx_codes(uint64_t seed, uint32_t tensor, uint32_t expert,
                             int64_t rows, int64_t K, uint8_t *out) {
    if (K % 32 != 0 || rows < 0) return -1;
    int64_t nb = K / 2;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        uint8_t *dst = out + r * nb;
        for (int64_t b = 0; b < nb / 16; ++b) {
            synth_u32x4 w = synth_block(seed, tensor, expert, (uint32_t)r, (uint32_t)b);
            for (int i = 0; i < 4; ++i) {
                dst[b * 16 + 4 * i + 0] = (uint8_t)(w.v[i]);
                dst[b * 16 + 4 * i + 1] = (uint8_t)(w.v[i] >> 8);
                dst[b * 16 + 4 * i + 2] = (uint8_t)(w.v[i] >> 16);
                dst[b * 16 + 4 * i + 3] = (uint8_t)(w.v[i] >> 24);
            }
        }
    }
    return 0;
}

/* Packed E2M1 codes under distribution `dist` (0: uniform, as synth_mx_codes;
 * 1: peaked, see philox.h). */
SYNTH_API int synth_mx_codes_dist(uint64_t seed, uint32_t tensor, uint32_t expert,
                                  int64_t rows, int64_t K, int dist, uint8_t *out) {
    if (dist == 0) return synth_mx_codes(seed, tensor, expert, rows, K, out);
    if (dist != 1 || K % 32 != 0 || rows < 0) return -1;
    int64_t nb = K / 2;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nb / 16; ++b)
            synth_peaked_block(seed, tensor, expert, (uint32_t)r, (uint32_t)b, out + r * nb + b * 16);
    return 0;
}

/* E8M0 scale bytes: rows x (K/32) bytes, each uniform over {lo .. lo+n-1}. */
SYNTH_API int synth_mx_scales(uint64_t seed, uint32_t tensor, uint32_t expert,
                              int64_t rows, int64_t K, int lo, int n, uint8_t *out) {
    if (K % 32 != 0 || rows < 0 || n < 1 || lo < 0 || lo + n - 1 > 254) return -1;
    int64_t ns = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t i = 0; i < ns; ++i) {
            synth_u32x4 w = synth_block(seed, tensor, expert, (uint32_t)r, (uint32_t)(i / 4));
            out[r * ns + i] = (uint8_t)synth_uniform_int(w.v[i % 4], (uint32_t)lo, (uint32_t)n);
        }
    }
    return 0;
}

/* FP8 expert codes: rows x K bytes (K a multiple of 16), byte j of 16-byte
 * block b of row r from Philox block (r, b), mapped by synth_fp8_code. */
SYNTH_API int synth_fp8_codes(uint64_t seed, uint32_t tensor, uint32_t expert, int64_t rows,
                              int64_t K, uint8_t *out) {
    if (K % 16 != 0 || rows < 0) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t b = 0; b < K / 16; ++b) {
            synth_u32x4 w = synth_block(seed, tensor, expert, (uint32_t)r, (uint32_t)b);
            for (int j = 0; j < 16; ++j)
                out[r * K + b * 16 + j] = (uint8_t)synth_fp8_code((w.v[j / 4] >> (8 * (j % 4))) & 0xFFu);
        }
    }
    return 0;
}

/* FP8 block scales: fp32 [ceil(rows/128)][ceil(K/128)], entry (i, j) from word
 * j % 4 of Philox block (i, j / 4). */
SYNTH_API int synth_fp8_scales(uint64_t seed, uint32_t tensor, uint32_t expert, int64_t rows,
                               int64_t K, float *out) {
    if (rows < 0 || K < 0) return -1;
    const int64_t nr = (rows + 127) / 128, nk = (K + 127) / 128;
    for (int64_t i = 0; i < nr; ++i)
        for (int64_t j = 0; j < nk; ++j) {
            synth_u32x4 w = synth_block(seed, tensor, expert, (uint32_t)i, (uint32_t)(j / 4));
            const uint32_t bits = synth_fp8_scale_bits(w.v[j % 4]);
            memcpy(&out[i * nk + j], &bits, 4);
        }
    return 0;
}

static double synth_normal_at(uint64_t seed, uint32_t tensor, int64_t r, int64_t c) {
    synth_u32x4 w = synth_block(seed, tensor, 0, (uint32_t)r, (uint32_t)(c / 4));
    int pair = (int)((c % 4) / 2);
    double u1 = ((double)w.v[2 * pair] + 0.5) * (1.0 / 4294967296.0);
    double u2 = (double)w.v[2 * pair + 1] * (1.0 / 4294967296.0);
    double rad = sqrt(-2.0 * log(u1));
    double ang = 6.283185307179586 * u2;
    return (c % 2 == 0) ? rad * cos(ang) : rad * sin(ang);
}

/* fp32 normals N(mean, sigma^2): rows x cols, row-major. */
SYNTH_API void synth_normal_f32(uint64_t seed, uint32_t tensor, int64_t rows, int64_t cols,
                                double mean, double sigma, float *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] = (float)(mean + sigma * synth_normal_at(seed, tensor, r, c));
}

static uint16_t synth_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* bf16 normals N(0, sigma^2), rounded to fp32 then to bf16 (RNE). */
SYNTH_API void synth_normal_bf16(uint64_t seed, uint32_t tensor, int64_t rows, int64_t cols,
                                 double sigma, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[r * cols + c] =
                synth_f32_to_bf16_rne((float)(sigma * synth_normal_at(seed, tensor, r, c)));
}

/*
 * Zipf popularity bias over a seeded permutation of the experts:
 *   rank(e) = pi(e) + 1,  bias[e] = -s * ln(rank(e)).
 * pi comes from a Fisher-Yates shuffle driven by one Philox stream.
 */
SYNTH_API void synth_zipf_bias(uint64_t seed, int E, double s, int32_t *perm_out, float *bias) {
    for (int i = 0; i < E; ++i) perm_out[i] = i;
    for (int i = E - 1; i > 0; --i) {
        synth_u32x4 w = synth_block(seed, SYNTH_T_ZIPF, 0, 0, (uint32_t)i);
        int j = (int)synth_uniform_int(w.v[0], 0, (uint32_t)(i + 1));
        int32_t t = perm_out[i]; perm_out[i] = perm_out[j]; perm_out[j] = t;
    }
    for (int e = 0; e < E; ++e) bias[e] = (float)(-s * log((double)(perm_out[e] + 1)));
}
