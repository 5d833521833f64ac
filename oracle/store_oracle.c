/*
 * CPU oracle of the compressed expert store (test infrastructure only).
 *
 * The pages describe the store only in outline (Moonshine GitHub README,
 * "Expert-stream compression" / "MZG2 production store"): rANS-coded 16 KiB
 * tiles that can be decoded independently on the GPU straight into ordinary
 * expert cache slots, redundant MXFP4 negative zeros canonicalised first, a
 * checksum per tile and a check of the coder's final state. They fix no byte
 * format, so this file states one plain reading and is its definition; the
 * CUDA library implements the same format independently. Integer arithmetic
 * only, one tile at a time, in the order the steps are stated.
 *
 * Format:
 *  - An expert's six arrays in the order gate_q, gate_s, up_q, up_s, down_q,
 *    down_s (n_a = D*F/2 bytes for codes, D*F/32 for scales).
 *  - Canonical bytes: in the code arrays each 4-bit E2M1 code 0x8 (negative
 *    zero) becomes 0x0; scale bytes are kept.
 *  - Model: one table per (expert, array): f[256], sum 4096 over the bytes
 *    that occur (quantisation rule in oracle_store_freq).
 *  - Tiles: each array is cut into 16384-byte tiles (the last may be
 *    shorter). A tile of n bytes is coded by 32 interleaved rANS coders with
 *    32-bit states in [2^16, 2^32), 12-bit frequencies and 16-bit
 *    renormalisation words: byte i belongs to coder i % 32 at step i / 32.
 *    Encoding runs the steps backwards and, within a step, coders 31..0; each
 *    coder starts at 2^16, emits its low 16 bits once when its state is at
 *    least f * 2^20, then x = (x / f) * 4096 + x % f + cum. The stored tile is
 *    the 32 final states (coder 0 first) and then the words in the reverse of
 *    the order they were emitted. Decoding runs the steps forwards: every coder
 *    with a byte in the step takes q = x % 4096, the byte s with
 *    cum[s] <= q < cum[s] + f[s], sets x = f * (x / 4096) + q - cum, and, if x
 *    fell below 2^16, reads the next word (x = x * 2^16 + w), coders in
 *    increasing order. A sound tile ends with every state at 2^16 and every
 *    word read.
 *  - A tile is stored coded when 128 + 2 * words < n, else raw (its n
 *    canonical bytes). Stored tiles are zero-padded to a multiple of 16 bytes
 *    and laid out back to back, expert by expert, tile by tile.
 *  - Tile record (8 x u32): offset (low, high word; bytes from the start of
 *    the blob), n_bytes, n_words (0 when raw), adler (Adler-32 of the tile's
 *    canonical bytes), flags (bit 0: raw), two zero words.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

enum { TILE = 16384, PREC = 12, M = 1 << PREC, LANES = 32 };
static const uint32_t LOW = 1u << 16;

/* E2M1 negative zero (code 0x8) -> 0x0 in both nibbles of every byte. */
ORACLE_API void oracle_store_canonical(const uint8_t *in, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) {
        uint8_t lo = in[i] & 15, hi = in[i] >> 4;
        if (lo == 8) lo = 0;
        if (hi == 8) hi = 0;
        out[i] = (uint8_t)(lo | (hi << 4));
    }
}

/* Adler-32 as zlib defines it (RFC 1950, section 8): A = 1 + sum of the bytes,
 * B = sum of the successive values of A, both mod 65521; B * 65536 + A. */
ORACLE_API uint32_t oracle_adler32(const uint8_t *p, int64_t n) {
    uint32_t a = 1, b = 0;
    for (int64_t i = 0; i < n; ++i) {
        a = (a + p[i]) % 65521u;
        b = (b + a) % 65521u;
    }
    return (b << 16) | a;
}

/* Table of one array's canonical bytes: f[s] = 0 for bytes that never occur,
 * else max(1, floor(count * 4096 / n)); then, while the total exceeds 4096,
 * the largest f (smallest byte value among equals) loses one, and while it
 * falls short, the largest gains one. Returns -1 for n <= 0. */
ORACLE_API int oracle_store_freq(const uint8_t *canon, int64_t n, uint16_t f[256]) {
    if (n <= 0) return -1;
    int64_t count[256];
    memset(count, 0, sizeof(count));
    for (int64_t i = 0; i < n; ++i) count[canon[i]]++;
    int64_t total = 0;
    for (int s = 0; s < 256; ++s) {
        int64_t v = count[s] ? (count[s] * M) / n : 0;
        if (count[s] && v < 1) v = 1;
        f[s] = (uint16_t)v;
        total += v;
    }
    while (total != M) {
        int best = 0;
        for (int s = 1; s < 256; ++s)
            if (f[s] > f[best]) best = s;
        if (total > M) {
            f[best]--;
            total--;
        } else {
            f[best]++;
            total++;
        }
    }
    return 0;
}

/* Encodes one tile (n <= 16384 canonical bytes) with table f. out receives the
 * stored tile (at most 128 + 2 * 16384 bytes before padding; coded or raw);
 * returns its unpadded size and sets *n_words (0 when stored raw) and *raw. */
ORACLE_API int64_t oracle_store_encode_tile(const uint8_t *d, int64_t n, const uint16_t f[256],
                                            uint8_t *out, uint32_t *n_words, int *raw) {
    uint32_t cum[256];
    uint32_t c = 0;
    for (int s = 0; s < 256; ++s) {
        cum[s] = c;
        c += f[s];
    }
    uint32_t x[LANES];
    for (int j = 0; j < LANES; ++j) x[j] = LOW;
    uint16_t *pushed = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1));
    int64_t np = 0;
    const int64_t steps = (n + LANES - 1) / LANES;
    for (int64_t t = steps - 1; t >= 0; --t) {
        for (int j = LANES - 1; j >= 0; --j) {
            const int64_t i = t * LANES + j;
            if (i >= n) continue;
            const uint32_t s = d[i], fs = f[s];
            if (fs == 0) {  /* byte absent from the table: not encodable */
                free(pushed);
                return -1;
            }
            if ((uint64_t)x[j] >= ((uint64_t)fs << 20)) {
                pushed[np++] = (uint16_t)(x[j] & 0xFFFFu);
                x[j] >>= 16;
            }
            x[j] = (x[j] / fs) * M + (x[j] % fs) + cum[s];
        }
    }
    if (128 + 2 * np < n) {
        for (int j = 0; j < LANES; ++j)
            for (int b = 0; b < 4; ++b) out[4 * j + b] = (uint8_t)(x[j] >> (8 * b));
        for (int64_t k = 0; k < np; ++k) {
            const uint16_t w = pushed[np - 1 - k];
            out[128 + 2 * k] = (uint8_t)w;
            out[128 + 2 * k + 1] = (uint8_t)(w >> 8);
        }
        free(pushed);
        *n_words = (uint32_t)np;
        *raw = 0;
        return 128 + 2 * np;
    }
    free(pushed);
    memcpy(out, d, (size_t)n);
    *n_words = 0;
    *raw = 1;
    return n;
}

/* Decodes one stored tile into n bytes. Returns 0 when the tile is sound
 * (coded: every state back at 2^16 and exactly n_words words read), 1 when
 * not; reads never go past the n_words words (a missing word reads as 0). */
ORACLE_API int oracle_store_decode_tile(const uint8_t *in, int64_t n, uint32_t n_words, int raw,
                                        const uint16_t f[256], uint8_t *d) {
    if (raw) {
        memcpy(d, in, (size_t)n);
        return 0;
    }
    uint32_t cum[257];
    cum[0] = 0;
    for (int s = 0; s < 256; ++s) cum[s + 1] = cum[s] + f[s];
    if (cum[256] != M) return 1;
    uint32_t x[LANES];
    for (int j = 0; j < LANES; ++j)
        x[j] = (uint32_t)in[4 * j] | (uint32_t)in[4 * j + 1] << 8 | (uint32_t)in[4 * j + 2] << 16 |
               (uint32_t)in[4 * j + 3] << 24;
    int bad = 0;
    uint32_t r = 0;
    const int64_t steps = (n + LANES - 1) / LANES;
    for (int64_t t = 0; t < steps; ++t) {
        for (int j = 0; j < LANES; ++j) {
            const int64_t i = t * LANES + j;
            if (i >= n) continue;
            const uint32_t q = x[j] % M;
            int s = 0;
            while (!(cum[s] <= q && q < cum[s + 1])) ++s;  /* f[s] > 0 there */
            d[i] = (uint8_t)s;
            x[j] = f[s] * (x[j] / M) + q - cum[s];
            if (x[j] < LOW) {
                uint32_t w = 0;
                if (r < n_words)
                    w = (uint32_t)in[128 + 2 * r] | (uint32_t)in[128 + 2 * r + 1] << 8;
                else
                    bad = 1;
                ++r;
                x[j] = (x[j] << 16) | w;
            }
        }
    }
    for (int j = 0; j < LANES; ++j)
        if (x[j] != LOW) bad = 1;
    if (r != n_words) bad = 1;
    return bad;
}

static int64_t round16(int64_t v) { return (v + 15) / 16 * 16; }

/* Tiles of one expert of a d_model x d_ff layer, and the six array sizes. */
static int64_t arrays(int64_t D, int64_t F, int64_t nb[6]) {
    const int64_t n = D * F;
    int64_t t = 0;
    for (int a = 0; a < 6; ++a) {
        nb[a] = (a % 2 == 0) ? n / 2 : n / 32;
        t += (nb[a] + TILE - 1) / TILE;
    }
    return t;
}

ORACLE_API int64_t oracle_store_tiles_per_expert(int64_t D, int64_t F) {
    int64_t nb[6];
    return arrays(D, F, nb);
}

/* Whole store of experts 0..E-1. w[a] points at array a of all experts
 * ([E][n_a] bytes). Writes the blob (capacity cap bytes), the tile records
 * ([E][tiles per expert][8] u32) and the tables ([E][6][256] u16); returns the
 * blob's size, or -1 when cap is too small or an argument is invalid. */
ORACLE_API int64_t oracle_store_build(int64_t E, int64_t D, int64_t F, const uint8_t *const w[6],
                                      uint8_t *blob, int64_t cap, uint32_t *rec, uint16_t *tab) {
    int64_t nb[6];
    const int64_t tpe = arrays(D, F, nb);
    if (E <= 0 || D <= 0 || F <= 0 || D % 32 || F % 32) return -1;  /* MXFP4 layouts */
    uint8_t *canon = (uint8_t *)malloc((size_t)nb[0]);
    uint8_t *tile = (uint8_t *)malloc(128 + 2 * TILE);
    int64_t off = 0;
    for (int64_t e = 0; e < E; ++e) {
        int64_t t = 0;
        for (int a = 0; a < 6; ++a) {
            const uint8_t *src = w[a] + e * nb[a];
            if (a % 2 == 0)
                oracle_store_canonical(src, nb[a], canon);
            else
                memcpy(canon, src, (size_t)nb[a]);
            uint16_t *f = tab + (e * 6 + a) * 256;
            oracle_store_freq(canon, nb[a], f);
            for (int64_t p = 0; p < nb[a]; p += TILE, ++t) {
                const int64_t n = nb[a] - p < TILE ? nb[a] - p : TILE;
                uint32_t nw = 0;
                int raw = 0;
                const int64_t sz = oracle_store_encode_tile(canon + p, n, f, tile, &nw, &raw);
                if (sz < 0 || off + round16(sz) > cap) {
                    free(canon);
                    free(tile);
                    return -1;
                }
                memcpy(blob + off, tile, (size_t)sz);
                memset(blob + off + sz, 0, (size_t)(round16(sz) - sz));
                uint32_t *r = rec + (e * tpe + t) * 8;
                r[0] = (uint32_t)off;
                r[1] = (uint32_t)((uint64_t)off >> 32);
                r[2] = (uint32_t)n;
                r[3] = nw;
                r[4] = oracle_adler32(canon + p, n);
                r[5] = raw ? 1u : 0u;
                r[6] = r[7] = 0;
                off += round16(sz);
            }
        }
    }
    free(canon);
    free(tile);
    return off;
}
