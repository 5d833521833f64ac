// Host encoder of the compressed expert store (format stated in moe.h;
// Moonshine GitHub README, "Expert-stream compression" / "MZG2 production
// store": canonical negative zeros, independent 16 KiB rANS tiles, a
// checksum per tile). Experts are encoded in parallel by host threads, each
// into its own stretch of the blob at a fixed stride (an expert's raw size,
// which bounds its stored size); the stretches are then packed in expert
// order.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "../../include/moe.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int64_t kTile = 16384;
constexpr uint32_t kProbBits = 12;
constexpr uint32_t kProbTotal = 1u << kProbBits;
constexpr uint32_t kStateLow = 1u << 16;  // states live in [kStateLow, 2^32)
constexpr int kCoders = 32;

struct Layout {
    int64_t bytes[6];     // per expert and array
    int64_t first[7];     // first tile of each array within an expert; first[6] = tiles
    int64_t stride;       // raw bytes of an expert's tiles, each rounded up to 16
};

bool layout_of(int64_t D, int64_t F, Layout &L) {
    if (D <= 0 || F <= 0 || D % 32 != 0 || F % 32 != 0) return false;  // MXFP4 layouts
    L.first[0] = 0;
    L.stride = 0;
    for (int a = 0; a < 6; ++a) {
        L.bytes[a] = (a & 1) ? D * F / 32 : D * F / 2;
        const int64_t full = L.bytes[a] / kTile, tail = L.bytes[a] % kTile;
        L.first[a + 1] = L.first[a] + full + (tail ? 1 : 0);
        L.stride += full * kTile + (tail + 15) / 16 * 16;
    }
    return true;
}

// Canonical byte of every byte value: an E2M1 nibble 0x8 (negative zero)
// becomes 0x0, in either half.
struct Canon {
    uint8_t to[256];
    Canon() {
        for (int v = 0; v < 256; ++v) {
            const int lo = (v & 0x0F) == 0x08 ? 0 : (v & 0x0F);
            const int hi = (v & 0xF0) == 0x80 ? 0 : (v & 0xF0);
            to[v] = (uint8_t)(hi | lo);
        }
    }
};
const Canon kCanon;

// Frequency table of an array from its byte counts (the rule in moe.h).
void quantise(const uint64_t count[256], uint64_t n, uint16_t f[256]) {
    int64_t sum = 0;
    for (int b = 0; b < 256; ++b) {
        uint64_t v = count[b] ? count[b] * kProbTotal / n : 0;
        if (count[b] && v == 0) v = 1;
        f[b] = (uint16_t)v;
        sum += (int64_t)v;
    }
    for (; sum != (int64_t)kProbTotal; sum += sum > (int64_t)kProbTotal ? -1 : 1) {
        int top = 0;
        for (int b = 1; b < 256; ++b)
            if (f[b] > f[top]) top = b;
        f[top] = (uint16_t)(sum > (int64_t)kProbTotal ? f[top] - 1 : f[top] + 1);
    }
}

// Adler-32 of n bytes (zlib's definition), sums reduced every 4096 bytes.
uint32_t adler32(const uint8_t *p, int64_t n) {
    uint64_t a = 1, b = 0;
    while (n > 0) {
        const int64_t k = n < 4096 ? n : 4096;
        for (int64_t i = 0; i < k; ++i) {
            a += p[i];
            b += a;
        }
        a %= 65521u;
        b %= 65521u;
        p += k;
        n -= k;
    }
    return (uint32_t)((b << 16) | a);
}

// Stores one tile of n canonical bytes at dst (coded or raw, zero-padded to
// 16); returns the padded size. `words` is scratch for kTile words.
int64_t store_tile(const uint8_t *src, int64_t n, const uint16_t f[256], const uint32_t cum[256],
                   uint16_t *words, uint8_t *dst, moe_tile_rec &rec) {
    uint32_t state[kCoders];
    for (int c = 0; c < kCoders; ++c) state[c] = kStateLow;
    int64_t head = kTile;  // words are produced last-read-first: fill from the end
    const int64_t steps = (n + kCoders - 1) / kCoders;
    for (int64_t t = steps - 1; t >= 0; --t) {
        const int64_t base = t * kCoders;
        const int last = (int)((n - base < kCoders ? n - base : kCoders) - 1);
        for (int c = last; c >= 0; --c) {
            const uint32_t b = src[base + c], fb = f[b];
            uint32_t x = state[c];
            if ((uint64_t)x >= ((uint64_t)fb << (32 - kProbBits))) {
                words[--head] = (uint16_t)x;
                x >>= 16;
            }
            state[c] = (x / fb) * kProbTotal + x % fb + cum[b];
        }
    }
    const int64_t nw = kTile - head;
    int64_t size;
    if (128 + 2 * nw < n) {
        for (int c = 0; c < kCoders; ++c)
            for (int k = 0; k < 4; ++k) dst[4 * c + k] = (uint8_t)(state[c] >> (8 * k));
        for (int64_t w = 0; w < nw; ++w) {
            dst[128 + 2 * w] = (uint8_t)words[head + w];
            dst[128 + 2 * w + 1] = (uint8_t)(words[head + w] >> 8);
        }
        size = 128 + 2 * nw;
        rec.n_words = (uint32_t)nw;
        rec.flags = 0;
    } else {
        memcpy(dst, src, (size_t)n);
        size = n;
        rec.n_words = 0;
        rec.flags = 1;
    }
    const int64_t padded = (size + 15) / 16 * 16;
    memset(dst + size, 0, (size_t)(padded - size));
    rec.n_bytes = (uint32_t)n;
    rec.adler = adler32(src, n);
    rec.reserved[0] = rec.reserved[1] = 0;
    return padded;
}

// One expert into its stretch of the blob; records carry offsets relative to
// the stretch. Returns the stretch's packed size.
int64_t encode_expert(const Layout &L, const uint8_t *const arr[6], int64_t e, uint8_t *out,
                      moe_tile_rec *rec, uint16_t *tab, std::vector<uint8_t> &canon,
                      std::vector<uint16_t> &words) {
    int64_t pos = 0;
    for (int a = 0; a < 6; ++a) {
        const uint8_t *src = arr[a] + e * L.bytes[a];
        const int64_t n = L.bytes[a];
        uint64_t count[256] = {0};
        if (a & 1) {  // scales: kept as they are
            memcpy(canon.data(), src, (size_t)n);
        } else {
            for (int64_t i = 0; i < n; ++i) canon[i] = kCanon.to[src[i]];
        }
        for (int64_t i = 0; i < n; ++i) count[canon[i]]++;
        uint16_t *f = tab + a * 256;
        quantise(count, (uint64_t)n, f);
        uint32_t cum[256];
        for (int b = 0, c = 0; b < 256; c += f[b], ++b) cum[b] = (uint32_t)c;
        for (int64_t t = L.first[a]; t < L.first[a + 1]; ++t) {
            const int64_t p = (t - L.first[a]) * kTile;
            const int64_t len = n - p < kTile ? n - p : kTile;
            rec[t].offset_lo = (uint32_t)pos;
            rec[t].offset_hi = (uint32_t)((uint64_t)pos >> 32);
            pos += store_tile(canon.data() + p, len, f, cum, words.data(), out + pos, rec[t]);
        }
    }
    return pos;
}

}  // namespace

MOE_API int32_t moe_store_tiles_per_expert(int32_t d_model, int32_t d_ff) {
    Layout L;
    return layout_of(d_model, d_ff, L) ? (int32_t)L.first[6] : -1;
}

MOE_API int64_t moe_store_blob_bound(int32_t n_experts, int32_t d_model, int32_t d_ff) {
    Layout L;
    if (n_experts <= 0 || !layout_of(d_model, d_ff, L)) return -1;
    return (int64_t)n_experts * L.stride;
}

MOE_API int moe_store_encode(int32_t n_experts, int32_t d_model, int32_t d_ff,
                             const moe_weights *host_w, uint8_t *blob, int64_t blob_cap,
                             int64_t *blob_bytes, moe_tile_rec *tiles, uint16_t *tables,
                             int32_t n_threads) {
    Layout L;
    if (n_experts <= 0 || !layout_of(d_model, d_ff, L) || !host_w || !blob || !blob_bytes ||
        !tiles || !tables)
        return MOE_ERR_INVALID_ARG;
    const uint8_t *arr[6] = {host_w->gate_q, host_w->gate_s, host_w->up_q,
                             host_w->up_s, host_w->down_q, host_w->down_s};
    for (const uint8_t *p : arr)
        if (!p) return MOE_ERR_INVALID_ARG;
    if (blob_cap < (int64_t)n_experts * L.stride) return MOE_ERR_INVALID_ARG;
    int workers = n_threads > 0 ? n_threads : (int)std::thread::hardware_concurrency();
    if (workers < 1) workers = 1;
    if (workers > n_experts) workers = n_experts;
    const int64_t tpe = L.first[6];
    std::vector<int64_t> packed((size_t)n_experts, 0);
    std::atomic<int> next{0};
    auto work = [&]() {
        std::vector<uint8_t> canon((size_t)L.bytes[0]);
        std::vector<uint16_t> words((size_t)kTile);
        for (int e; (e = next.fetch_add(1)) < n_experts;)
            packed[e] = encode_expert(L, arr, e, blob + (int64_t)e * L.stride, tiles + e * tpe,
                                      tables + (int64_t)e * 6 * 256, canon, words);
    };
    std::vector<std::thread> pool;
    for (int i = 1; i < workers; ++i) pool.emplace_back(work);
    work();
    for (auto &t : pool) t.join();
    // pack the stretches in expert order (each moves down, never past an
    // unmoved one) and turn the offsets absolute
    int64_t off = 0;
    for (int64_t e = 0; e < n_experts; ++e) {
        if (off != e * L.stride) memmove(blob + off, blob + e * L.stride, (size_t)packed[e]);
        for (int64_t t = 0; t < tpe; ++t) {
            moe_tile_rec &r = tiles[e * tpe + t];
            const uint64_t o = ((uint64_t)r.offset_hi << 32 | r.offset_lo) + (uint64_t)off;
            r.offset_lo = (uint32_t)o;
            r.offset_hi = (uint32_t)(o >> 32);
        }
        off += packed[e];
    }
    *blob_bytes = off;
    return MOE_OK;
}
