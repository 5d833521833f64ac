// GPU decode of compressed-store experts straight into cache slots (the
// pages' GPU-rANS expert store: Moonshine GitHub README, "Expert-stream
// compression" / "MZG2 production store"; format stated in moe.h).
//
// One warp decodes one 16 KiB tile: it stages the stored tile from host
// memory into its shared memory with 16-byte loads (coalesced reads over the
// host link; the warps of a CTA read neighbouring tiles), then its 32 lanes run the tile's 32 interleaved rANS coders in
// lock step, one output byte per lane per step, so each step stores 32
// consecutive bytes; lanes that renormalise take the next words of the shared
// stream in lane order (ballot + prefix count). The warp keeps the decode
// table (slot-to-byte lookup of 4096 entries plus packed f/cum per byte) of
// its current (expert, array) in shared memory; a CTA's warps share a
// contiguous run of tiles, so a table is rebuilt only where the run crosses
// an array. Every tile
// is checked: its record against the layer shape and the blob, the table's
// total, the coders' final states, the word count and the Adler-32 of the
// bytes written; a failed check is recorded (MOE_ERR_CORRUPT_TILE) and no
// access ever leaves the tile's stored bytes or its slot.
#include "common.cuh"
#include "kernels.h"

#define FULL_MASK 0xFFFFFFFFu

namespace {

constexpr int SD_TILE = 16384;
constexpr int SD_WARPS = 8;
constexpr int SD_LUT = 4096;
constexpr int SD_WARP_SMEM = SD_TILE + SD_LUT + 256 * 4;  // stage, lookup, f | cum << 16
constexpr int SD_SMEM = SD_WARPS * SD_WARP_SMEM;
constexpr uint32_t SD_LOW = 1u << 16;

// Warp-wide: decode table of one (expert, array) from its 256 frequencies.
// False (warp-uniform) when they do not sum to 4096.
__device__ bool build_table(const uint16_t *__restrict__ f, uint8_t *lut, uint32_t *fc, int lane) {
    const uint4 v = *reinterpret_cast<const uint4 *>(f + 8 * lane);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t fl[8], mine = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        fl[k] = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
        mine += fl[k];
    }
    uint32_t incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(FULL_MASK, incl, o);
        if (lane >= o) incl += u;
    }
    const uint32_t total = __shfl_sync(FULL_MASK, incl, 31);
    uint32_t c = incl - mine;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        fc[8 * lane + k] = fl[k] | (c << 16);
        c += fl[k];
    }
    __syncwarp();
    if (total != (uint32_t)SD_LUT) return false;
    for (int b = 0; b < 256; ++b) {
        const uint32_t e = fc[b], fb = e & 0xFFFFu, cb = e >> 16;
        for (uint32_t q = lane; q < fb; q += 32) lut[cb + q] = (uint8_t)b;
    }
    __syncwarp();
    return true;
}

// One work item (a tile of one expert's copy into one slot), checked against
// the layer shape and the blob before anything is read through it.
struct Item {
    int e, s, a, ta, n;
    bool raw;
    int status;          // 0, MOE_ERR_BAD_INDEX or MOE_ERR_CORRUPT_TILE
    int64_t off, padded;
    uint32_t n_words, adler;
};

__device__ __forceinline__ Item plan_item(const MoeStoreJob &j, int64_t w) {
    Item it;
    const int m = (int)(w / j.tpe), t = (int)(w - (int64_t)m * j.tpe);
    int a = 0;
    while (a < 5 && t >= j.first[a + 1]) ++a;
    it.a = a;
    it.ta = t - j.first[a];
    it.e = j.experts[m];
    it.s = j.slots[m];
    it.status = 0;
    if (it.e < 0 || it.e >= j.E || it.s < 0 || it.s >= j.n_slots) {
        it.status = MOE_ERR_BAD_INDEX;
        return it;
    }
    const moe_tile_rec rec = j.tiles[(int64_t)it.e * j.tpe + t];
    const int64_t left = j.bytes[a] - (int64_t)it.ta * SD_TILE;
    it.n = (int)(left < SD_TILE ? left : SD_TILE);
    it.raw = rec.flags & 1u;
    it.off = (int64_t)((uint64_t)rec.offset_hi << 32 | rec.offset_lo);
    const int64_t size = it.raw ? (int64_t)rec.n_bytes : 128 + 2 * (int64_t)rec.n_words;
    it.padded = (size + 15) & ~(int64_t)15;
    it.n_words = rec.n_words;
    it.adler = rec.adler;
    const bool ok = rec.n_bytes == (uint32_t)it.n && (rec.flags & ~1u) == 0 &&
                    (it.raw ? rec.n_words == 0 : size < it.n) && it.off >= 0 &&
                    (it.off & 15) == 0 && it.off + it.padded <= j.blob_bytes;
    if (!ok) it.status = MOE_ERR_CORRUPT_TILE;  // then padded <= 16 KiB is not known
    return it;
}

// Copies a checked item's stored bytes (<= 16 KiB = 32 16-byte chunks per
// lane) into the warp's stage buffer: every load of the tile is issued before
// the first store, so a warp keeps its whole tile in flight on the host link.
__device__ __forceinline__ void stage_item(const MoeStoreJob &j, const Item &it, uint4 *buf,
                                           int lane) {
    const uint4 *src = reinterpret_cast<const uint4 *>(j.blob + it.off);
    const int chunks = (int)(it.padded >> 4);
    uint4 v[SD_TILE / 16 / 32];
#pragma unroll
    for (int k = 0; k < SD_TILE / 16 / 32; ++k) {
        const int c = k * 32 + lane;
        if (c < chunks) v[k] = src[c];
    }
#pragma unroll
    for (int k = 0; k < SD_TILE / 16 / 32; ++k) {
        const int c = k * 32 + lane;
        if (c < chunks) buf[c] = v[k];
    }
    __syncwarp();
}

__global__ void __launch_bounds__(SD_WARPS * 32, 1) moe_store_decode_kernel(MoeStoreJob j) {
    extern __shared__ __align__(16) unsigned char sd_smem[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned char *mine = sd_smem + wid * SD_WARP_SMEM;
    uint4 *stage = reinterpret_cast<uint4 *>(mine);
    uint8_t *lut = mine + SD_TILE;
    uint32_t *fc = reinterpret_cast<uint32_t *>(mine + SD_TILE + SD_LUT);

    int n_items = j.n_dev ? *j.n_dev : j.n_host;
    if (n_items < 0) n_items = 0;
    if (n_items > j.max_items) n_items = j.max_items;
    // Each CTA takes a contiguous run of tiles and its warps interleave
    // through it (warp k takes tiles k, k + SD_WARPS, ...), so the CTA reads
    // neighbouring stored tiles -- one sequential stream through the blob --
    // and tables still change only where the run crosses an array.
    const int64_t W = (int64_t)n_items * j.tpe;
    const int64_t c0 = (int64_t)blockIdx.x * W / gridDim.x;
    const int64_t c1 = ((int64_t)blockIdx.x + 1) * W / gridDim.x;
    int key = -1;
    bool key_ok = false;
    for (int64_t w = c0 + wid; w < c1; w += SD_WARPS) {
        const Item it = plan_item(j, w);
        if (it.status != 0) {
            if (lane == 0) moe_flag(j.status, it.status);
            continue;
        }
        if (!it.raw && it.e * 6 + it.a != key) {
            key = it.e * 6 + it.a;
            key_ok = build_table(j.tables + (int64_t)key * 256, lut, fc, lane);
        }
        if (!it.raw && !key_ok) {
            if (lane == 0) moe_flag(j.status, MOE_ERR_CORRUPT_TILE);
            continue;
        }
        stage_item(j, it, stage, lane);
        const uint8_t *sb = reinterpret_cast<const uint8_t *>(stage);
        const int n = it.n;
        uint8_t *out = j.dst[it.a] + (int64_t)it.s * j.bytes[it.a] + (int64_t)it.ta * SD_TILE;
        // Adler-32 sums per lane: at most 512 bytes of 255 each and weights
        // n - i <= 16384, so both fit 32 bits before the warp reduction
        uint32_t asum = 0, bsum = 0;
        bool bad = false;
        if (it.raw) {
            for (int i = lane; i < n; i += 32) {
                const uint32_t v = sb[i];
                out[i] = (uint8_t)v;
                asum += v;
                bsum += (uint32_t)(n - i) * v;
            }
        } else {
            uint32_t x = reinterpret_cast<const uint32_t *>(sb)[lane];
            const uint16_t *words = reinterpret_cast<const uint16_t *>(sb + 128);
            const uint32_t nw = it.n_words;
            uint32_t r = 0;
            for (int i0 = 0; i0 < n; i0 += 32) {
                const int i = i0 + lane;
                const bool act = i < n;
                uint32_t v = 0;
                if (act) {
                    const uint32_t q = x & (uint32_t)(SD_LUT - 1);
                    v = lut[q];
                    const uint32_t e = fc[v];
                    x = (e & 0xFFFFu) * (x >> 12) + q - (e >> 16);
                }
                const bool need = act && x < SD_LOW;
                const uint32_t mask = __ballot_sync(FULL_MASK, need);
                if (need) {
                    const uint32_t k = r + __popc(mask & lanemask_lt());
                    x = (x << 16) | (k < nw ? (uint32_t)words[k] : 0u);
                }
                r += __popc(mask);
                if (act) {
                    out[i] = (uint8_t)v;
                    asum += v;
                    bsum += (uint32_t)(n - i) * v;
                }
            }
            bad = x != SD_LOW || r != nw;
        }
        unsigned long long bs = bsum;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            asum += __shfl_xor_sync(FULL_MASK, asum, o);
            bs += __shfl_xor_sync(FULL_MASK, bs, o);
        }
        bad = __any_sync(FULL_MASK, bad);
        if (lane == 0) {
            const uint32_t A = (1u + asum) % 65521u;
            const uint32_t B = (uint32_t)(((unsigned long long)n + bs) % 65521ull);
            if (bad || ((B << 16) | A) != it.adler) moe_flag(j.status, MOE_ERR_CORRUPT_TILE);
        }
        __syncwarp();  // the stage is rewritten by the next tile
    }
}

}  // namespace

bool moe_store_job_shape(int D, int F, MoeStoreJob &j) {
    if (D <= 0 || F <= 0 || D % 32 != 0 || F % 32 != 0) return false;  // MXFP4 layouts
    const int64_t n = (int64_t)D * F;
    j.first[0] = 0;
    for (int a = 0; a < 6; ++a) {
        j.bytes[a] = (a & 1) ? n / 32 : n / 2;
        j.first[a + 1] = j.first[a] + (int)((j.bytes[a] + SD_TILE - 1) / SD_TILE);
    }
    j.tpe = j.first[6];
    return true;
}

cudaError_t moe_launch_store_decode(const MoeStoreJob &j, int nsm, cudaStream_t st) {
    // set on every launch (a host-side call): per device and thread-safe
    cudaError_t e = cudaFuncSetAttribute(moe_store_decode_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SD_SMEM);
    if (e != cudaSuccess) return e;
    moe_store_decode_kernel<<<nsm, SD_WARPS * 32, SD_SMEM, st>>>(j);
    return cudaGetLastError();
}
