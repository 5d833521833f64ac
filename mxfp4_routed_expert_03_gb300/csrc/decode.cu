// Token-major expert FFN (decode): streams only the active experts' packed
// MXFP4 codes with 128-bit loads (16 bytes = one 32-element MX block of one
// row) and reduces on CUDA cores with fp32 accumulation, then combines the
// per-slot expert outputs back to token order deterministically.
//
// Decode is token-major and reads only the selected experts (Moonshine README,
// "How the engine works"; Moonshine GitHub README, "Decode"); the per-expert
// SwiGLU FFN on MXFP4 weights is the routed expert FFN (MoonTail,
// requester/volunteer table) and the final step is the MoE tail's weighted
// reduction (Moonshine README, "Run layer-major prefill").
//
// Arithmetic: an E2M1 pair is converted to f16x2 exactly (cvt.rn.f16x2.e2m1x2);
// each 32-element block is reduced with exact f16 x f16 products accumulated
// in fp32 (fma.rn.f32.f16), multiplied by its E8M0 scale and added to the
// row's fp32 sum. Activations enter as f16 with one power-of-two exponent per
// 32-element block of x, chosen so that the block's largest magnitude lands in
// [2^14, 2^15): every bf16 value, from subnormals to 3.4e38, then fits f16
// without overflow, and every element within 2^-28 of its block's maximum
// converts exactly (bf16 has 8 significant bits, f16 11). The block's
// exponent multiplies its partial sum together with the weight scale. The
// intermediate h is stored the same way, as f16 with one power-of-two
// exponent per 32 consecutive rows of F, which lets the down projection use
// the same exact f16 x f16 -> fp32 inner loop.
//
// Work split: persistent grids, each CTA walking a contiguous range of the
// (active expert, row) space, so every weight row is read exactly once and
// the grid stays balanced for any number of active experts.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"

#define FULL_MASK 0xFFFFFFFFu

namespace {

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
        : "=r"(r)
        : "r"(byte));
    return r;
}

// acc + sum over the 8 codes of word w (element 2i in the low nibble of byte i)
// times the 8 f16 activations in xa..xd: products exact, sums in fp32.
__device__ __forceinline__ float word_dot(uint32_t w, uint32_t xa, uint32_t xb, uint32_t xc,
                                          uint32_t xd, float acc) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t.reg .b32 h0, h1, h2, h3;\n\t"
        ".reg .f16 wl, wh, al, ah;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h0, b0;\n\tcvt.rn.f16x2.e2m1x2 h1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 h2, b2;\n\tcvt.rn.f16x2.e2m1x2 h3, b3;\n\t"
        "mov.b32 {wl, wh}, h0;\n\tmov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t"
        "mov.b32 {wl, wh}, h1;\n\tmov.b32 {al, ah}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t"
        "mov.b32 {wl, wh}, h2;\n\tmov.b32 {al, ah}, %4;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t"
        "mov.b32 {wl, wh}, h3;\n\tmov.b32 {al, ah}, %5;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(xa), "r"(xb), "r"(xc), "r"(xd));
    return acc;
}

// Dot product of one 32-element MX block (16 code bytes) with 32 f16
// activations held as four 16-byte chunks; fp32 result before the block scale.
__device__ __forceinline__ float block_dot_f16(const uint4 &q, const uint4 *xs) {
    const uint4 x0 = xs[0], x1 = xs[1], x2 = xs[2], x3 = xs[3];
    float a0 = word_dot(q.x, x0.x, x0.y, x0.z, x0.w, 0.f);
    float a1 = word_dot(q.y, x1.x, x1.y, x1.z, x1.w, 0.f);
    a0 = word_dot(q.z, x2.x, x2.y, x2.z, x2.w, a0);
    a1 = word_dot(q.w, x3.x, x3.y, x3.z, x3.w, a1);
    return a0 + a1;
}

// The same for four E4M3 codes (one word, element i in byte i): each byte
// pair converts exactly to f16x2 (E4M3's range and 4 significant bits fit f16).
__device__ __forceinline__ float word_dot_e4m3(uint32_t w, uint32_t xa, uint32_t xb, float acc) {
    asm("{\n\t.reg .b16 p0, p1;\n\t.reg .b32 h0, h1;\n\t"
        ".reg .f16 wl, wh, al, ah;\n\t"
        "mov.b32 {p0, p1}, %1;\n\t"
        "cvt.rn.f16x2.e4m3x2 h0, p0;\n\tcvt.rn.f16x2.e4m3x2 h1, p1;\n\t"
        "mov.b32 {wl, wh}, h0;\n\tmov.b32 {al, ah}, %2;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t"
        "mov.b32 {wl, wh}, h1;\n\tmov.b32 {al, ah}, %3;\n\t"
        "fma.rn.f32.f16 %0, wl, al, %0;\n\tfma.rn.f32.f16 %0, wh, ah, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(xa), "r"(xb));
    return acc;
}

// One 32-element block of weights as the kernels load it: 16 bytes of packed
// E2M1 codes (MXFP4) or 32 bytes of E4M3 codes (FP8), with the block's scale.
template <bool F8>
struct WBlock {
    uint4 q0, q1;  // q1 used by FP8 only
};

// Block b of a weight row: MXFP4 rows are K/2 bytes with one E8M0 scale byte
// per block; FP8 rows are K bytes and take the fp32 scale of their
// 128 x 128 block (sc_row: the row's row of block scales, K/128 entries).
template <bool F8>
__device__ __forceinline__ void load_block(const uint8_t *__restrict__ row, const void *sc_row, int b,
                                           WBlock<F8> &w, float &sc) {
    if constexpr (F8) {
        w.q0 = __ldg((const uint4 *)row + 2 * b);
        w.q1 = __ldg((const uint4 *)row + 2 * b + 1);
        sc = __ldg((const float *)sc_row + (b >> 2));
    } else {
        w.q0 = __ldg((const uint4 *)row + b);
        sc = e8m0_to_f32(__ldg((const uint8_t *)sc_row + b));
    }
}

// Dot product of a weight block with 32 f16 activations (four 16-byte chunks).
template <bool F8>
__device__ __forceinline__ float block_dot(const WBlock<F8> &w, const uint4 *xs) {
    if constexpr (F8) {
        const uint4 x0 = xs[0], x1 = xs[1], x2 = xs[2], x3 = xs[3];
        float a0 = word_dot_e4m3(w.q0.x, x0.x, x0.y, 0.f);
        float a1 = word_dot_e4m3(w.q0.y, x0.z, x0.w, 0.f);
        a0 = word_dot_e4m3(w.q0.z, x1.x, x1.y, a0);
        a1 = word_dot_e4m3(w.q0.w, x1.z, x1.w, a1);
        a0 = word_dot_e4m3(w.q1.x, x2.x, x2.y, a0);
        a1 = word_dot_e4m3(w.q1.y, x2.z, x2.w, a1);
        a0 = word_dot_e4m3(w.q1.z, x3.x, x3.y, a0);
        a1 = word_dot_e4m3(w.q1.w, x3.z, x3.w, a1);
        return a0 + a1;
    } else {
        return block_dot_f16(w.q0, xs);
    }
}

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t v) {
    __half2 hv = *reinterpret_cast<__half2 *>(&v);
    return __half22float2(hv);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.f + expf(-z)); }

// Flat-index bounds of expert e's rows, validated.
__device__ __forceinline__ bool segment_of(int a, int E, int n_rows, const int32_t *active,
                                          const int32_t *offsets, int &e, int &s0, int &n,
                                          int *status) {
    if (a >= active[0]) return false;
    e = active[1 + a];
    if (e < 0 || e >= E) { moe_flag(status, MOE_ERR_BAD_INDEX); return false; }
    s0 = offsets[e];
    int s1 = offsets[e + 1];
    if (s0 < 0 || s1 < s0 || s1 > n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); return false; }
    n = s1 - s0;
    return true;
}

}  // namespace

// Shared-memory activation rows: each 32-element block (64 bytes of f16) is
// stored with 16 bytes of padding, so the 16-byte reads of eight consecutive
// lanes (one block each) fall in distinct bank groups. For x the padding's
// first 4 bytes hold the block's scale 2^ex (fp32).
constexpr int kBlkStride = 80;   // bytes per staged block
constexpr int kBlkScale = 64;    // byte offset of a staged x block's scale
constexpr int kStageTok = 4;     // tokens staged at once

// Exponent ex (clamped to [-126, 113]) with amax * 2^-ex in [2^14, 2^15) for a
// finite non-zero amax; 0 for zero, infinity or NaN.
__device__ __forceinline__ int f16_block_exp(float amax) {
    const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF);
    if (amax == 0.f || e == 255) return 0;
    int ex = (e == 0 ? -126 : e - 127) - 14;  // fp32 subnormal amax: below 2^-126
    return max(-126, min(113, ex));
}

__device__ __forceinline__ float exp2_int(int ex) {  // 2^ex for ex in [-126, 127]
    return __uint_as_float((uint32_t)(ex + 127) << 23);
}

// ---------------------------------------------------------------------------
// Gate/up + SwiGLU. The (active expert, 32-row block of F) steps are split
// into contiguous ranges, one per CTA, so a CTA restages the activations
// (bf16 -> f16 into shared memory) only when its expert changes. In a step
// the 8 warps compute g, u for the 32 rows (lanes grouped LPR per row, each
// lane owning PER_LANE MX blocks), then one warp per token stores the 32
// values of h = silu(g) * u as f16 with their shared power-of-two exponent.
// ---------------------------------------------------------------------------
template <int PER_LANE, bool F8>
__global__ void __launch_bounds__(256, F8 ? 1 : 2) moe_decode_gateup_kernel(
    int D, int F, int E, int k, int n_rows, const uint16_t *__restrict__ x,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const int32_t *__restrict__ active, const uint8_t *__restrict__ gate_q,
    const uint8_t *__restrict__ gate_s, const uint8_t *__restrict__ up_q,
    const uint8_t *__restrict__ up_s, __half *__restrict__ h16, int8_t *__restrict__ hexp,
    int *status) {
    constexpr int NT = 2, NW = 8;
    extern __shared__ __align__(16) unsigned char xs[];  // [kStageTok][nblk][kBlkStride]
    __shared__ float s_h[kStageTok][32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nblk = D / 32;
    const int LPR = nblk / PER_LANE;
    const int RPW = 32 / LPR;
    const int sub = lane % LPR, grp = lane / LPR;
    // bytes per weight row; scale entries per row (MXFP4: per 32-block bytes;
    // FP8: a row of 128 x 128 block scales, shared by 128 rows)
    const size_t qrow = F8 ? (size_t)D : (size_t)D / 2, srow = F8 ? (size_t)D / 128 : (size_t)nblk;
    int n_active = active[0];
    if (n_active < 0 || n_active > E) {
        if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        return;
    }
    const int spe = F / 32;  // steps per expert
    const long long total = (long long)n_active * spe;
    const long long b0 = total * blockIdx.x / gridDim.x, b1 = total * (blockIdx.x + 1) / gridDim.x;
    int staged_a = -1, staged_g0 = -1;
    for (long long step = b0; step < b1; ++step) {
        const int a = (int)(step / spe), f_base = (int)(step % spe) * 32;
        int e, s0, n;
        if (!segment_of(a, E, n_rows, active, offsets, e, s0, n, status)) continue;
        const uint8_t *gq = gate_q + (size_t)e * F * qrow, *uq = up_q + (size_t)e * F * qrow;
        // the expert's scales: MXFP4 bytes [F][nblk]; FP8 floats [F/128][D/128]
        const size_t es = F8 ? (size_t)e * (F / 128) * srow * 4 : (size_t)e * F * srow;
        const uint8_t *gs = gate_s + es, *us = up_s + es;
        for (int g0 = 0; g0 < n; g0 += kStageTok) {
            const int ns = min(kStageTok, n - g0);
            if (a != staged_a || g0 != staged_g0) {
                __syncthreads();
                // one 32-element block of token j per thread iteration: 32 bf16
                // -> 32 f16 scaled by 2^-ex, and the block's scale 2^ex
                for (int i = threadIdx.x; i < ns * nblk; i += blockDim.x) {
                    const int j = i / nblk, b = i % nblk;
                    int fl = perm[s0 + g0 + j];
                    if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
                    const uint4 *src = (const uint4 *)(x + (size_t)(fl / k) * D) + 4 * b;
                    uint32_t w[16];
                    float amax = 0.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 v = __ldg(src + c);
                        w[4 * c] = v.x;
                        w[4 * c + 1] = v.y;
                        w[4 * c + 2] = v.z;
                        w[4 * c + 3] = v.w;
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[q] << 16)),
                                                 fabsf(__uint_as_float(w[q] & 0xFFFF0000u))));
                    const int ex = f16_block_exp(amax);
                    const float inv = exp2_int(-ex);  // exact: a power of two times bf16
                    unsigned char *dst = xs + ((size_t)j * nblk + b) * kBlkStride;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint32_t u = w[4 * c + q];
                            __half2 hh = __floats2half2_rn(__uint_as_float(u << 16) * inv,
                                                           __uint_as_float(u & 0xFFFF0000u) * inv);
                            o[q] = *reinterpret_cast<uint32_t *>(&hh);
                        }
                        *(uint4 *)(dst + 16 * c) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    *(float *)(dst + kBlkScale) = exp2_int(ex);
                }
                __syncthreads();
                staged_a = a;
                staged_g0 = g0;
            }
            for (int rl = wid * RPW + grp; rl - grp < 32; rl += NW * RPW) {
                const bool row_ok = rl < 32;
                const int f = f_base + (row_ok ? rl : 0);
                WBlock<F8> gqv[PER_LANE], uqv[PER_LANE];
                float gsc[PER_LANE], usc[PER_LANE];
                const size_t so = F8 ? (size_t)(f / 128) * srow * 4 : (size_t)f * srow;
#pragma unroll
                for (int p = 0; p < PER_LANE; ++p) {
                    const int b = sub + LPR * p;
                    load_block<F8>(gq + (size_t)f * qrow, gs + so, b, gqv[p], gsc[p]);
                    load_block<F8>(uq + (size_t)f * qrow, us + so, b, uqv[p], usc[p]);
                }
                for (int j0 = 0; j0 < ns; j0 += NT) {
                    const int nt = min(NT, ns - j0);
                    float ag[NT], au[NT];
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        ag[j] = 0.f;
                        au[j] = 0.f;
                        if (j < nt) {
#pragma unroll
                            for (int p = 0; p < PER_LANE; ++p) {
                                const unsigned char *xbb =
                                    xs + ((size_t)(j0 + j) * nblk + sub + LPR * p) * kBlkStride;
                                const uint4 *xb = (const uint4 *)xbb;
                                const float xsc = *(const float *)(xbb + kBlkScale);
                                ag[j] = fmaf(block_dot<F8>(gqv[p], xb), gsc[p] * xsc, ag[j]);
                                au[j] = fmaf(block_dot<F8>(uqv[p], xb), usc[p] * xsc, au[j]);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1) {
                            if (off < LPR) {
                                ag[j] += __shfl_xor_sync(FULL_MASK, ag[j], off);
                                au[j] += __shfl_xor_sync(FULL_MASK, au[j], off);
                            }
                        }
                    }
                    if (row_ok && sub == 0) {
#pragma unroll
                        for (int j = 0; j < NT; ++j)
                            if (j < nt) s_h[j0 + j][rl] = silu_f(ag[j]) * au[j];
                    }
                }
            }
            __syncthreads();
            if (wid < ns) {
                const float v = s_h[wid][lane];
                float amax = fabsf(v);
#pragma unroll
                for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL_MASK, amax, off));
                // exponent so that amax / 2^ex lies in [2^14, 2^15): f16-safe, 11 significant bits
                int ex = ((int)((__float_as_uint(amax) >> 23) & 0xFF)) - 127 - 14;
                if (amax == 0.f || !(amax < INFINITY)) ex = 0;
                ex = max(-126, min(127, ex));
                const float sc = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-ex
                const size_t slot = (size_t)(s0 + g0 + wid);
                h16[slot * F + f_base + lane] = __float2half_rn(v * sc);
                if (lane == 0) hexp[slot * (F / 32) + f_base / 32] = (int8_t)ex;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Down projection: y[slot][d] = sum_f W_down[e][d][f] * h[slot][f] (fp32).
// Units of consecutive rows of one expert are split into contiguous ranges
// per CTA; h of the expert's slots is staged (padded blocks) when the expert
// changes. Each warp issues all loads of RG groups of RPW rows before any
// arithmetic.
// ---------------------------------------------------------------------------
template <int PER_LANE, bool F8>
__global__ void __launch_bounds__(256, F8 ? 1 : 2) moe_decode_down_kernel(
    int D, int F, int E, int n_rows, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ active, const uint8_t *__restrict__ down_q,
    const uint8_t *__restrict__ down_s, const __half *__restrict__ h16,
    const int8_t *__restrict__ hexp, float *__restrict__ y, int *status) {
    constexpr int NT = 2, NW = 8, RG = 2;
    extern __shared__ __align__(16) unsigned char hs[];  // [kStageTok][nblk][kBlkStride]
    __shared__ float s_hsc[kStageTok][MOE_MAX_DFF / 32];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nblk = F / 32;
    const int LPR = nblk / PER_LANE;
    const int RPW = 32 / LPR;
    const int sub = lane % LPR, grp = lane / LPR;
    const size_t qrow = F8 ? (size_t)F : (size_t)F / 2, srow = F8 ? (size_t)F / 128 : (size_t)nblk;
    int n_active = active[0];
    if (n_active < 0 || n_active > E) {
        if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        return;
    }
    const int unit = NW * RG * RPW;  // rows per unit (D is a multiple of 128)
    const int upe = (D + unit - 1) / unit;
    const long long total = (long long)n_active * upe;
    const long long b0 = total * blockIdx.x / gridDim.x, b1 = total * (blockIdx.x + 1) / gridDim.x;
    int staged_a = -1, staged_g0 = -1;
    for (long long u = b0; u < b1; ++u) {
        const int a = (int)(u / upe), d_base = (int)(u % upe) * unit;
        int e, s0, n;
        if (!segment_of(a, E, n_rows, active, offsets, e, s0, n, status)) continue;
        const uint8_t *dq = down_q + (size_t)e * D * qrow;
        const uint8_t *ds = down_s + (F8 ? (size_t)e * (D / 128) * srow * 4 : (size_t)e * D * srow);
        int drow[RG];
        bool ok[RG];
        WBlock<F8> qv[RG][PER_LANE];
        float sc[RG][PER_LANE];
#pragma unroll
        for (int r = 0; r < RG; ++r) {
            drow[r] = d_base + (wid * RG + r) * RPW + grp;
            ok[r] = drow[r] < D;
            const int d = ok[r] ? drow[r] : 0;
            const size_t so = F8 ? (size_t)(d / 128) * srow * 4 : (size_t)d * srow;
#pragma unroll
            for (int p = 0; p < PER_LANE; ++p)
                load_block<F8>(dq + (size_t)d * qrow, ds + so, sub + LPR * p, qv[r][p], sc[r][p]);
        }
        for (int g0 = 0; g0 < n; g0 += kStageTok) {
            const int ns = min(kStageTok, n - g0);
            if (a != staged_a || g0 != staged_g0) {
                __syncthreads();
                for (int i = threadIdx.x; i < ns * nblk * 4; i += blockDim.x) {
                    const int j = i / (nblk * 4), r = i % (nblk * 4);
                    const uint4 v = __ldg((const uint4 *)(h16 + (size_t)(s0 + g0 + j) * F) + r);
                    *(uint4 *)(hs + ((size_t)j * nblk + r / 4) * kBlkStride + (r % 4) * 16) = v;
                }
                for (int i = threadIdx.x; i < ns * nblk; i += blockDim.x) {
                    const int j = i / nblk, b = i % nblk;
                    const int ex = __ldg(hexp + (size_t)(s0 + g0 + j) * nblk + b);
                    s_hsc[j][b] = __uint_as_float((uint32_t)(ex + 127) << 23);  // 2^ex
                }
                __syncthreads();
                staged_a = a;
                staged_g0 = g0;
            }
            for (int j0 = 0; j0 < ns; j0 += NT) {
                const int nt = min(NT, ns - j0);
                float acc[RG][NT];
#pragma unroll
                for (int r = 0; r < RG; ++r)
#pragma unroll
                    for (int j = 0; j < NT; ++j) acc[r][j] = 0.f;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    if (j < nt) {
#pragma unroll
                        for (int p = 0; p < PER_LANE; ++p) {
                            const int b = sub + LPR * p;
                            const uint4 *hb =
                                (const uint4 *)(hs + ((size_t)(j0 + j) * nblk + b) * kBlkStride);
                            const float hsc = s_hsc[j0 + j][b];
#pragma unroll
                            for (int r = 0; r < RG; ++r)
                                acc[r][j] = fmaf(block_dot<F8>(qv[r][p], hb), sc[r][p] * hsc, acc[r][j]);
                        }
                    }
                }
#pragma unroll
                for (int r = 0; r < RG; ++r)
#pragma unroll
                    for (int j = 0; j < NT; ++j)
#pragma unroll
                        for (int off = 1; off < 32; off <<= 1)
                            if (off < LPR) acc[r][j] += __shfl_xor_sync(FULL_MASK, acc[r][j], off);
                if (sub == 0) {
#pragma unroll
                    for (int r = 0; r < RG; ++r)
                        if (ok[r])
#pragma unroll
                            for (int j = 0; j < NT; ++j)
                                if (j < nt) y[(size_t)(s0 + g0 + j0 + j) * D + drow[r]] = acc[r][j];
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Combine: out[t][d] = bf16( sum_j w[t][j] * y[inv[t*k+j]][d] [+ shared[t][d]] ),
// j ascending, the shared expert's output (weight 1.0) added last.
// ---------------------------------------------------------------------------
// Y: the row element type, float or bf16 bits (uint16_t). One block of 128
// threads per (token, 128 x V columns); a thread takes V = 16 bytes of
// each row (8 bf16 or 4 fp32 columns). The token's k slots and weights are
// read once per block into shared memory, so each thread's k row loads are
// independent of one another and issue back to back (the loop is unrolled):
// the loads of one row per iteration behind a slot read made this kernel
// latency-bound at ~4 TB/s. D is a multiple of 32 (the ABI's shape check).
template <typename Y>
__global__ void __launch_bounds__(128) moe_combine_slots_kernel(int T, int D, int k, int n_rows,
                                                                const float *__restrict__ topk_w,
                                                                const int32_t *__restrict__ inv,
                                                                const Y *__restrict__ y,
                                                                const float *__restrict__ shared,
                                                                uint16_t *__restrict__ out,
                                                                int *status) {
    constexpr int V = 16 / (int)sizeof(Y);  // columns per thread
    __shared__ int s_slot[MOE_MAX_TOPK];
    __shared__ float s_w[MOE_MAX_TOPK];
    grid_dep_wait();  // (a dependent launch after the down GEMM that wrote y)
    const int c = (blockIdx.x * blockDim.x + threadIdx.x) * V;  // first column of the thread
    for (int t = blockIdx.y; t < T; t += gridDim.y) {
        if ((int)threadIdx.x < k) {
            int slot = inv[(size_t)t * k + threadIdx.x];
            if (slot < 0 || slot >= n_rows) {
                moe_flag(status, MOE_ERR_BAD_INDEX);
                slot = -1;
            }
            s_slot[threadIdx.x] = slot;
            s_w[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
        }
        __syncthreads();
        if (c < D) {
            float acc[V];
#pragma unroll
            for (int i = 0; i < V; ++i) acc[i] = 0.f;
#pragma unroll 8
            for (int j = 0; j < k; ++j) {
                const int slot = s_slot[j];
                if (slot < 0) continue;
                const float w = s_w[j];
                const uint4 u = *(const uint4 *)(y + (size_t)slot * D + c);
                const uint32_t q[4] = {u.x, u.y, u.z, u.w};
                if constexpr (sizeof(Y) == 2) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
                        acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(w, __uint_as_float(q[i]), acc[i]);
                }
            }
            if (shared) {
#pragma unroll
                for (int i = 0; i < V; i += 4) {
                    const float4 v = *(const float4 *)(shared + (size_t)t * D + c + i);
                    acc[i] += v.x;
                    acc[i + 1] += v.y;
                    acc[i + 2] += v.z;
                    acc[i + 3] += v.w;
                }
            }
            uint32_t o[V / 2];
#pragma unroll
            for (int i = 0; i < V / 2; ++i)
                o[i] = (uint32_t)f32_to_bf16_bits(acc[2 * i]) |
                       ((uint32_t)f32_to_bf16_bits(acc[2 * i + 1]) << 16);
            if constexpr (V == 8)
                *(uint4 *)(out + (size_t)t * D + c) = make_uint4(o[0], o[1], o[2], o[3]);
            else
                *(uint2 *)(out + (size_t)t * D + c) = make_uint2(o[0], o[1]);
        }
        __syncthreads();  // the slots of the block's next token
    }
}

cudaError_t moe_launch_combine_slots(int T, int D, int k, int n_rows, const float *topk_w,
                                     const int32_t *inv, const float *y, const float *shared,
                                     uint16_t *out, int *status, cudaStream_t st) {
    if (k < 1 || k > MOE_MAX_TOPK || D % 8) return cudaErrorInvalidValue;
    const dim3 g((unsigned)((D / 4 + 127) / 128), (unsigned)min(T, 65535));
    return launch_pdl(moe_combine_slots_kernel<float>, g, dim3(128), 0, st, T, D, k, n_rows,
                      topk_w, inv, y, shared, out, status);
}

cudaError_t moe_launch_combine_slots_bf16(int T, int D, int k, int n_rows, const float *topk_w,
                                          const int32_t *inv, const uint16_t *y,
                                          const float *shared, uint16_t *out, int *status,
                                          cudaStream_t st) {
    if (k < 1 || k > MOE_MAX_TOPK || D % 8) return cudaErrorInvalidValue;
    const dim3 g((unsigned)((D / 8 + 127) / 128), (unsigned)min(T, 65535));
    return launch_pdl(moe_combine_slots_kernel<uint16_t>, g, dim3(128), 0, st, T, D, k, n_rows,
                      topk_w, inv, y, shared, out, status);
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
// MX blocks per lane for a row of K elements: the smallest p <= 8 with
// (K/32) % p == 0 and (K/32)/p a power of two <= 32; 0 if none.
int moe_decode_per_lane(int K) {
    int nblk = K / 32;
    for (int p = 1; p <= 8; ++p) {
        if (nblk % p) continue;
        int l = nblk / p;
        if (l <= 32 && (l & (l - 1)) == 0) return p;
    }
    return 0;
}

namespace {
struct DecodeLayout {
    size_t h16, hexp, y, total;
};

DecodeLayout decode_layout(int T, int D, int F, int k) {
    DecodeLayout L;
    size_t off = 0;
    auto take = [&](size_t b) {
        size_t o = off;
        off += (b + 255) / 256 * 256;
        return o;
    };
    size_t rows = (size_t)T * k;
    L.h16 = take(rows * F * 2);
    L.hexp = take(rows * F / 32);
    L.y = take(rows * D * sizeof(float));
    L.total = off;
    return L;
}

int g_num_sms = 0;
int num_sms() {
    if (!g_num_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    return g_num_sms;
}
}  // namespace

size_t moe_decode_ws_bytes(int T, int D, int F, int k) { return decode_layout(T, D, F, k).total; }

namespace {
template <int P, bool F8>
void launch_gateup(int grid, cudaStream_t st, int D, int F, int E, int k, int n_rows,
                   const uint16_t *x, const moe_plan_buf *p, const moe_weights *w, __half *h16,
                   int8_t *hexp, int *status) {
    const size_t sm = (size_t)kStageTok * (D / 32) * kBlkStride;
    cudaFuncSetAttribute(moe_decode_gateup_kernel<P, F8>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    moe_decode_gateup_kernel<P, F8><<<F8 ? grid / 2 : grid, 256, sm, st>>>(
        D, F, E, k, n_rows, x, p->offsets, p->perm, p->active, w->gate_q, w->gate_s, w->up_q,
        w->up_s, h16, hexp, status);
}

template <int P, bool F8>
void launch_down(int grid, cudaStream_t st, int D, int F, int E, int n_rows, const moe_plan_buf *p,
                 const moe_weights *w, const __half *h16, const int8_t *hexp, float *y,
                 int *status) {
    const size_t sm = (size_t)kStageTok * (F / 32) * kBlkStride;
    cudaFuncSetAttribute(moe_decode_down_kernel<P, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)sm);
    moe_decode_down_kernel<P, F8><<<F8 ? grid / 2 : grid, 256, sm, st>>>(D, F, E, n_rows, p->offsets, p->active,
                                                         w->down_q, w->down_s, h16, hexp, y,
                                                         status);
}

typedef void (*gateup_fn)(int, cudaStream_t, int, int, int, int, int, const uint16_t *,
                          const moe_plan_buf *, const moe_weights *, __half *, int8_t *, int *);
typedef void (*down_fn)(int, cudaStream_t, int, int, int, int, const moe_plan_buf *,
                        const moe_weights *, const __half *, const int8_t *, float *, int *);
const gateup_fn kGateup[2][9] = {
    {nullptr, launch_gateup<1, false>, launch_gateup<2, false>, launch_gateup<3, false>,
     launch_gateup<4, false>, launch_gateup<5, false>, launch_gateup<6, false>,
     launch_gateup<7, false>, launch_gateup<8, false>},
    {nullptr, launch_gateup<1, true>, launch_gateup<2, true>, launch_gateup<3, true>,
     launch_gateup<4, true>, launch_gateup<5, true>, launch_gateup<6, true>,
     launch_gateup<7, true>, launch_gateup<8, true>}};
const down_fn kDown[2][9] = {
    {nullptr, launch_down<1, false>, launch_down<2, false>, launch_down<3, false>,
     launch_down<4, false>, launch_down<5, false>, launch_down<6, false>, launch_down<7, false>,
     launch_down<8, false>},
    {nullptr, launch_down<1, true>, launch_down<2, true>, launch_down<3, true>,
     launch_down<4, true>, launch_down<5, true>, launch_down<6, true>, launch_down<7, true>,
     launch_down<8, true>}};
}  // namespace

cudaError_t moe_launch_decode(int T, int D, int F, int E, int k, const uint16_t *x,
                              const moe_plan_buf *p, const moe_weights *w, int fp8,
                              const float *shared_out, uint16_t *out, void *ws, int *status,
                              const MoeProf &prof, cudaStream_t st) {
    const int n_rows = T * k;
    const DecodeLayout L = decode_layout(T, D, F, k);
    unsigned char *base = (unsigned char *)ws;
    __half *h16 = (__half *)(base + L.h16);
    int8_t *hexp = (int8_t *)(base + L.hexp);
    float *y = (float *)(base + L.y);
    const int grid = 2 * num_sms();
    const int pd = moe_decode_per_lane(D), pf = moe_decode_per_lane(F);
    if (pd < 1 || pd > 8 || pf < 1 || pf > 8) return cudaErrorInvalidValue;
    prof.before(MOE_PROF_DECODE_GATEUP, st);
    kGateup[fp8 ? 1 : 0][pd](grid, st, D, F, E, k, n_rows, x, p, w, h16, hexp, status);
    prof.after(MOE_PROF_DECODE_GATEUP, st);
    prof.before(MOE_PROF_DECODE_DOWN, st);
    kDown[fp8 ? 1 : 0][pf](grid, st, D, F, E, n_rows, p, w, h16, hexp, y, status);
    prof.after(MOE_PROF_DECODE_DOWN, st);
    return moe_launch_combine_slots(T, D, k, n_rows, p->topk_w, p->inv, y, shared_out, out, status,
                                    st);
}
