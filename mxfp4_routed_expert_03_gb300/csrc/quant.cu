// Small kernels around the grouped GEMMs: the activation split-quantiser
// (bf16 -> two-term MXFP8), the per-expert token-tile schedule, and the final
// fp32 -> bf16 cast of the combined output.
#include "common.cuh"
#include "kernels.h"
#include "mx8.cuh"

#define FULL_MASK 0xFFFFFFFFu

// Two-term MXFP8 split of 32 consecutive bf16 values: hi = E4M3(v / 2^sh),
// lo = E4M3((v - hi 2^sh) / 2^sl), sh and sl the E8M0 exponents of the block
// maxima; hw / lw receive the 32 hi / lo bytes (element 2i in the low byte of
// each pair).
__device__ __forceinline__ void split_block32(const uint16_t *__restrict__ src16, uint32_t (&hw)[8],
                                              uint32_t (&lw)[8], int &sh, int &sl) {
    const uint4 *src = (const uint4 *)src16;
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 u = src[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
            v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    sh = mx8::scale_exp(amax);
    float inv_h = mx8::exp2i(-sh), sc_h = mx8::exp2i(sh);
    float r[32];
    float ramax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t p = mx8::to_e4m3x2(v[2 * i] * inv_h, v[2 * i + 1] * inv_h);
        float2 back = mx8::from_e4m3x2(p);
        r[2 * i] = v[2 * i] - back.x * sc_h;
        r[2 * i + 1] = v[2 * i + 1] - back.y * sc_h;
        ramax = fmaxf(ramax, fmaxf(fabsf(r[2 * i]), fabsf(r[2 * i + 1])));
        if (i % 2 == 0) hw[i / 2] = p;
        else hw[i / 2] |= p << 16;
    }
    sl = mx8::scale_exp(ramax);
    float inv_l = mx8::exp2i(-sl);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        uint32_t p = mx8::to_e4m3x2(r[2 * i] * inv_l, r[2 * i + 1] * inv_l);
        if (i % 2 == 0) lw[i / 2] = p;
        else lw[i / 2] |= p << 16;
    }
}

// One thread per 32-element block of x: hi/lo E4M3 bytes and their E8M0 scales.
__global__ void __launch_bounds__(256) moe_quant_x_kernel(int64_t n_blocks, int D,
                                                          const uint16_t *__restrict__ x,
                                                          uint8_t *__restrict__ q_hi,
                                                          uint8_t *__restrict__ q_lo,
                                                          uint8_t *__restrict__ s_hi,
                                                          uint8_t *__restrict__ s_lo) {
    int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (b >= n_blocks) return;
    uint32_t hw[8], lw[8];
    int sh, sl;
    split_block32(x + b * 32, hw, lw, sh, sl);
    uint4 *dh = (uint4 *)(q_hi + b * 32), *dl = (uint4 *)(q_lo + b * 32);
    dh[0] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    dh[1] = make_uint4(hw[4], hw[5], hw[6], hw[7]);
    dl[0] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    dl[1] = make_uint4(lw[4], lw[5], lw[6], lw[7]);
    s_hi[b] = (uint8_t)(sh + 127);
    s_lo[b] = (uint8_t)(sl + 127);
}

// tt_prefix[a] = token tiles of active experts before a; tt_prefix[n] = total.
__global__ void __launch_bounds__(1024) moe_schedule_kernel(int E, int ntmax,
                                                            const int32_t *__restrict__ offsets,
                                                            const int32_t *__restrict__ active,
                                                            int32_t *__restrict__ tt_prefix,
                                                            int *status) {
    __shared__ int s_tot[33];
    int a = threadIdx.x, lane = a & 31, wid = a >> 5;
    int n = active[0];
    if (n < 0 || n > E) {
        if (a == 0) { moe_flag(status, MOE_ERR_BAD_INDEX); tt_prefix[0] = 0; }
        n = 0;
    }
    int ntt = 0;
    if (a < n) {
        int e = active[1 + a];
        if (e >= 0 && e < E) {
            int c = offsets[e + 1] - offsets[e];
            ntt = c > 0 ? (c + ntmax - 1) / ntmax : 0;
        } else {
            moe_flag(status, MOE_ERR_BAD_INDEX);
        }
    }
    int inc = ntt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(FULL_MASK, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) s_tot[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        int t = s_tot[lane], ti = t;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(FULL_MASK, ti, off);
            if (lane >= off) ti += o;
        }
        s_tot[lane] = ti - t;
        if (lane == 31) s_tot[32] = ti;
    }
    __syncthreads();
    int excl = s_tot[wid] + inc - ntt;
    if (a < n) tt_prefix[a] = excl;
    if (a == 0) tt_prefix[n] = s_tot[32];
}

__global__ void __launch_bounds__(256) moe_finalize_kernel(int64_t n4, const float *__restrict__ acc,
                                                           uint16_t *__restrict__ out) {
    grid_dep_wait();    // acc is complete once the down GEMM is
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n4) return;
    float4 v = ((const float4 *)acc)[i];
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(v.x) | ((uint32_t)f32_to_bf16_bits(v.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(v.z) | ((uint32_t)f32_to_bf16_bits(v.w) << 16);
    ((uint2 *)out)[i] = o;
}

// Token tile tt -> its expert's active index a, first row r0 and row count n
// (the same split the grouped GEMMs use: ntt = ceil(count / ntmax) tiles of
// near-equal size per expert).
__device__ __forceinline__ bool token_tile(int tt, int n_active, const int32_t *prefix,
                                           const int32_t *active, const int32_t *offsets, int E,
                                           int n_rows, int &e, int &sb, int &r0, int &n) {
    if (n_active <= 0 || tt >= prefix[n_active]) return false;
    int lo = 0, hi = n_active - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tt) lo = mid;
        else hi = mid - 1;
    }
    int ntt = prefix[lo + 1] - prefix[lo];
    int j = tt - prefix[lo];
    e = active[1 + lo];
    if (ntt <= 0 || e < 0 || e >= E) return false;
    sb = offsets[e];
    int cnt = offsets[e + 1] - sb;
    if (sb < 0 || cnt <= 0 || sb + cnt > n_rows) return false;
    r0 = (int)((long long)j * cnt / ntt);
    n = (int)((long long)(j + 1) * cnt / ntt) - r0;
    return true;
}

// Lays out the quantised activation rows of one token tile as the grouped
// GEMM's B operand: for each 128-wide K chunk one block of 2 * NTMAX rows of
// 128 bytes (row r = tile row r's hi term, row nmma + r = its lo term; nmma =
// rows rounded up to 16), each row pre-swizzled for the 128-byte shared-memory
// swizzle (16-byte chunk c stored at c ^ (row % 8)), so one contiguous bulk
// copy per chunk lands a ready MMA tile. The scales go into a 1 KB block per
// chunk: B row n, 32-wide block c at byte
// (i / 8) * 256 + (j / 4) * 128 + (i % 8) * 16 + (j % 4) * 4 + c with
// i = n % 32, j = n / 32 (32 lanes x 8 columns as tcgen05.cp.128x256b reads
// K-major 8 x 16-byte core matrices).
__global__ void __launch_bounds__(256) moe_gather_x_kernel(
    int E, int k, int n_rows, int D, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const int32_t *__restrict__ prefix, const uint8_t *__restrict__ q_hi,
    const uint8_t *__restrict__ q_lo, const uint8_t *__restrict__ s_hi,
    const uint8_t *__restrict__ s_lo, uint8_t *__restrict__ tiles, uint8_t *__restrict__ atoms,
    int *status) {
    __shared__ int s_tok[MOE_GEMM_NTMAX];
    const int tt = blockIdx.x;
    int n_active = active[0];
    if (n_active < 0 || n_active > E) return;
    int e, sb, r0, n;
    if (!token_tile(tt, n_active, prefix, active, offsets, E, n_rows, e, sb, r0, n)) return;
    if (n > MOE_GEMM_NTMAX) { if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX); return; }
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
        int fl = perm[sb + r0 + r];
        if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
        s_tok[r] = fl / k;
    }
    __syncthreads();
    const int KC = D / 128, nmma = (n + 15) & ~15;
    // 16-byte pieces: (row r, chunk kc, piece c) for hi and lo
    for (int i = threadIdx.x; i < n * KC * 8; i += blockDim.x) {
        const int r = i / (KC * 8), rem = i % (KC * 8), kc = rem / 8, c = rem % 8;
        const size_t src = (size_t)s_tok[r] * D + kc * 128 + c * 16;
        uint8_t *blk = tiles + ((size_t)tt * KC + kc) * MOE_GEMM_BTILE;
        const int rl = nmma + r;
        *(uint4 *)(blk + r * 128 + ((c ^ (r & 7)) * 16)) = *(const uint4 *)(q_hi + src);
        *(uint4 *)(blk + rl * 128 + ((c ^ (rl & 7)) * 16)) = *(const uint4 *)(q_lo + src);
    }
    const int nb = D / 32;
    auto off = [](int row, int c) {
        const int i = row & 31, j = row >> 5;
        return (i >> 3) * 256 + (j >> 2) * 128 + (i & 7) * 16 + (j & 3) * 4 + c;
    };
    for (int i = threadIdx.x; i < n * nb; i += blockDim.x) {
        const int r = i / nb, b = i % nb, c = b & 3;
        const size_t at = ((size_t)tt * KC + b / 4) * 1024;
        atoms[at + off(r, c)] = s_hi[(size_t)s_tok[r] * nb + b];
        atoms[at + off(nmma + r, c)] = s_lo[(size_t)s_tok[r] * nb + b];
    }
}

// Batches of at most MOE_GEMM_NT_NARROW tokens: every active expert has one
// token tile (a token chooses an expert at most once), so token tile a is
// active expert a and the schedule is the identity. One block per active
// expert quantises its tokens' x rows straight into the B tile and scale
// block layout the gather kernel writes (same split as moe_quant_x_kernel,
// same bytes), writes tt_prefix[a] = a, and every block zeroes its share of
// the fp32 accumulator when one is given. Replaces quant, schedule, gather
// and the accumulator memset of larger batches.
__global__ void __launch_bounds__(256) moe_prep_small_kernel(
    int E, int k, int n_rows, int D, int T, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const uint16_t *__restrict__ x, int32_t *__restrict__ tt_prefix, uint8_t *__restrict__ tiles,
    uint8_t *__restrict__ atoms, float *__restrict__ acc, int *__restrict__ sk_count, int n_sk,
    int *status) {
    __shared__ int s_tok[MOE_GEMM_NT_NARROW];
    grid_dep_wait();    // the plan comes from the previous kernel
    grid_dep_launch();
    if (acc) {  // zero this block's share of acc [T][D]
        const int64_t n4 = (int64_t)T * D / 4, per = (n4 + gridDim.x - 1) / gridDim.x;
        const int64_t i0 = (int64_t)blockIdx.x * per, i1 = min(i0 + per, n4);
        for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x)
            ((float4 *)acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the grouped GEMMs' split-tile counters
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_sk; i += gridDim.x * blockDim.x)
        sk_count[i] = 0;
    int n_active = active[0];
    if (n_active < 0 || n_active > E) {
        if (blockIdx.x == 0 && threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        return;
    }
    const int a = blockIdx.x;
    if (a == 0 && threadIdx.x == 0) tt_prefix[n_active] = n_active;
    if (a >= n_active) return;
    if (threadIdx.x == 0) tt_prefix[a] = a;
    const int e = active[1 + a];
    if (e < 0 || e >= E) { if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX); return; }
    const int sb = offsets[e], n = offsets[e + 1] - sb;
    if (sb < 0 || n <= 0 || n > MOE_GEMM_NT_NARROW || sb + n > n_rows) {
        if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        return;
    }
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
        int fl = perm[sb + r];
        if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
        s_tok[r] = fl / k;
    }
    __syncthreads();
    const int KC = D / 128, nb = D / 32, nmma = (n + 15) & ~15;
    auto off = [](int row, int c) {
        const int i = row & 31, j = row >> 5;
        return (i >> 3) * 256 + (j >> 2) * 128 + (i & 7) * 16 + (j & 3) * 4 + c;
    };
    for (int i = threadIdx.x; i < n * nb; i += blockDim.x) {
        const int r = i / nb, b = i % nb, kc = b >> 2, c = b & 3;
        uint32_t hw[8], lw[8];
        int sh, sl;
        split_block32(x + (size_t)s_tok[r] * D + (size_t)b * 32, hw, lw, sh, sl);
        uint8_t *blk = tiles + ((size_t)a * KC + kc) * MOE_GEMM_BTILE;
        const int rl = nmma + r, p0 = 2 * c, p1 = 2 * c + 1;  // 16-byte pieces of the row
        *(uint4 *)(blk + r * 128 + ((p0 ^ (r & 7)) * 16)) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *(uint4 *)(blk + r * 128 + ((p1 ^ (r & 7)) * 16)) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
        *(uint4 *)(blk + rl * 128 + ((p0 ^ (rl & 7)) * 16)) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        *(uint4 *)(blk + rl * 128 + ((p1 ^ (rl & 7)) * 16)) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
        const size_t at = ((size_t)a * KC + kc) * 1024;
        atoms[at + off(r, c)] = (uint8_t)(sh + 127);
        atoms[at + off(rl, c)] = (uint8_t)(sl + 127);
    }
}

// ---------------------------------------------------------------------------
// FP4 x FP4 mode: activations as one MXFP4 term (E2M1 codes, one E8M0 scale
// per 32 values; OCP MX conversion, see mx8.cuh).
// ---------------------------------------------------------------------------

// MXFP4 conversion of 32 consecutive bf16 values: 16 bytes of E2M1 codes
// (element 2i in the low nibble of byte i) and the scale exponent.
__device__ __forceinline__ void mxfp4_block32(const uint16_t *__restrict__ src16,
                                              uint32_t (&w)[4], int &s) {
    const uint4 *src = (const uint4 *)src16;
    float v[32];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 u = src[i];
        const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = __uint_as_float(q[j] << 16);
            v[8 * i + 2 * j + 1] = __uint_as_float(q[j] & 0xFFFF0000u);
        }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    s = mx4::scale_exp(amax);
    const float inv = mx8::exp2i(-s);
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        w[i / 4] |= mx4::to_e2m1x2(v[2 * i] * inv, v[2 * i + 1] * inv) << (8 * (i % 4));
}

// Row r of a token tile, 32-element block b of its K: the 16 code bytes go to
// the tile's packed block of K chunk b / 8 (one 128-byte row per token,
// 16-byte piece b % 8 stored at piece (b % 8) ^ (r % 8), the 128-byte
// swizzle), the scale to the 1 KB block of K block b / 4 (same placement as
// the two-term mode's hi rows).
__device__ __forceinline__ void put_fp4_block(uint8_t *tiles, uint8_t *atoms, size_t tt, int KC2,
                                              int KC, int r, int b, const uint32_t (&w)[4],
                                              int s) {
    uint8_t *blk = tiles + (tt * KC2 + b / 8) * MOE_GEMM_BTILE;
    *(uint4 *)(blk + r * 128 + (((b & 7) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    const int i = r & 31, j = r >> 5, c = b & 3;
    atoms[(tt * KC + b / 4) * 1024 + (i >> 3) * 256 + (j >> 2) * 128 + (i & 7) * 16 + (j & 3) * 4 + c] =
        (uint8_t)(s + 127);
}

// Small batches in the FP4 mode: as moe_prep_small_kernel (one block per
// active expert, identity schedule, accumulator zeroed), with one MXFP4 term.
__global__ void __launch_bounds__(256) moe_prep_small_fp4_kernel(
    int E, int k, int n_rows, int D, int T, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const uint16_t *__restrict__ x, int32_t *__restrict__ tt_prefix, uint8_t *__restrict__ tiles,
    uint8_t *__restrict__ atoms, float *__restrict__ acc, int *__restrict__ sk_count, int n_sk,
    int *status) {
    __shared__ int s_tok[MOE_GEMM_NT_NARROW];
    grid_dep_wait();    // the plan comes from the previous kernel
    grid_dep_launch();
    if (acc) {  // zero this block's share of acc [T][D]
        const int64_t n4 = (int64_t)T * D / 4, per = (n4 + gridDim.x - 1) / gridDim.x;
        const int64_t i0 = (int64_t)blockIdx.x * per, i1 = min(i0 + per, n4);
        for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x)
            ((float4 *)acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the grouped GEMMs' split-tile counters
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_sk; i += gridDim.x * blockDim.x)
        sk_count[i] = 0;
    int n_active = active[0];
    if (n_active < 0 || n_active > E) {
        if (blockIdx.x == 0 && threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        return;
    }
    const int a = blockIdx.x;
    if (a == 0 && threadIdx.x == 0) tt_prefix[n_active] = n_active;
    if (a >= n_active) return;
    if (threadIdx.x == 0) tt_prefix[a] = a;
    const int e = active[1 + a];
    if (e < 0 || e >= E) { if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX); return; }
    const int sb = offsets[e], n = offsets[e + 1] - sb;
    if (sb < 0 || n <= 0 || n > MOE_GEMM_NT_NARROW || sb + n > n_rows) {
        if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        return;
    }
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
        int fl = perm[sb + r];
        if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
        s_tok[r] = fl / k;
    }
    __syncthreads();
    const int nb = D / 32, KC = D / 128, KC2 = (KC + 1) / 2;
    for (int i = threadIdx.x; i < n * nb; i += blockDim.x) {
        const int r = i / nb, b = i % nb;
        uint32_t w[4];
        int sc;
        mxfp4_block32(x + (size_t)s_tok[r] * D + (size_t)b * 32, w, sc);
        put_fp4_block(tiles, atoms, (size_t)a, KC2, KC, r, b, w, sc);
    }
}

// Larger batches in the FP4 mode: one block per token tile quantises its
// rows straight from x into the tile layout (no separate quantise pass).
// Larger batches in the FP4 x FP4 mode, first pass: every token's row once
// to MXFP4, q [T][D/2] (16 code bytes per 32-element block, element 2i in
// the low nibble of byte i) and s [T][D/32] (biased E8M0 scale bytes).
__global__ void __launch_bounds__(256) moe_quant_x_fp4_kernel(int64_t n_blocks, int D,
                                                              const uint16_t *__restrict__ x,
                                                              uint8_t *__restrict__ q,
                                                              uint8_t *__restrict__ s) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;  // 32-element block
    if (i >= n_blocks) return;
    uint32_t w[4];
    int sc;
    mxfp4_block32(x + i * 32, w, sc);
    *(uint4 *)(q + i * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    s[i] = (uint8_t)(sc + 127);
}

// Second pass: token tile tt's rows copied from q / s into the tile layout
// put_fp4_block writes (one 16-byte piece and one scale byte per block).
__global__ void __launch_bounds__(256) moe_gather_x_fp4_kernel(
    int E, int k, int n_rows, int D, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const int32_t *__restrict__ prefix, const uint8_t *__restrict__ q,
    const uint8_t *__restrict__ s, uint8_t *__restrict__ tiles, uint8_t *__restrict__ atoms,
    int *status) {
    __shared__ int s_tok[MOE_GEMM_NTMAX];
    const int tt = blockIdx.x;
    int n_active = active[0];
    if (n_active < 0 || n_active > E) return;
    int e, sb, r0, n;
    if (!token_tile(tt, n_active, prefix, active, offsets, E, n_rows, e, sb, r0, n)) return;
    if (n > MOE_GEMM_NTMAX) { if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX); return; }
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
        int fl = perm[sb + r0 + r];
        if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
        s_tok[r] = fl / k;
    }
    __syncthreads();
    const int nb = D / 32, KC = D / 128, KC2 = (KC + 1) / 2;
    for (int i = threadIdx.x; i < n * nb; i += blockDim.x) {
        const int r = i / nb, b = i % nb;
        const size_t src = (size_t)s_tok[r] * nb + b;
        uint8_t *blk = tiles + ((size_t)tt * KC2 + b / 8) * MOE_GEMM_BTILE;
        *(uint4 *)(blk + r * 128 + (((b & 7) ^ (r & 7)) << 4)) = *(const uint4 *)(q + src * 16);
        const int ri = r & 31, rj = r >> 5;
        atoms[((size_t)tt * KC + b / 4) * 1024 + (ri >> 3) * 256 + (rj >> 2) * 128 + (ri & 7) * 16 +
              (rj & 3) * 4 + (b & 3)] = s[src];
    }
}

cudaError_t moe_launch_prep_small_fp4(int T, int E, int k, int D, const int32_t *offsets,
                                      const int32_t *perm, const int32_t *active,
                                      const uint16_t *x, int32_t *tt_prefix, uint8_t *tiles,
                                      uint8_t *atoms, float *acc, int *sk_count, int n_sk,
                                      int *status, cudaStream_t st) {
    const int grid = min(T * k, E);  // an upper bound on the active experts
    return launch_pdl(moe_prep_small_fp4_kernel, dim3(grid), dim3(256), 0, st, E, k, T * k, D, T,
                      offsets, perm, active, x, tt_prefix, tiles, atoms, acc, sk_count, n_sk,
                      status);
}

cudaError_t moe_launch_quant_x_fp4(int T, int D, const uint16_t *x, uint8_t *q, uint8_t *s,
                                   cudaStream_t st) {
    const int64_t nb = (int64_t)T * D / 32;
    moe_quant_x_fp4_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>(nb, D, x, q, s);
    return cudaGetLastError();
}

cudaError_t moe_launch_gather_x_fp4(int max_tt, int E, int k, int n_rows, int D,
                                    const int32_t *offsets, const int32_t *perm,
                                    const int32_t *active, const int32_t *tt_prefix,
                                    const uint8_t *q, const uint8_t *s, uint8_t *tiles,
                                    uint8_t *atoms, int *status, cudaStream_t st) {
    moe_gather_x_fp4_kernel<<<max_tt, 256, 0, st>>>(E, k, n_rows, D, offsets, perm, active,
                                                    tt_prefix, q, s, tiles, atoms, status);
    return cudaGetLastError();
}

cudaError_t moe_launch_prep_small(int T, int E, int k, int D, const int32_t *offsets,
                                  const int32_t *perm, const int32_t *active, const uint16_t *x,
                                  int32_t *tt_prefix, uint8_t *tiles, uint8_t *atoms, float *acc,
                                  int *sk_count, int n_sk, int *status, cudaStream_t st) {
    const int grid = min(T * k, E);  // an upper bound on the active experts
    return launch_pdl(moe_prep_small_kernel, dim3(grid), dim3(256), 0, st, E, k, T * k, D, T,
                      offsets, perm, active, x, tt_prefix, tiles, atoms, acc, sk_count, n_sk,
                      status);
}

cudaError_t moe_launch_gather_x(int max_tt, int E, int k, int n_rows, int D, int ntmax,
                                const int32_t *offsets, const int32_t *perm, const int32_t *active,
                                const int32_t *tt_prefix, const uint8_t *q_hi, const uint8_t *q_lo,
                                const uint8_t *s_hi, const uint8_t *s_lo, uint8_t *tiles,
                                uint8_t *atoms, int *status, cudaStream_t st) {
    (void)ntmax;
    moe_gather_x_kernel<<<max_tt, 256, 0, st>>>(E, k, n_rows, D, offsets, perm, active, tt_prefix,
                                                q_hi, q_lo, s_hi, s_lo, tiles, atoms, status);
    return cudaGetLastError();
}

cudaError_t moe_launch_quant_x(int T, int D, const uint16_t *x, uint8_t *q_hi, uint8_t *q_lo,
                               uint8_t *s_hi, uint8_t *s_lo, cudaStream_t st) {
    int64_t nb = (int64_t)T * D / 32;
    moe_quant_x_kernel<<<(unsigned)((nb + 255) / 256), 256, 0, st>>>(nb, D, x, q_hi, q_lo, s_hi,
                                                                       s_lo);
    return cudaGetLastError();
}

cudaError_t moe_launch_schedule(int E, int ntmax, const int32_t *offsets, const int32_t *active,
                                int32_t *tt_prefix, int *status, cudaStream_t st) {
    moe_schedule_kernel<<<1, 1024, 0, st>>>(E, ntmax, offsets, active, tt_prefix, status);
    return cudaGetLastError();
}

cudaError_t moe_launch_finalize(int T, int D, const float *acc, uint16_t *out, cudaStream_t st) {
    int64_t n4 = (int64_t)T * D / 4;
    return launch_pdl(moe_finalize_kernel, dim3((unsigned)((n4 + 255) / 256)), dim3(256), 0, st,
                      n4, acc, out);
}
