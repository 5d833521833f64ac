// FP8 expert lane: routed experts held as FP8 E4M3FN codes with one fp32
// scale per 128 x 128 block (Moonshine GitHub README, "GLM 5.3 Flash
// status": FP8 E4M3FN experts, a fused decode GEMV and a BF16-dequant
// prefill). The decode GEMV is the CUDA-core decode path of decode.cu on
// E4M3 codes; this file holds the prefill's side:
//   - the one-time dequantisation of every expert to bf16 (value(code) x
//     block scale, rounded to nearest even) into a caller buffer, which the
//     bf16 grouped tcgen05 GEMMs (kind::f16) then stream;
//   - the activation tiles those GEMMs read: bf16 x rows laid out per token
//     tile and 64-wide K block, one 128-byte row per token, pre-swizzled for
//     the 128-byte shared-memory swizzle (16-byte piece c at c ^ (row % 8)).
#include "common.cuh"
#include "kernels.h"

namespace {

// E4M3FN code -> fp32 (exact): sign, 4 exponent bits with bias 7, 3 mantissa
// bits, exponent 0 subnormal (m * 2^-9), S.1111.111 NaN, no infinities.
__device__ __forceinline__ float e4m3_to_f32(uint32_t c) {
    const uint32_t e = (c >> 3) & 0xFu, m = c & 7u;
    float v;
    if (e == 0xFu && m == 7u) v = __uint_as_float(0x7FC00000u);
    else if (e == 0u) v = (float)m * 0.001953125f;  // m * 2^-9
    else v = __uint_as_float(((e + 120u) << 23) | (m << 20));  // (1 + m/8) 2^(e-7)
    return (c & 0x80u) ? -v : v;
}

}  // namespace

// out[e][n][k] = bf16(value(codes[e][n][k]) * scales[e][n / 128][k / 128]);
// one thread per 8 consecutive codes of a row (K a multiple of 128).
__global__ void __launch_bounds__(256) moe_fp8_dequant_kernel(int64_t n8, int N, int K,
                                                              const uint8_t *__restrict__ codes,
                                                              const float *__restrict__ scales,
                                                              uint16_t *__restrict__ out) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const int64_t per_row = K / 8;
    const int64_t row = i / per_row;  // e * N + n
    const int k0 = (int)(i % per_row) * 8;
    const int64_t e = row / N;
    const int n = (int)(row % N);
    const int nk = K / 128;
    const float sc = scales[(e * ((N + 127) / 128) + n / 128) * nk + k0 / 128];
    const uint2 q = *(const uint2 *)(codes + i * 8);
    const uint32_t w[2] = {q.x, q.y};
    uint32_t o[4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const float a = e4m3_to_f32((w[h] >> (16 * j)) & 0xFFu) * sc;
            const float b = e4m3_to_f32((w[h] >> (16 * j + 8)) & 0xFFu) * sc;
            o[2 * h + j] = (uint32_t)f32_to_bf16_bits(a) | ((uint32_t)f32_to_bf16_bits(b) << 16);
        }
    *(uint4 *)(out + i * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

// Rows r < n of a token tile: the 64-element K block b of token row tok is
// the 128 bytes of x[tok][64 b ..], stored at row r of the tile's block b
// with the 128-byte swizzle.
__device__ __forceinline__ void put_bf16_rows(const uint16_t *__restrict__ x, int D,
                                              const int *s_tok, int n, uint8_t *tiles, size_t tt) {
    const int KB = D / 64;
    for (int i = threadIdx.x; i < n * KB * 8; i += blockDim.x) {
        const int r = i / (KB * 8), rem = i % (KB * 8), b = rem / 8, c = rem % 8;
        const uint4 v = *((const uint4 *)(x + (size_t)s_tok[r] * D + (size_t)b * 64) + c);
        uint8_t *blk = tiles + (tt * KB + b) * MOE_GEMM_BTILE;
        *(uint4 *)(blk + r * 128 + ((c ^ (r & 7)) << 4)) = v;
    }
}

// Small batches: one block per active expert (token tile a = active expert a,
// identity schedule), the fp32 accumulator zeroed when given.
__global__ void __launch_bounds__(256) moe_prep_small_bf16_kernel(
    int E, int k, int n_rows, int D, int T, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const uint16_t *__restrict__ x, int32_t *__restrict__ tt_prefix, uint8_t *__restrict__ tiles,
    float *__restrict__ acc, int *__restrict__ sk_count, int n_sk, int *status) {
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
    put_bf16_rows(x, D, s_tok, n, tiles, (size_t)a);
}

// Larger batches: one block per token tile tt (the schedule's split of each
// expert's rows into ceil(count / NTMAX) near-equal tiles).
__global__ void __launch_bounds__(256) moe_gather_x_bf16_kernel(
    int E, int k, int n_rows, int D, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, const int32_t *__restrict__ active,
    const int32_t *__restrict__ prefix, const uint16_t *__restrict__ x,
    uint8_t *__restrict__ tiles, int *status) {
    __shared__ int s_tok[MOE_GEMM_NTMAX];
    const int tt = blockIdx.x;
    const int n_active = active[0];
    if (n_active <= 0 || n_active > E || tt >= prefix[n_active]) return;
    int lo = 0, hi = n_active - 1;  // the active expert owning token tile tt
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tt) lo = mid;
        else hi = mid - 1;
    }
    const int ntt = prefix[lo + 1] - prefix[lo], j = tt - prefix[lo];
    const int e = active[1 + lo];
    if (ntt <= 0 || e < 0 || e >= E) return;
    const int sb = offsets[e], cnt = offsets[e + 1] - sb;
    if (sb < 0 || cnt <= 0 || sb + cnt > n_rows) return;
    const int r0 = (int)((long long)j * cnt / ntt);
    const int n = (int)((long long)(j + 1) * cnt / ntt) - r0;
    if (n > MOE_GEMM_NTMAX) { if (threadIdx.x == 0) moe_flag(status, MOE_ERR_BAD_INDEX); return; }
    for (int r = threadIdx.x; r < n; r += blockDim.x) {
        int fl = perm[sb + r0 + r];
        if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
        s_tok[r] = fl / k;
    }
    __syncthreads();
    put_bf16_rows(x, D, s_tok, n, tiles, (size_t)tt);
}

cudaError_t moe_launch_fp8_dequant(int E, int N, int K, const uint8_t *codes, const float *scales,
                                   uint16_t *out, cudaStream_t st) {
    const int64_t n8 = (int64_t)E * N * K / 8;
    if (n8 <= 0 || K % 128) return cudaErrorInvalidValue;
    moe_fp8_dequant_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, st>>>(n8, N, K, codes, scales,
                                                                         out);
    return cudaGetLastError();
}

cudaError_t moe_launch_prep_small_bf16(int T, int E, int k, int D, const int32_t *offsets,
                                       const int32_t *perm, const int32_t *active,
                                       const uint16_t *x, int32_t *tt_prefix, uint8_t *tiles,
                                       float *acc, int *sk_count, int n_sk, int *status,
                                       cudaStream_t st) {
    const int grid = min(T * k, E);  // an upper bound on the active experts
    return launch_pdl(moe_prep_small_bf16_kernel, dim3(grid), dim3(256), 0, st, E, k, T * k, D, T,
                      offsets, perm, active, x, tt_prefix, tiles, acc, sk_count, n_sk, status);
}

cudaError_t moe_launch_gather_x_bf16(int max_tt, int E, int k, int n_rows, int D,
                                     const int32_t *offsets, const int32_t *perm,
                                     const int32_t *active, const int32_t *tt_prefix,
                                     const uint16_t *x, uint8_t *tiles, int *status,
                                     cudaStream_t st) {
    moe_gather_x_bf16_kernel<<<max_tt, 256, 0, st>>>(E, k, n_rows, D, offsets, perm, active,
                                                     tt_prefix, x, tiles, status);
    return cudaGetLastError();
}
