// Device half of the seeded synthetic-input generator: fills a whole routed
// layer's MXFP4 expert weights in HBM with the same bytes the host half emits
// (see synth_host.c for the stream addressing and distributions). Integer work
// only, so host and device agree bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>
#include "philox.h"

#define SYNTH_API extern "C" __attribute__((visibility("default")))

// One thread per 16-byte Philox block of one row.
__global__ void synth_codes_kernel(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t rows,
                                   int64_t nblk, int64_t n_experts, uint4 *out) {
    int64_t total = n_experts * rows * nblk;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t b = i % nblk;
        int64_t r = (i / nblk) % rows;
        int64_t e = i / (nblk * rows);
        synth_u32x4 w = synth_block(seed, tensor, e0 + (uint32_t)e, (uint32_t)r, (uint32_t)b);
        out[i] = make_uint4(w.v[0], w.v[1], w.v[2], w.v[3]);
    }
}

// Peaked code distribution: one thread per 16-byte block of one row.
__global__ void synth_codes_peaked_kernel(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t rows,
                                          int64_t nblk, int64_t n_experts, uint4 *out) {
    int64_t total = n_experts * rows * nblk;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t b = i % nblk;
        int64_t r = (i / nblk) % rows;
        int64_t e = i / (nblk * rows);
        union { uint8_t b[16]; uint4 v; } u;
        synth_peaked_block(seed, tensor, e0 + (uint32_t)e, (uint32_t)r, (uint32_t)b, u.b);
        out[i] = u.v;
    }
}

// One thread per group of four scale bytes of one row.
__global__ void synth_scales_kernel(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t rows,
                                    int64_t ns, int64_t n_experts, uint32_t lo, uint32_t n,
                                    uint8_t *out) {
    int64_t ngrp = (ns + 3) / 4;
    int64_t total = n_experts * rows * ngrp;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t g = i % ngrp;
        int64_t r = (i / ngrp) % rows;
        int64_t e = i / (ngrp * rows);
        synth_u32x4 w = synth_block(seed, tensor, e0 + (uint32_t)e, (uint32_t)r, (uint32_t)g);
        uint8_t *dst = out + (e * rows + r) * ns;
        for (int q = 0; q < 4; ++q) {
            int64_t c = g * 4 + q;
            if (c < ns) dst[c] = (uint8_t)synth_uniform_int(w.v[q], lo, n);
        }
    }
}

// codes: n_experts x rows x (K/2) bytes starting at expert e0 (K % 32 == 0).
SYNTH_API int synth_dev_mx_codes(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t n_experts,
                                 int64_t rows, int64_t K, void *out, void *stream) {
    if (K % 32 != 0 || rows <= 0 || n_experts <= 0 || ((uintptr_t)out & 15)) return -1;
    int64_t nblk = K / 32;  // 16-byte blocks per row
    synth_codes_kernel<<<152 * 8, 256, 0, (cudaStream_t)stream>>>(seed, tensor, e0, rows, nblk,
                                                                   n_experts, (uint4 *)out);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// codes under distribution `dist` (0 uniform, 1 peaked).
SYNTH_API int synth_dev_mx_codes_dist(uint64_t seed, uint32_t tensor, uint32_t e0,
                                      int64_t n_experts, int64_t rows, int64_t K, int dist,
                                      void *out, void *stream) {
    if (dist == 0) return synth_dev_mx_codes(seed, tensor, e0, n_experts, rows, K, out, stream);
    if (dist != 1 || K % 32 != 0 || rows <= 0 || n_experts <= 0 || ((uintptr_t)out & 15))
        return -1;
    synth_codes_peaked_kernel<<<152 * 8, 256, 0, (cudaStream_t)stream>>>(
        seed, tensor, e0, rows, K / 32, n_experts, (uint4 *)out);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// scales: n_experts x rows x (K/32) bytes, uniform over {lo .. lo+n-1}.
SYNTH_API int synth_dev_mx_scales(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t n_experts,
                                  int64_t rows, int64_t K, int lo, int n, void *out, void *stream) {
    if (K % 32 != 0 || rows <= 0 || n_experts <= 0 || n < 1 || lo < 0 || lo + n - 1 > 254)
        return -1;
    synth_scales_kernel<<<152 * 8, 256, 0, (cudaStream_t)stream>>>(
        seed, tensor, e0, rows, K / 32, n_experts, (uint32_t)lo, (uint32_t)n, (uint8_t *)out);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// FP8 expert codes: one thread per 16-byte Philox block of one row.
__global__ void synth_fp8_codes_kernel(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t rows,
                                       int64_t nblk, int64_t n_experts, uint4 *out) {
    int64_t total = n_experts * rows * nblk;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t b = i % nblk;
        int64_t r = (i / nblk) % rows;
        int64_t e = i / (nblk * rows);
        synth_u32x4 w = synth_block(seed, tensor, e0 + (uint32_t)e, (uint32_t)r, (uint32_t)b);
        uint32_t o[4];
        for (int q = 0; q < 4; ++q) {
            o[q] = 0;
            for (int j = 0; j < 4; ++j)
                o[q] |= synth_fp8_code((w.v[q] >> (8 * j)) & 0xFFu) << (8 * j);
        }
        out[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// FP8 block scales: one thread per entry.
__global__ void synth_fp8_scales_kernel(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t nr,
                                        int64_t nk, int64_t n_experts, uint32_t *out) {
    int64_t total = n_experts * nr * nk;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t j = i % nk;
        int64_t r = (i / nk) % nr;
        int64_t e = i / (nk * nr);
        synth_u32x4 w = synth_block(seed, tensor, e0 + (uint32_t)e, (uint32_t)r, (uint32_t)(j / 4));
        out[i] = synth_fp8_scale_bits(w.v[j % 4]);
    }
}

// FP8 codes of n_experts experts from e0: n_experts x rows x K bytes (K % 16 == 0).
SYNTH_API int synth_dev_fp8_codes(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t n_experts,
                                  int64_t rows, int64_t K, void *out, void *stream) {
    if (K % 16 != 0 || rows <= 0 || n_experts <= 0 || ((uintptr_t)out & 15)) return -1;
    synth_fp8_codes_kernel<<<152 * 8, 256, 0, (cudaStream_t)stream>>>(seed, tensor, e0, rows, K / 16,
                                                                       n_experts, (uint4 *)out);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}

// FP8 block scales: n_experts x ceil(rows/128) x ceil(K/128) fp32.
SYNTH_API int synth_dev_fp8_scales(uint64_t seed, uint32_t tensor, uint32_t e0, int64_t n_experts,
                                   int64_t rows, int64_t K, void *out, void *stream) {
    if (rows <= 0 || K <= 0 || n_experts <= 0 || ((uintptr_t)out & 3)) return -1;
    synth_fp8_scales_kernel<<<152 * 4, 256, 0, (cudaStream_t)stream>>>(
        seed, tensor, e0, (rows + 127) / 128, (K + 127) / 128, n_experts, (uint32_t *)out);
    return cudaGetLastError() == cudaSuccess ? 0 : -2;
}
