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
// row's fp32 sum. The activation row is held in shared memory as f16 (bf16 ->
// f16 is exact for |x| in [2^-14, 65504), the range of these inputs).
// In the down projection the intermediate h stays fp32 and the codes are
// widened to fp32.
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

// acc + lo(a)*lo(b) + hi(a)*hi(b), products exact, sums in fp32.
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc)
        : "r"(a), "r"(b));
    return acc;
}

// Dot product of one 32-element MX block (16 code bytes) with 32 f16
// activations (as 16 f16x2 words), fp32 result before the block scale.
__device__ __forceinline__ float block_dot_f16(const uint4 &q, const uint4 *xs) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 xv = xs[i];  // elements 8i .. 8i+7
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int b = 0; b < 4; ++b) acc = fma2_f16_f32(e2m1x2_to_f16x2((w[i] >> (8 * b)) & 0xFF), xw[b], acc);
    }
    return acc;
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

// ---------------------------------------------------------------------------
// Gate/up + SwiGLU. grid = (F / ROWS, max active experts); each CTA handles
// ROWS consecutive f of one expert for all of its tokens, NT tokens at a time.
// Lanes are grouped LPR per row; each lane owns PER_LANE MX blocks of the row.
// h[slot][f] = silu(g) * u (fp32), slot = position in the plan's perm order.
// ---------------------------------------------------------------------------
template <int PER_LANE, int NT>
__global__ void __launch_bounds__(256) moe_decode_gateup_kernel(
    int D, int F, int E, int k, int n_rows, int rows_per_cta, const uint16_t *__restrict__ x,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const int32_t *__restrict__ active, const uint8_t *__restrict__ gate_q,
    const uint8_t *__restrict__ gate_s, const uint8_t *__restrict__ up_q,
    const uint8_t *__restrict__ up_s, float *__restrict__ h, int *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    __half *xs = (__half *)smem;  // [NT][D]
    int e, s0, n;
    if (!segment_of(blockIdx.y, E, n_rows, active, offsets, e, s0, n, status)) return;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nblk = D / 32;               // MX blocks per row
    const int LPR = nblk / PER_LANE;       // lanes per row (power of two <= 32)
    const int RPW = 32 / LPR;              // rows per warp pass
    const int sub = lane % LPR, grp = lane / LPR;
    const int f_begin = blockIdx.x * rows_per_cta;
    const int f_end = min(F, f_begin + rows_per_cta);
    const size_t qrow = (size_t)D / 2, srow = (size_t)nblk;
    const uint8_t *gq = gate_q + (size_t)e * F * qrow, *uq = up_q + (size_t)e * F * qrow;
    const uint8_t *gs = gate_s + (size_t)e * F * srow, *us = up_s + (size_t)e * F * srow;

    for (int g0 = 0; g0 < n; g0 += NT) {
        const int nt = min(NT, n - g0);
        __syncthreads();
        // Stage the group's activation rows as f16.
        for (int i = threadIdx.x; i < nt * (D / 2); i += blockDim.x) {
            int tl = i / (D / 2), c = i % (D / 2);
            int fl = perm[s0 + g0 + tl];
            if (fl < 0 || fl >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); fl = 0; }
            int t = fl / k;
            uint32_t two = ((const uint32_t *)(x + (size_t)t * D))[c];
            float2 v = make_float2(bf16_bits_to_f32(two & 0xFFFF), bf16_bits_to_f32(two >> 16));
            ((__half2 *)xs)[(size_t)tl * (D / 2) + c] = __float22half2_rn(v);
        }
        __syncthreads();
        for (int f = f_begin + wid * RPW + grp; f - grp < f_end; f += 8 * RPW) {
            const bool row_ok = f < f_end;
            uint4 gqv[PER_LANE], uqv[PER_LANE];
            float gsc[PER_LANE], usc[PER_LANE];
#pragma unroll
            for (int p = 0; p < PER_LANE; ++p) {
                int b = sub + LPR * p;
                if (row_ok) {
                    gqv[p] = __ldg((const uint4 *)(gq + (size_t)f * qrow) + b);
                    uqv[p] = __ldg((const uint4 *)(uq + (size_t)f * qrow) + b);
                    gsc[p] = e8m0_to_f32(__ldg(gs + (size_t)f * srow + b));
                    usc[p] = e8m0_to_f32(__ldg(us + (size_t)f * srow + b));
                } else {
                    gqv[p] = uqv[p] = make_uint4(0, 0, 0, 0);
                    gsc[p] = usc[p] = 0.f;
                }
            }
            float ag[NT], au[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                ag[j] = 0.f;
                au[j] = 0.f;
                if (j < nt) {
#pragma unroll
                    for (int p = 0; p < PER_LANE; ++p) {
                        int b = sub + LPR * p;
                        const uint4 *xb = (const uint4 *)(xs + (size_t)j * D + 32 * b);
                        ag[j] = fmaf(block_dot_f16(gqv[p], xb), gsc[p], ag[j]);
                        au[j] = fmaf(block_dot_f16(uqv[p], xb), usc[p], au[j]);
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
                    if (j < nt) h[(size_t)(s0 + g0 + j) * F + f] = silu_f(ag[j]) * au[j];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Down projection: y[slot][d] = sum_f W_down[e][d][f] * h[slot][f] (fp32).
// ---------------------------------------------------------------------------
template <int PER_LANE, int NT>
__global__ void __launch_bounds__(256) moe_decode_down_kernel(
    int D, int F, int E, int n_rows, int rows_per_cta, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ active, const uint8_t *__restrict__ down_q,
    const uint8_t *__restrict__ down_s, const float *__restrict__ h, float *__restrict__ y,
    int *status) {
    extern __shared__ __align__(16) unsigned char smem[];
    float *hs = (float *)smem;  // [NT][F]
    int e, s0, n;
    if (!segment_of(blockIdx.y, E, n_rows, active, offsets, e, s0, n, status)) return;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nblk = F / 32;
    const int LPR = nblk / PER_LANE;
    const int RPW = 32 / LPR;
    const int sub = lane % LPR, grp = lane / LPR;
    const int d_begin = blockIdx.x * rows_per_cta;
    const int d_end = min(D, d_begin + rows_per_cta);
    const size_t qrow = (size_t)F / 2, srow = (size_t)nblk;
    const uint8_t *dq = down_q + (size_t)e * D * qrow;
    const uint8_t *ds = down_s + (size_t)e * D * srow;

    for (int g0 = 0; g0 < n; g0 += NT) {
        const int nt = min(NT, n - g0);
        __syncthreads();
        for (int i = threadIdx.x; i < nt * (F / 4); i += blockDim.x) {
            int tl = i / (F / 4), c = i % (F / 4);
            ((float4 *)hs)[(size_t)tl * (F / 4) + c] =
                ((const float4 *)(h + (size_t)(s0 + g0 + tl) * F))[c];
        }
        __syncthreads();
        for (int d = d_begin + wid * RPW + grp; d - grp < d_end; d += 8 * RPW) {
            const bool row_ok = d < d_end;
            uint4 qv[PER_LANE];
            float sc[PER_LANE];
#pragma unroll
            for (int p = 0; p < PER_LANE; ++p) {
                int b = sub + LPR * p;
                if (row_ok) {
                    qv[p] = __ldg((const uint4 *)(dq + (size_t)d * qrow) + b);
                    sc[p] = e8m0_to_f32(__ldg(ds + (size_t)d * srow + b));
                } else {
                    qv[p] = make_uint4(0, 0, 0, 0);
                    sc[p] = 0.f;
                }
            }
            float acc[NT];
#pragma unroll
            for (int j = 0; j < NT; ++j) acc[j] = 0.f;
#pragma unroll
            for (int p = 0; p < PER_LANE; ++p) {
                int b = sub + LPR * p;
                const uint32_t w[4] = {qv[p].x, qv[p].y, qv[p].z, qv[p].w};
                float part[NT];
#pragma unroll
                for (int j = 0; j < NT; ++j) part[j] = 0.f;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb) {
                        float2 wf = f16x2_to_float2(e2m1x2_to_f16x2((w[i] >> (8 * bb)) & 0xFF));
                        int kk = 32 * b + 8 * i + 2 * bb;
#pragma unroll
                        for (int j = 0; j < NT; ++j) {
                            if (j < nt) {
                                float2 hv = *(const float2 *)(hs + (size_t)j * F + kk);
                                part[j] = fmaf(wf.x, hv.x, part[j]);
                                part[j] = fmaf(wf.y, hv.y, part[j]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[j] = fmaf(part[j], sc[p], acc[j]);
            }
#pragma unroll
            for (int j = 0; j < NT; ++j) {
#pragma unroll
                for (int off = 1; off < 32; off <<= 1)
                    if (off < LPR) acc[j] += __shfl_xor_sync(FULL_MASK, acc[j], off);
            }
            if (row_ok && sub == 0) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    if (j < nt) y[(size_t)(s0 + g0 + j) * D + d] = acc[j];
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Combine: out[t][d] = bf16( sum_j w[t][j] * y[inv[t*k+j]][d] ), j ascending.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_combine_slots_kernel(int T, int D, int k, int n_rows,
                                                                const float *__restrict__ topk_w,
                                                                const int32_t *__restrict__ inv,
                                                                const float *__restrict__ y,
                                                                uint16_t *__restrict__ out,
                                                                int *status) {
    int t = blockIdx.y;
    int d4 = blockIdx.x * blockDim.x + threadIdx.x;  // group of 4 columns
    if (t >= T || d4 * 4 >= D) return;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        int slot = inv[(size_t)t * k + j];
        if (slot < 0 || slot >= n_rows) { moe_flag(status, MOE_ERR_BAD_INDEX); continue; }
        float w = topk_w[(size_t)t * k + j];
        float4 v = ((const float4 *)(y + (size_t)slot * D))[d4];
        acc.x = fmaf(w, v.x, acc.x);
        acc.y = fmaf(w, v.y, acc.y);
        acc.z = fmaf(w, v.z, acc.z);
        acc.w = fmaf(w, v.w, acc.w);
    }
    uint2 o;
    o.x = (uint32_t)f32_to_bf16_bits(acc.x) | ((uint32_t)f32_to_bf16_bits(acc.y) << 16);
    o.y = (uint32_t)f32_to_bf16_bits(acc.z) | ((uint32_t)f32_to_bf16_bits(acc.w) << 16);
    ((uint2 *)(out + (size_t)t * D))[d4] = o;
}

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
namespace {
constexpr int kDecodeNT = 4;
constexpr int kRowsPerCta = 16;

template <int P>
cudaError_t launch_gateup(dim3 g, size_t sm, cudaStream_t st, int D, int F, int E, int k,
                          int n_rows, const uint16_t *x, const moe_plan_buf *p,
                          const moe_weights *w, float *h, int *status) {
    auto kern = moe_decode_gateup_kernel<P, kDecodeNT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (err != cudaSuccess) return err;
    kern<<<g, 256, sm, st>>>(D, F, E, k, n_rows, kRowsPerCta, x, p->offsets, p->perm, p->active,
                             w->gate_q, w->gate_s, w->up_q, w->up_s, h, status);
    return cudaGetLastError();
}

template <int P>
cudaError_t launch_down(dim3 g, size_t sm, cudaStream_t st, int D, int F, int E, int n_rows,
                        const moe_plan_buf *p, const moe_weights *w, const float *h, float *y,
                        int *status) {
    auto kern = moe_decode_down_kernel<P, kDecodeNT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (err != cudaSuccess) return err;
    kern<<<g, 256, sm, st>>>(D, F, E, n_rows, kRowsPerCta, p->offsets, p->active, w->down_q,
                             w->down_s, h, y, status);
    return cudaGetLastError();
}
}  // namespace

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

size_t moe_decode_ws_bytes(int T, int D, int F, int k) {
    size_t rows = (size_t)T * k;
    return rows * F * sizeof(float) + rows * D * sizeof(float);
}

cudaError_t moe_launch_decode(int T, int D, int F, int E, int k, const uint16_t *x,
                              const moe_plan_buf *p, const moe_weights *w, uint16_t *out,
                              void *ws, int *status, cudaStream_t st) {
    const int n_rows = T * k;
    float *h = (float *)ws;
    float *y = h + (size_t)n_rows * F;
    const int max_active = n_rows < E ? n_rows : E;
    cudaError_t err;
    {
        dim3 g((F + kRowsPerCta - 1) / kRowsPerCta, max_active);
        size_t sm = (size_t)kDecodeNT * D * sizeof(__half);
        switch (moe_decode_per_lane(D)) {
            case 1: err = launch_gateup<1>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 2: err = launch_gateup<2>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 3: err = launch_gateup<3>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 4: err = launch_gateup<4>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 5: err = launch_gateup<5>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 6: err = launch_gateup<6>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 7: err = launch_gateup<7>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            case 8: err = launch_gateup<8>(g, sm, st, D, F, E, k, n_rows, x, p, w, h, status); break;
            default: return cudaErrorInvalidValue;
        }
        if (err != cudaSuccess) return err;
    }
    {
        dim3 g((D + kRowsPerCta - 1) / kRowsPerCta, max_active);
        size_t sm = (size_t)kDecodeNT * F * sizeof(float);
        switch (moe_decode_per_lane(F)) {
            case 1: err = launch_down<1>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 2: err = launch_down<2>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 3: err = launch_down<3>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 4: err = launch_down<4>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 5: err = launch_down<5>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 6: err = launch_down<6>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 7: err = launch_down<7>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            case 8: err = launch_down<8>(g, sm, st, D, F, E, n_rows, p, w, h, y, status); break;
            default: return cudaErrorInvalidValue;
        }
        if (err != cudaSuccess) return err;
    }
    dim3 g((D / 4 + 255) / 256, T);
    moe_combine_slots_kernel<<<g, 256, 0, st>>>(T, D, k, n_rows, p->topk_w, p->inv, y, out, status);
    return cudaGetLastError();
}
