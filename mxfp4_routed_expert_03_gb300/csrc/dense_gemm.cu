// Dense bf16 GEMMs on tcgen05 tensor cores (kind::f16, fp32 accumulation in
// TMEM) for the layer's non-routed parts, both kept in the resident static
// tier (Moonshine README, "How the engine works"):
//   - the router, logits[t][e] = sum_d x[t][d] * W_r[e][d] in fp32. W_r is
//     split once into three bf16 terms whose sum is exactly W_r (each term
//     holds the next 8 significant bits), and every product of two bf16
//     values is exact in fp32, so three MMAs per K step against the same bf16
//     x tile give the fp32 products on tensor cores. The tensor core's own
//     accumulator update does not round to nearest (its error grows by about
//     one ulp of the running sum per MMA), so the router MMAs accumulate only
//     one 64-wide K chunk at a time in TMEM; CUDA cores add the chunks with
//     round-to-nearest fp32, which keeps the result at fp32 summation accuracy.
//   - the always-on shared expert: gate/up with SwiGLU in the epilogue (64
//     gate rows stacked over the matching 64 up rows, as in the routed GEMM),
//     h kept in bf16, then down, written as fp32 (weight 1.0).
//
// D[M x N] = sum_terms A_term[M x K] . B[N x K]^T with A and B K-major bf16
// read by TMA with 128-byte swizzle; tiles of 128 A rows x DN tokens. One
// persistent CTA per SM, 7 warps: TMA producer (one thread), MMA issuer (one
// thread), TMEM allocator, 4 epilogue warps; one smem ring, double-buffered
// TMEM accumulators, every wait bounded.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace {

constexpr int DK = 64;               // bf16 per 128-byte row = K per stage
constexpr int DN = MOE_DENSE_NTILE;  // tokens per tile
constexpr int DTHREADS = 224;
constexpr uint32_t DTMEM_COLS = 512;
constexpr uint32_t DACC_COLS = 256;
constexpr int D_A_BYTES = 128 * DK * 2;  // 16 KB per A term
constexpr int D_B_BYTES = DN * DK * 2;   // 24 KB

template <int EPI>
struct DCfg {
    static constexpr int NTERMS = 1;
    static constexpr int MROWS = (EPI == MOE_DENSE_SWIGLU) ? 64 : 128;  // output rows per tile
    static constexpr int STAGE = NTERMS * D_A_BYTES + D_B_BYTES;
    static constexpr int S = 5;
    static constexpr int BAR_BASE = S * STAGE;
    static constexpr int EPI_BASE = BAR_BASE + 256;  // barriers, TMEM slot, abort flag
    static constexpr int EPI_BYTES = (EPI == MOE_DENSE_SWIGLU) ? 16 * 64 * 4 : 0;
    static constexpr int SMEM = 1024 + EPI_BASE + EPI_BYTES;
    static_assert(STAGE % 1024 == 0, "stage alignment (128-byte swizzle atoms)");
    static_assert((2 * S + 5) * 8 + 12 <= 256, "barrier area");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(DN % 16 == 0 && DN <= 256 && 2 * DN <= (int)DTMEM_COLS, "tile width");
};

// The four epilogue warps (128 threads) meet at named barrier 1.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(DTHREADS, 1) moe_dense_gemm_kernel(
    const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mA1,
    const __grid_constant__ CUtensorMap mA2, const __grid_constant__ CUtensorMap mB,
    const MoeDenseArgs args) {
    using C = DCfg<EPI>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + C::BAR_BASE);
    uint64_t *empty = full + C::S;
    uint64_t *tfull = empty + C::S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;  // the issuer's MMAs in flight, waited on when giving up
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    int *abort_flag = (int *)(tmem_slot + 1);
    int *s_issued = abort_flag + 1;  // stages the producer filled
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        *abort_flag = 0;
        *s_issued = 0;
        for (int s = 0; s < C::S; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 4);
        }
        tc::mbar_init(drain, 1);
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, DTMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Tiles run m fastest: the CTAs of one wave share a few token tiles and
    // sweep all of A, which (router or shared weights) stays in L2.
    const int MT = (args.M + C::MROWS - 1) / C::MROWS;
    const int NT = (args.N + DN - 1) / DN, KC = args.K / DK;
    const int total = MT * NT;
    const long long LIMIT = args.timeout_cycles;
    volatile int *abort_p = abort_flag;
    auto fail = [&](void) {
        *abort_p = 1;
        moe_flag(args.status, MOE_ERR_DEVICE_TIMEOUT);
    };
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = tc::policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int mt = tile % MT, nt = tile / MT;
                for (int kc = 0; kc < KC; ++kc) {
                    const int s = it % C::S, round = it / C::S;
                    if (round > 0 && !tc::mbar_wait(&empty[s], (round - 1) & 1, LIMIT, abort_p)) {
                        fail();
                        ok = false;
                        break;
                    }
                    unsigned char *st = smem + s * C::STAGE;
                    tc::mbar_arrive_expect_tx(&full[s],
                                              (uint32_t)(C::NTERMS * D_A_BYTES + D_B_BYTES));
                    ++it;  // a fill of this stage is now in flight
                    const int row0 = mt * C::MROWS;
                    tc::tma_load_2d(st, &mA0, &full[s], kc * DK, row0, pol);
                    if (EPI == MOE_DENSE_SWIGLU)  // the matching up rows under the gate rows
                        tc::tma_load_2d(st + 64 * 128, &mA1, &full[s], kc * DK, row0, pol);
                    tc::tma_load_2d(st + C::NTERMS * D_A_BYTES, &mB, &full[s], kc * DK, nt * DN,
                                    pol);
                }
            }
            *s_issued = it;
        }
    } else if (warp == 2) {
        if (lane == 0) {
            int it = 0, lt = 0;
            bool ok = true;
            uint64_t *last = nullptr;
            uint32_t last_par = 0;
            const uint32_t idesc = tc::idesc_bf16(128, DN);
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++lt) {
                const int buf = lt & 1, use = lt >> 1;
                if (use > 0 && !tc::mbar_wait(&tempty[buf], (use - 1) & 1, LIMIT, abort_p)) {
                    fail();
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t acc = tmem + buf * DACC_COLS;
                for (int kc = 0; kc < KC; ++kc, ++it) {
                    const int s = it % C::S, round = it / C::S;
                    if (!tc::mbar_wait(&full[s], round & 1, LIMIT, abort_p)) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    unsigned char *st = smem + s * C::STAGE;
                    const uint32_t b_s = tc::smem_u32(st + C::NTERMS * D_A_BYTES);
#pragma unroll
                    for (int k = 0; k < DK / 16; ++k)
                        tc::mma_bf16(acc, tc::sdesc_sw128(tc::smem_u32(st) + 32 * k),
                                 tc::sdesc_sw128(b_s + 32 * k), idesc, (kc > 0 || k > 0) ? 1u : 0u);
                    tc::mma_commit(&empty[s]);
                    last = &empty[s];
                    last_par = round & 1;
                }
                if (!ok) break;
                tc::mma_commit(&tfull[buf]);
            }
            // the last MMAs must finish before the CTA releases TMEM
            if (ok && last && !tc::mbar_wait(last, last_par, LIMIT, abort_p)) fail();
            if (!ok || *abort_p) tc::drain_mmas(drain, LIMIT);
        }
        __syncwarp();
    } else if (warp >= 3) {
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int lt = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++lt) {
            const int mt = tile % MT, nt = tile / MT;
            const int buf = lt & 1, use = lt >> 1;
            const bool got = tc::mbar_wait(&tfull[buf], use & 1, LIMIT, abort_p);
            if (!tc::bar_and(1, 128, got)) {  // all four warps stop together
                if (!got && lane == 0) fail();
                break;
            }
            tc::tc_fence_after();
            const uint32_t acc = tmem + lane_base + buf * DACC_COLS;
            const int ncols = min(DN, args.N - nt * DN);
            for (int c0 = 0; c0 < ncols; c0 += 16) {
                uint32_t r[16];
                tc::tmem_ld_32x32b_x16(acc + c0, r);
                tc::tmem_ld_wait();
                if (EPI == MOE_DENSE_SWIGLU) {
                    // Lanes 0..63 hold gate rows, 64..127 the same up rows. Gate
                    // warps finish columns 0..7 of the chunk, up warps 8..15; each
                    // hands the other half to its partner through shared memory.
                    float *stg = (float *)(smem + C::EPI_BASE);  // [16 columns][64 rows]
                    const bool gate = q < 2;
                    const int rr = (q & 1) * 32 + lane;
#pragma unroll
                    for (int j = 0; j < 8; ++j)  // constant register indices, no local memory
                        stg[(gate ? j + 8 : j) * 64 + rr] = __uint_as_float(gate ? r[j + 8] : r[j]);
                    epi_sync();
                    const int f = mt * 64 + rr;
#pragma unroll
                    for (int j0 = 0; j0 < 8; ++j0) {
                        const int j = gate ? j0 : j0 + 8;
                        const float own = __uint_as_float(gate ? r[j0] : r[j0 + 8]);
                        const float other = stg[j * 64 + rr];
                        const float g = gate ? own : other;
                        const float u = gate ? other : own;
                        if (c0 + j < ncols)
                            args.out_bf16[(size_t)(nt * DN + c0 + j) * args.ldo + f] =
                                f32_to_bf16_bits(g / (1.f + expf(-g)) * u);
                    }
                    epi_sync();
                } else {
                    const int m = mt * 128 + q * 32 + lane;
                    if (m < args.M) {
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < ncols)
                                args.out_f32[(size_t)(nt * DN + c0 + j) * args.ldo + m] =
                                    __uint_as_float(r[j]);
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&tempty[buf]);
        }
    }
    __syncthreads();
    if (*abort_p && tid == 0) tc::wait_issued_fills(full, C::S, *s_issued, LIMIT);
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, DTMEM_COLS);
    }
}


// ---------------------------------------------------------------------------
// Router GEMM: logits[t][e] with the three W_r terms and chunked accumulation.
// Warps: 0 TMA producer, 1 TMEM allocator, 2 MMA issuer, 3..10 epilogue (two
// warps per TMEM lane quadrant, 96 token columns each, holding the fp32
// running sums of their 32 experts x 96 tokens in registers).
// ---------------------------------------------------------------------------
namespace {
constexpr int RTHREADS = 352;
constexpr int R_S = 3;
constexpr int R_STAGE = 3 * D_A_BYTES + D_B_BYTES;
constexpr int R_BAR = R_S * R_STAGE;
constexpr int R_SMEM = 1024 + R_BAR + 256;
constexpr int R_HALF = DN / 2;  // token columns per epilogue warp
static_assert(R_STAGE % 1024 == 0 && R_SMEM <= 232448, "router smem");
static_assert(R_HALF % 48 == 0, "epilogue drains 48 columns per batch");
}  // namespace

__global__ void __launch_bounds__(RTHREADS, 1) moe_router_gemm_kernel(
    const __grid_constant__ CUtensorMap mT0, const __grid_constant__ CUtensorMap mT1,
    const __grid_constant__ CUtensorMap mT2, const __grid_constant__ CUtensorMap mX,
    const MoeDenseArgs args) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + R_BAR);
    uint64_t *empty = full + R_S;
    uint64_t *cfull = empty + R_S;  // chunk accumulator c % 2 holds chunk c
    uint64_t *cempty = cfull + 2;
    uint64_t *drain = cempty + 2;  // the issuer's MMAs in flight, waited on when giving up
    uint32_t *tmem_slot = (uint32_t *)(drain + 1);
    int *abort_flag = (int *)(tmem_slot + 1);
    int *s_issued = abort_flag + 1;  // stages the producer filled
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        *abort_flag = 0;
        *s_issued = 0;
        tc::mbar_init(drain, 1);
        for (int s = 0; s < R_S; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&cfull[b], 1);
            tc::mbar_init(&cempty[b], 8);
        }
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, DTMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int MT = (args.M + 127) / 128, NT = (args.N + DN - 1) / DN, KC = args.K / DK;
    const int total = MT * NT;
    const long long LIMIT = args.timeout_cycles;
    volatile int *abort_p = abort_flag;
    auto fail = [&](void) {
        *abort_p = 1;
        moe_flag(args.status, MOE_ERR_DEVICE_TIMEOUT);
    };
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = tc::policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int mt = tile % MT, nt = tile / MT;
                for (int kc = 0; kc < KC; ++kc) {
                    const int s = it % R_S, round = it / R_S;
                    if (round > 0 && !tc::mbar_wait(&empty[s], (round - 1) & 1, LIMIT, abort_p)) {
                        fail();
                        ok = false;
                        break;
                    }
                    unsigned char *st = smem + s * R_STAGE;
                    tc::mbar_arrive_expect_tx(&full[s], (uint32_t)R_STAGE);
                    ++it;  // a fill of this stage is now in flight
                    tc::tma_load_2d(st, &mT0, &full[s], kc * DK, mt * 128, pol);
                    tc::tma_load_2d(st + D_A_BYTES, &mT1, &full[s], kc * DK, mt * 128, pol);
                    tc::tma_load_2d(st + 2 * D_A_BYTES, &mT2, &full[s], kc * DK, mt * 128, pol);
                    tc::tma_load_2d(st + 3 * D_A_BYTES, &mX, &full[s], kc * DK, nt * DN, pol);
                }
            }
            *s_issued = it;
        }
    } else if (warp == 2) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(128, DN);
            int it = 0;
            bool ok = true;
            uint64_t *last = nullptr;
            uint32_t last_par = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                for (int kc = 0; kc < KC; ++kc, ++it) {
                    const int s = it % R_S, round = it / R_S;
                    const int cb = it & 1, use = it >> 1;
                    if (!tc::mbar_wait(&full[s], round & 1, LIMIT, abort_p) ||
                        (use > 0 && !tc::mbar_wait(&cempty[cb], (use - 1) & 1, LIMIT, abort_p))) {
                        fail();
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    unsigned char *st = smem + s * R_STAGE;
                    const uint32_t b_s = tc::smem_u32(st + 3 * D_A_BYTES);
                    const uint32_t acc = tmem + cb * DACC_COLS;
                    // smallest term first: most truncating updates then act on a
                    // running sum 2^8 or 2^16 times smaller than the chunk's
#pragma unroll
                    for (int term = 2; term >= 0; --term) {
#pragma unroll
                        for (int k = 0; k < DK / 16; ++k)
                            tc::mma_bf16(acc, tc::sdesc_sw128(tc::smem_u32(st + term * D_A_BYTES) + 32 * k),
                                     tc::sdesc_sw128(b_s + 32 * k), idesc,
                                     (k > 0 || term < 2) ? 1u : 0u);
                    }
                    tc::mma_commit(&empty[s]);
                    tc::mma_commit(&cfull[cb]);
                    last = &cfull[cb];
                    last_par = use & 1;
                }
            }
            // the last MMAs must finish before the CTA releases TMEM
            if (ok && last && !tc::mbar_wait(last, last_par, LIMIT, abort_p)) fail();
            if (!ok || *abort_p) tc::drain_mmas(drain, LIMIT);
        }
        __syncwarp();
    } else if (warp >= 3) {
        const int q = warp & 3;               // TMEM lane quadrant this warp may access
        const int col0 = ((warp - 3) >> 2) * R_HALF;  // first token column of this warp
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const int mt = tile % MT, nt = tile / MT;
            float sum[R_HALF];
#pragma unroll
            for (int j = 0; j < R_HALF; ++j) sum[j] = 0.f;
            for (int kc = 0; kc < KC; ++kc, ++it) {
                const int cb = it & 1, use = it >> 1;
                if (!tc::mbar_wait(&cfull[cb], use & 1, LIMIT, abort_p)) {
                    if (lane == 0) fail();
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t acc = tmem + lane_base + cb * DACC_COLS + col0;
#pragma unroll
                for (int b = 0; b < R_HALF; b += 48) {
                    uint32_t r0[16], r1[16], r2[16];
                    tc::tmem_ld_32x32b_x16(acc + b, r0);
                    tc::tmem_ld_32x32b_x16(acc + b + 16, r1);
                    tc::tmem_ld_32x32b_x16(acc + b + 32, r2);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        sum[b + j] += __uint_as_float(r0[j]);
                        sum[b + 16 + j] += __uint_as_float(r1[j]);
                        sum[b + 32 + j] += __uint_as_float(r2[j]);
                    }
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&cempty[cb]);
            }
            if (!ok) break;
            const int m = mt * 128 + q * 32 + lane;
            const int t0 = nt * DN + col0;
            if (m < args.M) {
#pragma unroll
                for (int j = 0; j < R_HALF; ++j)
                    if (t0 + j < args.N) args.out_f32[(size_t)(t0 + j) * args.ldo + m] = sum[j];
            }
        }
    }
    __syncthreads();
    if (*abort_p && tid == 0) tc::wait_issued_fills(full, R_S, *s_issued, LIMIT);
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, DTMEM_COLS);
    }
}

// W (fp32, n values) -> three bf16 terms with w = t0 + t1 + t2: t0 is the
// round-to-nearest bf16 of w, t1 of the residual w - t0, t2 of what remains.
__global__ void __launch_bounds__(256) moe_split3_kernel(int64_t n, const float *__restrict__ w,
                                                         uint16_t *__restrict__ t0,
                                                         uint16_t *__restrict__ t1,
                                                         uint16_t *__restrict__ t2) {
    const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i >= n) return;
    float r = w[i];
    const uint16_t a = f32_to_bf16_bits(r);
    r -= bf16_bits_to_f32(a);
    const uint16_t b = f32_to_bf16_bits(r);
    r -= bf16_bits_to_f32(b);
    t0[i] = a;
    t1[i] = b;
    t2[i] = f32_to_bf16_bits(r);
}

cudaError_t moe_launch_split3(int64_t n, const float *w, uint16_t *t0, uint16_t *t1, uint16_t *t2,
                              cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    moe_split3_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n, w, t0, t1, t2);
    return cudaGetLastError();
}

int moe_dense_tiles(int epi, int M, int N) {
    const int mrows = epi == MOE_DENSE_SWIGLU ? 64 : 128;
    return ((M + mrows - 1) / mrows) * ((N + DN - 1) / DN);
}

namespace {
template <int EPI>
cudaError_t launch_dense(const CUtensorMap *a0, const CUtensorMap *a1, const CUtensorMap *a2,
                         const CUtensorMap *b, const MoeDenseArgs *args, int grid,
                         cudaStream_t st) {
    auto kern = moe_dense_gemm_kernel<EPI>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, DCfg<EPI>::SMEM);
    if (err != cudaSuccess) return err;
    kern<<<grid, DTHREADS, DCfg<EPI>::SMEM, st>>>(*a0, *a1, *a2, *b, *args);
    return cudaGetLastError();
}
}  // namespace

cudaError_t moe_launch_dense(int epi, const CUtensorMap *a0, const CUtensorMap *a1,
                             const CUtensorMap *a2, const CUtensorMap *b,
                             const MoeDenseArgs *args, int grid, cudaStream_t st) {
    if (args->K % DK || args->M <= 0 || args->N <= 0 || grid <= 0) return cudaErrorInvalidValue;
    switch (epi) {
        case MOE_DENSE_ROUTER: {
            cudaError_t err = cudaFuncSetAttribute(
                moe_router_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
            if (err != cudaSuccess) return err;
            moe_router_gemm_kernel<<<grid, RTHREADS, R_SMEM, st>>>(*a0, *a1, *a2, *b, *args);
            return cudaGetLastError();
        }
        case MOE_DENSE_SWIGLU: return launch_dense<MOE_DENSE_SWIGLU>(a0, a1, a2, b, args, grid, st);
        case MOE_DENSE_STORE: return launch_dense<MOE_DENSE_STORE>(a0, a1, a2, b, args, grid, st);
        default: return cudaErrorInvalidValue;
    }
}
