// Grouped block-scaled MXFP4 GEMMs on tcgen05 tensor cores (layer-major
// prefill): GEMM1 computes gate and up for a tile of 128 intermediate rows of
// one expert against up to 112 of that expert's routed tokens and applies
// SwiGLU in the epilogue; GEMM2 computes the down projection and adds the
// routing-weighted result into the token's fp32 output row.
//
// The pages' prefill "groups all rows selecting each expert" and reads only
// the selected experts (Moonshine README, "How the engine works"; Moonshine
// GitHub README, "Prefill"); each selected expert's FFN runs on MXFP4 weights
// (MoonTail, "Routed expert FFN"; Moonshine GitHub README, "MXFP4 kernels"),
// and the weighted reduction closes the MoE tail (Moonshine README,
// "Run layer-major prefill").
//
// Tensor-core formulation (kind::mxf8f6f4, block scale 1X): D[128 x N] in
// TMEM accumulates A[128 x K] (weights, E2M1 codes, one E8M0 scale per 32 K)
// times B[N x K]^T (activations, E4M3, one E8M0 scale per 32 K). Activations
// enter as a two-term split (hi + lo, see mx8.cuh): both terms run against the
// same weight tile into the same accumulator, so weights are read once.
//
// One persistent CTA per SM, 7 warps:
//   warp 0      TMA producer: weight tiles (2D, packed E2M1 expanded by TMA),
//               activation tiles (gather4 of token rows for GEMM1, 2D for GEMM2)
//   warp 1      scale producer (cp.async of 4-byte scale groups into the
//               128x4 scale atom layout) and TMEM allocator
//   warp 2      MMA issuer (one thread): tcgen05.cp scales, tcgen05.mma
//   warps 3-6   epilogue, one 32-lane TMEM quadrant each
// Stages ring through mbarriers; accumulators are double-buffered in TMEM so
// the epilogue of tile i overlaps the MMAs of tile i+1. Every wait is bounded:
// on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT and winds down.
#include "common.cuh"
#include "kernels.h"
#include "mx8.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int BM = 128;                 // weight rows per tile
constexpr int BK = 128;                 // K elements per stage
constexpr int NTMAX = MOE_GEMM_NTMAX;   // token rows per tile
constexpr int A_BYTES = BM * BK;        // smem bytes of one weight tile (E2M1 padded to 8 bit)
constexpr int A_TX = BM * BK / 2;       // bytes the TMA moves for it (packed)
constexpr int B_BYTES = NTMAX * BK;     // smem bytes of one activation term tile
constexpr int SF_BYTES = 512;           // one 128-row x 4-block scale atom
constexpr int NUM_THREADS = 224;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t SF_TMEM_COL = 448;   // scale atoms: 2 slots x 16 columns

template <int MODE>
struct Cfg {
    static constexpr int NA = (MODE == MOE_GEMM_GATEUP) ? 2 : 1;        // weight operands
    static constexpr int STAGES = (MODE == MOE_GEMM_GATEUP) ? 3 : 4;
    static constexpr int STAGE_BYTES = NA * A_BYTES + 2 * B_BYTES + 4 * SF_BYTES;
    static constexpr int OFF_B_HI = NA * A_BYTES;
    static constexpr int OFF_B_LO = OFF_B_HI + B_BYTES;
    static constexpr int OFF_SF = OFF_B_LO + B_BYTES;
    static constexpr int ACC_STRIDE = NA * NTMAX;  // TMEM columns per accumulator buffer
};

struct Tile {
    int e;      // expert
    int m0;     // first weight row (within the expert)
    int s0;     // first slot of the tile (position in perm order)
    int n;      // valid token rows
    int nmma;   // n rounded up to 16 (MMA N)
};

__device__ __forceinline__ bool tile_at(int tile, int n_active, int MT, const int *s_prefix,
                                        const int32_t *active, const int32_t *offsets, int E,
                                        int n_rows, Tile &t) {
    int lo = 0, hi = n_active - 1;
    while (lo < hi) {  // last a with MT * prefix[a] <= tile
        int mid = (lo + hi + 1) >> 1;
        if (MT * s_prefix[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    int a = lo;
    int ntt = s_prefix[a + 1] - s_prefix[a];
    if (ntt <= 0) return false;
    int local = tile - MT * s_prefix[a];
    int m = local / ntt, j = local % ntt;
    int e = active[1 + a];
    if (e < 0 || e >= E) return false;
    int sb = offsets[e], cnt = offsets[e + 1] - sb;
    if (sb < 0 || cnt <= 0 || sb + cnt > n_rows) return false;
    int r0 = (int)((long long)j * cnt / ntt), r1 = (int)((long long)(j + 1) * cnt / ntt);
    t.e = e;
    t.m0 = m * BM;
    t.s0 = sb + r0;
    t.n = r1 - r0;
    t.nmma = (t.n + 15) & ~15;
    return t.n > 0 && t.n <= NTMAX;
}

// Position of (row m, 32-wide K block c of the stage) inside a 128x4 scale atom.
__device__ __forceinline__ int atom_off(int m, int c) { return (m & 31) * 16 + (m >> 5) * 4 + c; }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1) moe_grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapA2,
    const __grid_constant__ CUtensorMap mapBhi, const __grid_constant__ CUtensorMap mapBlo,
    const MoeGemmArgs args) {
    using C = Cfg<MODE>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem =
        (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + C::STAGES;
    uint64_t *tfull = empty + C::STAGES;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = (uint32_t *)(tempty + 2);
    int *s_prefix = (int *)(tmem_slot + 4);
    __shared__ int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = args.E;
    int n_active = args.active[0];
    if (n_active < 0 || n_active > E) n_active = 0;
    for (int i = tid; i <= n_active; i += NUM_THREADS) s_prefix[i] = args.tt_prefix[i];
    if (tid == 0) {
        abort_flag = 0;
        for (int s = 0; s < C::STAGES; ++s) {
            tc::mbar_init(&full[s], 1 + 32);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 4);
        }
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int MT = args.MT, KC = args.KC;
    const int total_tiles = n_active > 0 ? s_prefix[n_active] * MT : 0;
    const long long LIMIT = args.timeout_cycles;
    volatile int *abort_p = &abort_flag;
    auto fail = [&](void) {
        abort_flag = 1;
        moe_flag(args.status, MOE_ERR_DEVICE_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        const uint64_t pol_w = tc::policy_evict_first();
        const uint64_t pol_x = tc::policy_evict_last();
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t)) {
                if (lane == 0) moe_flag(args.status, MOE_ERR_BAD_INDEX);
                continue;
            }
            // B rows: token rows (GEMM1, gathered 4 at a time) or slots (GEMM2, contiguous)
            const int ngrp = t.nmma / 4;
            const uint32_t tx = (uint32_t)(C::NA * A_TX + 2 * t.nmma * BK);
            for (int kc = 0; kc < KC; ++kc, ++it) {
                const int s = it % C::STAGES, round = it / C::STAGES;
                if (round > 0 && !tc::mbar_wait(&empty[s], (round - 1) & 1, LIMIT, abort_p)) {
                    if (lane == 0) fail();
                    ok = false;
                    break;
                }
                unsigned char *st = smem + s * C::STAGE_BYTES;
                if (lane == 0) {
                    tc::mbar_arrive_expect_tx(&full[s], tx);
                    tc::tma_load_2d(st, &mapA, &full[s], kc * BK, t.e * args.M + t.m0, pol_w);
                    if (C::NA == 2)
                        tc::tma_load_2d(st + A_BYTES, &mapA2, &full[s], kc * BK,
                                        t.e * args.M + t.m0, pol_w);
                }
                __syncwarp();
                if (MODE == MOE_GEMM_GATEUP) {
                    for (int g = lane; g < ngrp; g += 32) {
                        int tok[4];
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            int r = 4 * g + q;
                            int slot = t.s0 + (r < t.n ? r : 0);
                            int fl = args.perm[slot];
                            if (fl < 0 || fl >= args.n_rows) {
                                moe_flag(args.status, MOE_ERR_BAD_INDEX);
                                fl = 0;
                            }
                            tok[q] = fl / args.k;
                        }
                        tc::tma_gather4(st + C::OFF_B_HI + g * 4 * BK, &mapBhi, &full[s], kc * BK,
                                        tok[0], tok[1], tok[2], tok[3], pol_x);
                        tc::tma_gather4(st + C::OFF_B_LO + g * 4 * BK, &mapBlo, &full[s], kc * BK,
                                        tok[0], tok[1], tok[2], tok[3], pol_x);
                    }
                } else {
                    for (int g = lane; g < t.nmma / 16; g += 32) {
                        tc::tma_load_2d(st + C::OFF_B_HI + g * 16 * BK, &mapBhi, &full[s], kc * BK,
                                        t.s0 + 16 * g, pol_x);
                        tc::tma_load_2d(st + C::OFF_B_LO + g * 16 * BK, &mapBlo, &full[s], kc * BK,
                                        t.s0 + 16 * g, pol_x);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ scale producer
        int it = 0;
        bool ok = true;
        const int ksb = args.K / 32;  // scale bytes per row
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t))
                continue;
            // B scale rows handled by this lane (rows lane, lane+32, ...)
            int brows[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                int r = lane + 32 * q;
                brows[q] = -1;
                if (r < t.n) {
                    if (MODE == MOE_GEMM_GATEUP) {
                        int fl = args.perm[t.s0 + r];
                        if (fl < 0 || fl >= args.n_rows) fl = 0;
                        brows[q] = fl / args.k;
                    } else {
                        brows[q] = t.s0 + r;
                    }
                }
            }
            const uint8_t *a_s = args.a_s + ((size_t)t.e * args.M + t.m0) * ksb;
            const uint8_t *a2_s = args.a2_s ? args.a2_s + ((size_t)t.e * args.M + t.m0) * ksb : nullptr;
            for (int kc = 0; kc < KC; ++kc, ++it) {
                const int s = it % C::STAGES, round = it / C::STAGES;
                if (round > 0 && !tc::mbar_wait(&empty[s], (round - 1) & 1, LIMIT, abort_p)) {
                    if (lane == 0) fail();
                    ok = false;
                    break;
                }
                unsigned char *sf = smem + s * C::STAGE_BYTES + C::OFF_SF;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    int m = lane + 32 * q;
                    tc::cp_async_4(sf + atom_off(m, 0), a_s + (size_t)m * ksb + kc * 4);
                    if (C::NA == 2)
                        tc::cp_async_4(sf + SF_BYTES + atom_off(m, 0), a2_s + (size_t)m * ksb + kc * 4);
                    if (brows[q] >= 0) {
                        tc::cp_async_4(sf + 2 * SF_BYTES + atom_off(m, 0),
                                       args.b_s_hi + (size_t)brows[q] * ksb + kc * 4);
                        tc::cp_async_4(sf + 3 * SF_BYTES + atom_off(m, 0),
                                       args.b_s_lo + (size_t)brows[q] * ksb + kc * 4);
                    }
                }
                tc::cp_async_arrive_noinc(&full[s]);
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------------ MMA issuer
        int it = 0, lt = 0;
        bool ok = true;
        uint64_t *last_empty = nullptr;
        uint32_t last_parity = 0;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++lt) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t)) {
                --lt;
                continue;
            }
            const int buf = lt & 1, use = lt >> 1;
            if (use > 0 && !tc::mbar_wait(&tempty[buf], (use - 1) & 1, LIMIT, abort_p)) {
                if (lane == 0) fail();
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t acc0 = tmem + buf * C::ACC_STRIDE;
            const uint32_t acc1 = acc0 + NTMAX;  // GEMM1: up accumulator
            for (int kc = 0; kc < KC; ++kc, ++it) {
                const int s = it % C::STAGES, round = it / C::STAGES;
                if (!tc::mbar_wait(&full[s], round & 1, LIMIT, abort_p)) {
                    if (lane == 0) fail();
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                if (lane == 0) {
                    tc::fence_proxy_async_smem();
                    unsigned char *st = smem + s * C::STAGE_BYTES;
                    const uint32_t sfc = tmem + SF_TMEM_COL + (uint32_t)(it & 1) * 16;
                    const uint32_t sf_s = tc::smem_u32(st + C::OFF_SF);
                    tc::tmem_cp_32x128b_warpx4(sfc + 0, tc::sdesc_plain_32x16(sf_s));
                    if (C::NA == 2)
                        tc::tmem_cp_32x128b_warpx4(sfc + 4, tc::sdesc_plain_32x16(sf_s + SF_BYTES));
                    tc::tmem_cp_32x128b_warpx4(sfc + 8, tc::sdesc_plain_32x16(sf_s + 2 * SF_BYTES));
                    tc::tmem_cp_32x128b_warpx4(sfc + 12, tc::sdesc_plain_32x16(sf_s + 3 * SF_BYTES));
                    const uint32_t a_s = tc::smem_u32(st), b_hi = tc::smem_u32(st + C::OFF_B_HI),
                                   b_lo = tc::smem_u32(st + C::OFF_B_LO);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t idesc =
                            tc::idesc_mxf8f6f4(tc::FMT_E2M1, tc::FMT_E4M3, BM, t.nmma, k, k);
                        const uint32_t acc_first = (kc > 0 || k > 0) ? 1u : 0u;
                        const uint64_t da = tc::sdesc_sw128(a_s + 32 * k);
                        const uint64_t dbh = tc::sdesc_sw128(b_hi + 32 * k);
                        const uint64_t dbl = tc::sdesc_sw128(b_lo + 32 * k);
                        tc::mma_mxf8f6f4(acc0, da, dbh, idesc, sfc + 0, sfc + 8, acc_first);
                        tc::mma_mxf8f6f4(acc0, da, dbl, idesc, sfc + 0, sfc + 12, 1u);
                        if (C::NA == 2) {
                            const uint64_t da2 = tc::sdesc_sw128(a_s + A_BYTES + 32 * k);
                            tc::mma_mxf8f6f4(acc1, da2, dbh, idesc, sfc + 4, sfc + 8, acc_first);
                            tc::mma_mxf8f6f4(acc1, da2, dbl, idesc, sfc + 4, sfc + 12, 1u);
                        }
                    }
                    tc::mma_commit(&empty[s]);
                }
                __syncwarp();
                last_empty = &empty[s];
                last_parity = round & 1;
            }
            if (!ok) break;
            if (lane == 0) tc::mma_commit(&tfull[buf]);
            __syncwarp();
        }
        // the last stage release must land before the CTA can exit
        if (ok && last_empty && !tc::mbar_wait(last_empty, last_parity, LIMIT, abort_p)) {
            if (lane == 0) fail();
        }
    } else {
        // ------------------------------------------------ epilogue (warps 3..6)
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int lt = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++lt) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t)) {
                --lt;
                continue;
            }
            const int buf = lt & 1, use = lt >> 1;
            if (!tc::mbar_wait(&tfull[buf], use & 1, LIMIT, abort_p)) {
                if (lane == 0) fail();
                break;
            }
            tc::tc_fence_after();
            const uint32_t acc0 = tmem + lane_base + buf * C::ACC_STRIDE;
            const int row = t.m0 + q * 32 + lane;  // weight row this lane holds
            for (int c0 = 0; c0 < t.n; c0 += 16) {
                uint32_t ra[16], rb[16];
                tc::tmem_ld_32x32b_x16(acc0 + c0, ra);
                if (MODE == MOE_GEMM_GATEUP) tc::tmem_ld_32x32b_x16(acc0 + NTMAX + c0, rb);
                tc::tmem_ld_wait();
                if (MODE == MOE_GEMM_GATEUP) {
                    const int F = args.M;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j >= t.n) break;
                        const float g = __uint_as_float(ra[j]), u = __uint_as_float(rb[j]);
                        const float h = g / (1.f + expf(-g)) * u;
                        // two-term E4M3 split over the 32 rows of this warp (one MX block along F)
                        const int sh = mx8::scale_exp(warp_max(fabsf(h)));
                        const uint32_t hb = mx8::to_e4m3x2(h * mx8::exp2i(-sh), 0.f) & 0xFF;
                        const float back = mx8::from_e4m3x2(hb).x * mx8::exp2i(sh);
                        const float r = h - back;
                        const int sl = mx8::scale_exp(warp_max(fabsf(r)));
                        const uint32_t lb = mx8::to_e4m3x2(r * mx8::exp2i(-sl), 0.f) & 0xFF;
                        const size_t slot = (size_t)(t.s0 + c0 + j);
                        args.h_hi[slot * F + row] = (uint8_t)hb;
                        args.h_lo[slot * F + row] = (uint8_t)lb;
                        if (lane == 0) {
                            args.hs_hi[slot * (F / 32) + row / 32] = (uint8_t)(sh + 127);
                            args.hs_lo[slot * (F / 32) + row / 32] = (uint8_t)(sl + 127);
                        }
                    }
                } else {
                    int fl = 0;
                    float wv = 0.f;
                    if (lane < 16 && c0 + lane < t.n) {
                        fl = args.perm[t.s0 + c0 + lane];
                        if (fl < 0 || fl >= args.n_rows) {
                            moe_flag(args.status, MOE_ERR_BAD_INDEX);
                            fl = -1;
                        } else {
                            wv = args.topk_w[fl];
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int flj = __shfl_sync(0xFFFFFFFFu, fl, j);
                        const float wj = __shfl_sync(0xFFFFFFFFu, wv, j);
                        if (c0 + j >= t.n) break;
                        if (flj < 0) continue;
                        const int tok = flj / args.k;
                        atomicAdd(args.acc + (size_t)tok * args.Dout + row, wj * __uint_as_float(ra[j]));
                    }
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&tempty[buf]);
        }
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t moe_gemm_smem_bytes(int mode) {
    size_t stages = mode == MOE_GEMM_GATEUP ? Cfg<MOE_GEMM_GATEUP>::STAGES * (size_t)Cfg<MOE_GEMM_GATEUP>::STAGE_BYTES
                                            : Cfg<MOE_GEMM_DOWN>::STAGES * (size_t)Cfg<MOE_GEMM_DOWN>::STAGE_BYTES;
    return 1024 /*align*/ + stages + 16 * 8 /*barriers*/ + 16 /*tmem slot*/ +
           (MOE_MAX_EXPERTS + 1) * sizeof(int);
}

cudaError_t moe_launch_gemm(int mode, const CUtensorMap *mA, const CUtensorMap *mA2,
                            const CUtensorMap *mBhi, const CUtensorMap *mBlo,
                            const MoeGemmArgs *args, int grid, cudaStream_t st) {
    size_t sm = moe_gemm_smem_bytes(mode);
    cudaError_t err;
    if (mode == MOE_GEMM_GATEUP) {
        err = cudaFuncSetAttribute(moe_grouped_gemm_kernel<MOE_GEMM_GATEUP>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (err != cudaSuccess) return err;
        moe_grouped_gemm_kernel<MOE_GEMM_GATEUP><<<grid, NUM_THREADS, sm, st>>>(*mA, *mA2, *mBhi,
                                                                               *mBlo, *args);
    } else {
        err = cudaFuncSetAttribute(moe_grouped_gemm_kernel<MOE_GEMM_DOWN>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (err != cudaSuccess) return err;
        moe_grouped_gemm_kernel<MOE_GEMM_DOWN><<<grid, NUM_THREADS, sm, st>>>(*mA, *mA, *mBhi,
                                                                             *mBlo, *args);
    }
    return cudaGetLastError();
}
