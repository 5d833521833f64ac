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
//   warp 0      weight producer (one thread): weight tiles by TMA (packed
//               E2M1 expanded to the 8-bit MMA layout) and their prepared
//               512-byte scale atoms by bulk copy
//   warp 1      activation producer: rows of the token tile (slot order) by
//               2D TMA and their scale atoms by bulk copy; TMEM allocator
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

// Two rings: weights (+ their scale atoms) stream from HBM and get the deeper
// ring; activation terms (+ scales) come from L2.
template <int MODE>
struct Cfg {
    static constexpr int NA = (MODE == MOE_GEMM_GATEUP) ? 2 : 1;  // weight operands
    static constexpr int SA = (MODE == MOE_GEMM_GATEUP) ? 4 : 5;  // weight ring stages
    static constexpr int SB = (MODE == MOE_GEMM_GATEUP) ? 3 : 4;  // activation ring stages
    static constexpr int A_STAGE = (NA * (A_BYTES + SF_BYTES) + 1023) / 1024 * 1024;
    static constexpr int A_SF = NA * A_BYTES;                      // scale atoms within A stage
    static constexpr int B_STAGE = 2 * B_BYTES + 2 * SF_BYTES;
    static constexpr int B_BASE = SA * A_STAGE;
    static constexpr int B_SF = 2 * B_BYTES;
    static constexpr int BAR_BASE = B_BASE + SB * B_STAGE;
    static constexpr int N_BARS = 2 * SA + 2 * SB + 4;
    static constexpr int PREFIX_BASE = BAR_BASE + N_BARS * 8 + 16;
    static constexpr int EPI_BASE = PREFIX_BASE + (MOE_MAX_EXPERTS + 1) * 4 + 12;  // 16-B aligned
    static constexpr int EPI_BYTES = (MODE == MOE_GEMM_DOWN) ? 4 * 16 * 32 * 4 : 0;
    static constexpr int SMEM = 1024 + EPI_BASE + EPI_BYTES;
    static constexpr int ACC_STRIDE = NA * NTMAX;  // TMEM columns per accumulator buffer
    static_assert(B_STAGE % 1024 == 0, "activation stage must keep 1 KB alignment");
    static_assert(EPI_BASE % 16 == 0, "epilogue staging alignment");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Tile {
    int e;      // expert
    int m0;     // first weight row (within the expert)
    int mt;     // weight row tile index
    int s0;     // first slot of the tile (position in perm order)
    int n;      // valid token rows
    int nmma;   // n rounded up to 16 (MMA N)
    int tt;     // global token-tile index (activation / h scale atoms)
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
    t.mt = m;
    t.m0 = m * BM;
    t.s0 = sb + r0;
    t.n = r1 - r0;
    t.nmma = (t.n + 15) & ~15;
    t.tt = s_prefix[a] + j;
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
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *fullA = (uint64_t *)(smem + C::BAR_BASE);
    uint64_t *emptyA = fullA + C::SA;
    uint64_t *fullB = emptyA + C::SA;
    uint64_t *emptyB = fullB + C::SB;
    uint64_t *tfull = emptyB + C::SB;
    uint64_t *tempty = tfull + 2;
    uint32_t *tmem_slot = (uint32_t *)(tempty + 2);
    int *abort_flag = (int *)(tmem_slot + 1);
    int *s_prefix = (int *)(smem + C::PREFIX_BASE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = args.E;
    int n_active = args.active[0];
    if (n_active < 0 || n_active > E) n_active = 0;
    for (int i = tid; i <= n_active; i += NUM_THREADS) s_prefix[i] = args.tt_prefix[i];
    if (tid == 0) {
        *abort_flag = 0;
        for (int s = 0; s < C::SA; ++s) {
            tc::mbar_init(&fullA[s], 1);
            tc::mbar_init(&emptyA[s], 1);
        }
        for (int s = 0; s < C::SB; ++s) {
            tc::mbar_init(&fullB[s], 1);
            tc::mbar_init(&emptyB[s], 1);
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
    volatile int *abort_p = abort_flag;
    auto fail = [&](void) {
        *abort_p = 1;
        moe_flag(args.status, MOE_ERR_DEVICE_TIMEOUT);
    };

    if (warp == 0) {
        // ------------------------------------------ weight producer (one thread)
        if (lane == 0) {
            const uint64_t pol_w = tc::policy_evict_first();
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
                Tile t;
                if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E,
                             args.n_rows, t)) {
                    moe_flag(args.status, MOE_ERR_BAD_INDEX);
                    continue;
                }
                const size_t atom0 = ((size_t)t.e * MT + t.mt) * KC;
                for (int kc = 0; kc < KC; ++kc, ++it) {
                    const int s = it % C::SA, round = it / C::SA;
                    if (round > 0 && !tc::mbar_wait(&emptyA[s], (round - 1) & 1, LIMIT, abort_p)) {
                        fail();
                        ok = false;
                        break;
                    }
                    unsigned char *st = smem + s * C::A_STAGE;
                    tc::mbar_arrive_expect_tx(&fullA[s], (uint32_t)(C::NA * (A_TX + SF_BYTES)));
                    tc::tma_load_2d(st, &mapA, &fullA[s], kc * BK, t.e * args.M + t.m0, pol_w);
                    tc::bulk_copy_g2s(st + C::A_SF, args.a_atoms + (atom0 + kc) * SF_BYTES,
                                      SF_BYTES, &fullA[s], pol_w);
                    if (C::NA == 2) {
                        tc::tma_load_2d(st + A_BYTES, &mapA2, &fullA[s], kc * BK,
                                        t.e * args.M + t.m0, pol_w);
                        tc::bulk_copy_g2s(st + C::A_SF + SF_BYTES,
                                          args.a2_atoms + (atom0 + kc) * SF_BYTES, SF_BYTES,
                                          &fullA[s], pol_w);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------ activation producer (warp)
        const uint64_t pol_x = tc::policy_evict_last();
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t))
                continue;
            const uint32_t tx = (uint32_t)(2 * t.nmma * BK + 2 * SF_BYTES);
            const size_t atom0 = (size_t)t.tt * KC;
            for (int kc = 0; kc < KC; ++kc, ++it) {
                const int s = it % C::SB, round = it / C::SB;
                if (round > 0 && !tc::mbar_wait(&emptyB[s], (round - 1) & 1, LIMIT, abort_p)) {
                    if (lane == 0) fail();
                    ok = false;
                    break;
                }
                unsigned char *st = smem + C::B_BASE + s * C::B_STAGE;
                if (lane == 0) {
                    tc::mbar_arrive_expect_tx(&fullB[s], tx);
                    tc::bulk_copy_g2s(st + C::B_SF, args.b_atoms_hi + (atom0 + kc) * SF_BYTES,
                                      SF_BYTES, &fullB[s], pol_x);
                    tc::bulk_copy_g2s(st + C::B_SF + SF_BYTES,
                                      args.b_atoms_lo + (atom0 + kc) * SF_BYTES, SF_BYTES,
                                      &fullB[s], pol_x);
                }
                __syncwarp();
                if (lane < t.nmma / 16) {
                    tc::tma_load_2d(st + lane * 16 * BK, &mapBhi, &fullB[s], kc * BK,
                                    t.s0 + 16 * lane, pol_x);
                    tc::tma_load_2d(st + B_BYTES + lane * 16 * BK, &mapBlo, &fullB[s], kc * BK,
                                    t.s0 + 16 * lane, pol_x);
                }
            }
        }
    } else if (warp == 2) {
        // ------------------------------------------ MMA issuer
        int it = 0, lt = 0;
        bool ok = true;
        uint64_t *lastA = nullptr, *lastB = nullptr;
        uint32_t parA = 0, parB = 0;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t))
                continue;
            const int buf = lt & 1, use = lt >> 1;
            ++lt;
            if (use > 0 && !tc::mbar_wait(&tempty[buf], (use - 1) & 1, LIMIT, abort_p)) {
                if (lane == 0) fail();
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t acc0 = tmem + buf * C::ACC_STRIDE;
            const uint32_t acc1 = acc0 + NTMAX;  // GEMM1: up accumulator
            for (int kc = 0; kc < KC; ++kc, ++it) {
                const int sa = it % C::SA, ra = it / C::SA;
                const int sb = it % C::SB, rb = it / C::SB;
                if (!tc::mbar_wait(&fullA[sa], ra & 1, LIMIT, abort_p) ||
                    !tc::mbar_wait(&fullB[sb], rb & 1, LIMIT, abort_p)) {
                    if (lane == 0) fail();
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                if (lane == 0) {
                    unsigned char *sta = smem + sa * C::A_STAGE;
                    unsigned char *stb = smem + C::B_BASE + sb * C::B_STAGE;
                    const uint32_t sfc = tmem + SF_TMEM_COL + (uint32_t)(it & 1) * 16;
                    const uint32_t sfa = tc::smem_u32(sta + C::A_SF);
                    const uint32_t sfb = tc::smem_u32(stb + C::B_SF);
                    tc::tmem_cp_32x128b_warpx4(sfc + 0, tc::sdesc_plain_32x16(sfa));
                    if (C::NA == 2)
                        tc::tmem_cp_32x128b_warpx4(sfc + 4, tc::sdesc_plain_32x16(sfa + SF_BYTES));
                    tc::tmem_cp_32x128b_warpx4(sfc + 8, tc::sdesc_plain_32x16(sfb));
                    tc::tmem_cp_32x128b_warpx4(sfc + 12, tc::sdesc_plain_32x16(sfb + SF_BYTES));
                    const uint32_t a_s = tc::smem_u32(sta), b_hi = tc::smem_u32(stb),
                                   b_lo = tc::smem_u32(stb + B_BYTES);
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
                    tc::mma_commit(&emptyA[sa]);
                    tc::mma_commit(&emptyB[sb]);
                }
                __syncwarp();
                lastA = &emptyA[sa];
                parA = ra & 1;
                lastB = &emptyB[sb];
                parB = rb & 1;
            }
            if (!ok) break;
            if (lane == 0) tc::mma_commit(&tfull[buf]);
            __syncwarp();
        }
        // the last stage releases must land before the CTA can exit
        if (ok && lastA &&
            (!tc::mbar_wait(lastA, parA, LIMIT, abort_p) || !tc::mbar_wait(lastB, parB, LIMIT, abort_p))) {
            if (lane == 0) fail();
        }
    } else {
        // ------------------------------------------ epilogue (warps 3..6)
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        int lt = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            Tile t;
            if (!tile_at(tile, n_active, MT, s_prefix, args.active, args.offsets, E, args.n_rows, t))
                continue;
            const int buf = lt & 1, use = lt >> 1;
            ++lt;
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
                            // F chunk mt of GEMM2 = this weight tile; block q of the chunk
                            const size_t at = ((size_t)t.tt * MT + t.mt) * SF_BYTES +
                                              atom_off(c0 + j, q);
                            args.h_atoms_hi[at] = (uint8_t)(sh + 127);
                            args.h_atoms_lo[at] = (uint8_t)(sl + 127);
                        }
                    }
                } else {
                    // weighted values -> warp staging [16 columns][32 rows], then each
                    // lane adds 4 consecutive rows of one column with one vector reduction
                    float *stg = (float *)(smem + C::EPI_BASE) + (warp - 3) * 16 * 32;
                    int fl = -1;
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
                    for (int j = 0; j < 16; ++j)
                        stg[j * 32 + lane] = __shfl_sync(0xFFFFFFFFu, wv, j) * __uint_as_float(ra[j]);
                    __syncwarp();
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = lane + 32 * u;  // float4 index: column i/8, rows 4*(i%8)..+3
                        const int j = i >> 3, g = i & 7;
                        const int flj = __shfl_sync(0xFFFFFFFFu, fl, j);
                        if (c0 + j < t.n && flj >= 0) {
                            const float4 v = *(const float4 *)(stg + j * 32 + 4 * g);
                            float *dst = args.acc + (size_t)(flj / args.k) * args.Dout + t.m0 +
                                         q * 32 + 4 * g;
                            asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst),
                                         "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                                         : "memory");
                        }
                    }
                    __syncwarp();
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

// Weight scales re-laid as 512-byte tensor-core scale atoms: atom (e, mt, kc)
// holds rows mt*128 .. +127, 32-wide K blocks 4kc .. 4kc+3, byte (m%32)*16 +
// (m/32)*4 + c. One thread per 4-byte word.
__global__ void __launch_bounds__(256) moe_prepare_atoms_kernel(int64_t words, int M, int K,
                                                                const uint8_t *__restrict__ s,
                                                                uint32_t *__restrict__ out) {
    int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (w >= words) return;
    const int MT = M / BM, KC = K / BK, ksb = K / 32;
    int64_t atom = w / 128;
    int j = (int)(w % 128);
    int m = (j % 4) * 32 + j / 4;
    int kc = (int)(atom % KC);
    int64_t em = atom / KC;  // e * MT + mt
    int mt = (int)(em % MT);
    int64_t e = em / MT;
    const uint8_t *src = s + ((e * M + (int64_t)mt * BM + m) * ksb + kc * 4);
    out[w] = *(const uint32_t *)src;
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t moe_gemm_smem_bytes(int mode) {
    return mode == MOE_GEMM_GATEUP ? Cfg<MOE_GEMM_GATEUP>::SMEM : Cfg<MOE_GEMM_DOWN>::SMEM;
}

cudaError_t moe_launch_prepare_atoms(int E, int M, int K, const uint8_t *s, uint8_t *out,
                                     cudaStream_t st) {
    int64_t words = (int64_t)E * M * (K / 32) / 4;
    moe_prepare_atoms_kernel<<<(unsigned)((words + 255) / 256), 256, 0, st>>>(words, M, K, s,
                                                                             (uint32_t *)out);
    return cudaGetLastError();
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
