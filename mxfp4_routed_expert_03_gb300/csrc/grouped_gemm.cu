// Grouped block-scaled MXFP4 GEMMs on tcgen05 tensor cores (layer-major
// prefill). GEMM1 computes gate and up for 64 intermediate rows of one expert
// against up to 112 of that expert's routed tokens and applies SwiGLU in the
// epilogue; GEMM2 computes the down projection for 128 output rows and adds
// the routing-weighted result into each token's fp32 output row.
//
// The pages' prefill "groups all rows selecting each expert" and reads only
// the selected experts (Moonshine README, "How the engine works"; Moonshine
// GitHub README, "Prefill"); each selected expert's FFN runs on MXFP4 weights
// (MoonTail, "Routed expert FFN"; Moonshine GitHub README, "MXFP4 kernels"),
// and the weighted reduction closes the MoE tail (Moonshine README,
// "Run layer-major prefill").
//
// Tensor-core formulation (kind::mxf8f6f4, block scale 1X): D[128 x N] in
// TMEM accumulates A[128 x K] (weights, E2M1, one E8M0 scale per 32 K) times
// B[N x K]^T (activations, E4M3, one E8M0 scale per 32 K). On sm_103 a
// block-scaled MMA costs about the same up to N = 160 whatever N is, so the
// tiles are shaped for few, wide MMAs:
//   - the activations' two-term split (hi + lo, see mx8.cuh) is stacked
//     along N: B = [hi rows; lo rows], N = 2 * tokens, and the epilogue adds
//     the two halves of D;
//   - GEMM1 stacks 64 gate rows and the matching 64 up rows in one 128-row
//     A tile (two 64-row TMA boxes), so one MMA per 32-wide K step covers
//     gate and up; the epilogue pairs TMEM lanes r and 64 + r.
//
// Every CTA runs alone (no clusters): it fetches the whole activation chunk
// of its tile into its own shared memory and releases each stage with one
// local commit. The CTAs that work on one expert's token tile at the same
// time take adjacent weight tiles, so the activation chunk they all read is
// served from L2 after the first fetch.
//
// Two tile widths (template NT): the wide variant (112 token rows) for
// prefill, with 2-stage rings; the narrow variant (16 rows, chosen when no
// expert has more rows) with 5-stage rings and two MMA issuers. A pipeline
// stage carries two 128-wide K blocks; data
// layouts stay per K block. With expert streaming the weight producer
// addresses the expert's slot (args.w_index).
//
// One persistent CTA per SM, 7 warps (8 for the narrow variant):
//   warp 0      weight producer (one thread): weight tile(s) by TMA (packed
//               E2M1 expanded to the 8-bit MMA layout) and the prepared 1 KB
//               scale block holding the stage's K block(s)
//   warp 1      activation producer (one thread): the token tile's prepared
//               [hi; lo] B tile and its 1 KB scale block, each one contiguous
//               bulk copy per K block; TMEM allocator
//   warp 2      MMA issuer (one thread): tcgen05.cp scales, tcgen05.mma
//   warps 3-6   epilogue, one 32-lane TMEM quadrant each
//   warp 7      (narrow) second MMA issuer
// One "full" barrier per stage serves both operand rings (both producers
// arrive on it) and one "empty" barrier per stage releases it (one commit of
// the issuer that consumed it). The accumulator is double-buffered in TMEM so
// the epilogue of tile i overlaps the MMAs of tile i+1. Every wait is
// bounded: on expiry the CTA records MOE_ERR_DEVICE_TIMEOUT, each issuer
// drains its MMAs, and before the CTA leaves it waits (bounded) for every
// operand copy it issued to land, so nothing writes into shared memory the
// CTA no longer owns.
#include "common.cuh"
#include "kernels.h"
#include "mx8.cuh"
#include "tc_ptx.cuh"

namespace {

constexpr int BK = 128;                  // K elements per block (data-layout unit)
constexpr int ATOM_BLOCKS = 2;           // K blocks per prepared weight-scale block
constexpr int NTMAX = MOE_GEMM_NTMAX;    // token rows per tile (wide variant)
constexpr int A_BYTES = 128 * BK;        // smem bytes of the 128-row weight tile (E2M1 -> 8 bit)
constexpr int A_TX = 128 * BK / 2;       // bytes the TMA moves for it (packed)
constexpr int SF_BYTES = 1024;           // one prepared weight-scale block: 128 rows x 2 K blocks
constexpr int BSF_BYTES = 1024;          // activation scales of one chunk (256 B rows, 4 blocks)

// NT: token rows per tile. The wide variant (NT = NTMAX) serves prefill; the
// narrow one (NT = MOE_GEMM_NT_NARROW, when no expert has more than NT routed
// rows) spends the activation ring's shared memory on a deeper weight ring,
// since with few tokens per expert the GEMM streams weights and is bound by
// the weight bytes it keeps in flight. Scale blocks (1 KB per K block pair
// of weights, per K block of activations) land in shared memory once
// (narrow: read into tensor memory by 32x128b.warpx4 copies, which fill every
// lane quadrant) or once per lane quadrant (wide: one 128x256b copy reads
// all four, fewer instructions for the single issuer).
//
// FP4 selects the FP4 x FP4 mode (kind::mxf4): the activations are one MXFP4
// term (E2M1 with an E8M0 scale per 32) instead of two E4M3 terms, and both
// operands stay packed in shared memory, two elements per byte, so a stage's
// two K blocks are one 128-byte row per weight or token row and one MMA
// covers 64 K. A stage is half the bytes of the E4M3 path, so the rings are
// deeper.
template <int MODE, int NT, int AF>
struct Cfg {
    static constexpr bool FP4 = AF == MOE_AF_MXF4;
    static constexpr bool BF16 = AF == MOE_AF_BF16;
    static constexpr bool NARROW = NT <= 16;
    // MMA-issuing warps. One issuing thread spends about 75 cycles on each
    // tcgen05 instruction (MMA, scale copy, commit) whatever the MMA's N,
    // which is slower than the tensor pipe for the narrow tiles and for the
    // FP4 mode's one-term tiles; those variants therefore have two issuers,
    // each taking every other K stage of a tile into its own accumulator, and
    // the epilogue adds the two. (The two-term wide tiles' accumulators,
    // 2 x 112 columns, leave no tensor memory for a second pair.)
    // (Measured on the narrow tiles: a third issuer shortens the down GEMM,
    // whose pieces are short, by 7 %, and lengthens the gate/up GEMM, whose
    // epilogue then adds three accumulators, by 2 %.)
    static constexpr int NSPLIT = NARROW ? (MODE == MOE_GEMM_DOWN ? 3 : 2) : FP4 ? 2 : 1;
    static constexpr int THREADS = 224 + 32 * (NSPLIT - 1);  // warps 7, 8: further issuers
    static constexpr int TERMS = (FP4 || BF16) ? 1 : 2;  // activation terms stacked along N
    static constexpr uint32_t ACC_COLS = TERMS * NT;         // [hi | lo] columns of one accumulator
    static constexpr uint32_t BUF_COLS = NSPLIT * ACC_COLS;  // one of two accumulator buffers
    static constexpr uint32_t SF_TMEM_COL = 2 * BUF_COLS;    // then 2 scale slots per issuer
    // accumulators and scale slots, rounded up to a power of two
    static constexpr uint32_t TMEM_COLS = (NARROW && NSPLIT < 3) ? 256 : 512;
    // K blocks per pipeline stage: each wait, commit and loop step of an
    // issuer is shared by 8 MMAs (4 in the FP4 mode). (Single-block stages
    // with deeper rings measured slower for the wide variant: the issuer's
    // per-stage waits cost more than the extra depth returned.)
    static constexpr int KS = 2;
    // B scale columns per K block: 8 when B has more than 128 rows (two
    // 128-row halves), else 4
    static constexpr uint32_t BSF_COLS = TERMS * NT > 128 ? 8 : 4;
    static constexpr uint32_t SF_SLOT = KS * (4 + BSF_COLS);  // per stage: A 4 columns per block, then B
    // Copies of each scale block in smem: four let one 128x256b copy fill all
    // lane quadrants (weights: both K blocks of a stage at once), which costs
    // the wide variant's single issuer fewer operations. The narrow variant
    // is bound by shared-memory traffic (E2M1 tiles land expanded to 8 bits,
    // and every 128 x 32 MMA reads 4 KB of weights and 1 KB of tokens), so
    // it keeps one copy of each block and fills the lane quadrants with
    // 32x128b.warpx4 copies. The FP4 mode issues half the MMAs per stage and
    // spends the room of the extra copies on ring depth.
    static constexpr int SCALE_REP_A = BF16 ? 0 : (NARROW || FP4) ? 1 : 4;  // bf16: no scales
    static constexpr int SCALE_REP_B = BF16 ? 0 : (NARROW || FP4) ? 1 : 4;
    static_assert(SF_TMEM_COL + 2 * NSPLIT * SF_SLOT <= TMEM_COLS, "tensor memory budget");
    static constexpr int MROWS = (MODE == MOE_GEMM_GATEUP) ? 64 : 128;  // weight rows per tile
    // ring stages (KS blocks each)
    static constexpr int SA = NARROW ? (FP4 ? 10 : 5) : (FP4 ? 6 : BF16 ? 3 : 2);
    static constexpr int SB = SA;              // activation ring stages
    // one full barrier per stage for both operands (both producers arrive)
    // and one release barrier per stage (one commit)
    static constexpr bool MERGED = SA == SB;
    static_assert(MERGED, "the rings share their barriers");
    // weight tile of a stage in shared memory: FP4 packed 128-byte rows, else
    // one 128 x 128-byte tile per K block (E2M1 expanded to 8-bit containers,
    // or 64 bf16 per row)
    static constexpr int A_TILE = FP4 ? 128 * 128 : KS * A_BYTES;
    static constexpr int A_STAGE = A_TILE + SCALE_REP_A * SF_BYTES;  // tiles, then scales
    static constexpr int A_SF = A_TILE;
    // smem bytes of one K block's activation rows: [hi; lo] E4M3, or bf16
    static constexpr int B_BYTES = (BF16 ? 1 : 2) * NT * 128;
    // activation tile of a stage: FP4 one 128-byte row per token, else [hi; lo]
    // rows per K block
    static constexpr int B_TILE = FP4 ? NT * 128 : KS * B_BYTES;
    static constexpr int B_STAGE = B_TILE + KS * SCALE_REP_B * BSF_BYTES;  // tiles, then scales
    static constexpr int B_BASE = SA * A_STAGE;
    static constexpr int B_SF = B_TILE;
    static constexpr int BAR_BASE = B_BASE + SB * B_STAGE;
    static constexpr int N_FULL = SA;
    static constexpr int N_EMPTY = SA;
    // full(s), empty(s); tfull, tempty x2; one drain barrier per issuer
    static constexpr int N_BARS = N_FULL + N_EMPTY + 4 + NSPLIT;
    // after the barriers: TMEM address, abort flag, fills issued by each
    // producer, the epilogue's last-part flag
    // Tile lookup. Wide: shared-memory copies of the token-tile prefix, the
    // active experts and their row segments (NTAB entries). Narrow: every
    // expert has one token tile, so tile ct is active expert ct / MT; the
    // CTA's own tiles are decoded once into a list of TLIST entries (direct
    // loads from the plan past that), which frees the room for a 5th stage.
    static constexpr int NTAB = NARROW ? 0 : MOE_MAX_EXPERTS;
    static constexpr int TLIST = NARROW ? 256 : 0;
    static constexpr int PREFIX_BASE = (BAR_BASE + N_BARS * 8 + 20 + 15) / 16 * 16;  // int [active + 1]
    static constexpr int EXPERT_BASE = (PREFIX_BASE + (NTAB ? (NTAB + 1) * 4 : 0) + 15) / 16 * 16;
    static constexpr int SEG_BASE = (EXPERT_BASE + NTAB * 4 + 15) / 16 * 16;  // int2
    static constexpr int LIST_BASE = (SEG_BASE + NTAB * 8 + 15) / 16 * 16;   // int2 [TLIST]
    static constexpr int EPI_BASE = (LIST_BASE + TLIST * 8 + 15) / 16 * 16;
    // GEMM1: u values of 16 columns x 64 rows; GEMM2: 4 warps x 16 columns x 32 rows
    static constexpr int EPI_BYTES = (MODE == MOE_GEMM_GATEUP) ? 16 * 64 * 4 : 4 * 16 * 32 * 4;
    static constexpr int SMEM = 1024 + EPI_BASE + EPI_BYTES;
    static_assert(A_STAGE % 1024 == 0 && B_STAGE % 1024 == 0, "stages must keep 1 KB alignment");
    static_assert(NARROW || FP4 || BF16 || SCALE_REP_B == 4,
                  "wide two-term tiles need B scale columns 0..7");
    static_assert(TERMS * NT <= 128 || SCALE_REP_B == 4, "B rows past 127 need the 128x256b copy");
    static_assert(BAR_BASE % 8 == 0 && PREFIX_BASE % 16 == 0 && EXPERT_BASE % 16 == 0 &&
                      SEG_BASE % 16 == 0 && EPI_BASE % 16 == 0,
                  "shared-memory regions must be 16-byte aligned (int2 / float4 accesses)");
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct Seg {
    int tile;    // tile index in the schedule
    int s0, s1;  // its pipeline stages [s0, s1) (K blocks KS s0 .. KS s1 - 1)
};

struct Tile {
    int e;      // expert
    int mt;     // weight row tile index (rows mt * MROWS ..)
    int s0;     // first slot of the tile (position in perm order)
    int n;      // valid token rows
    int nmma;   // n rounded up to 16; the MMA's N is 2 * nmma
    int tt;     // global token-tile index (activation / h scale atoms)
};

// Tile `ct` of the schedule: active expert a owns MT * ntt(a) consecutive
// tiles. Normally the token tile varies fastest: the CTAs working on one
// weight tile run side by side and share it through L2, and so do the
// activations of the expert's few token tiles. In the gate/up GEMM an expert
// with more tiles than a wave of the grid (MT * ntt > G CTAs: a popular
// expert of a skewed batch, dozens of token tiles) takes its weight tiles
// fastest instead: the CTAs of one token tile share its activation rows (1.6
// MB at d_model 7168, two terms) while they are in L2, which token-tile-
// fastest order re-read from DRAM for every pair of weight tiles (skewed
// prefill, T = 8192: 17.3 -> 13.3 GB per launch). The down GEMM keeps the
// token tile fastest: there the expert's weights dominate what a token tile
// would re-read. s_prefix, s_expert and s_seg are the shared-memory copies of
// the token-tile prefix, the active experts and their (first slot, rows)
// segments. Each role visits its tiles in increasing order, so `a` (the
// caller's cursor, starting at 0) only moves forward: a few shared-memory
// reads per tile.
template <int NT, bool WM>
__device__ __forceinline__ bool tile_at(int ct, int n_active, int MT, const int *s_prefix,
                                        const int *s_expert, const int2 *s_seg, int &a, Tile &t) {
    while (a + 1 < n_active && MT * s_prefix[a + 1] <= ct) ++a;  // last a with MT*prefix[a] <= ct
    const int ntt = s_prefix[a + 1] - s_prefix[a];
    if (ntt <= 0 || s_expert[a] < 0) return false;
    const int local = ct - MT * s_prefix[a];
    const bool wide_expert = WM && (long long)MT * ntt > (long long)gridDim.x;
    const int mg = wide_expert ? local % MT : local / ntt;
    const int j = wide_expert ? local / MT : local % ntt;
    const int2 seg = s_seg[a];
    // token rows of the expert split evenly over its ntt tiles (32-bit
    // arithmetic unless the product is too large for it)
    const long long p0 = (long long)j * seg.y, p1 = p0 + seg.y;
    const int r0 = p1 <= 0x7FFFFFFFLL ? (int)p0 / ntt : (int)(p0 / ntt);
    const int r1 = p1 <= 0x7FFFFFFFLL ? (int)p1 / ntt : (int)(p1 / ntt);
    t.e = s_expert[a];
    t.mt = mg;
    t.s0 = seg.x + r0;
    t.n = r1 - r0;
    t.nmma = (t.n + 15) & ~15;
    t.tt = s_prefix[a] + j;
    return t.n > 0 && t.n <= NT;
}

// Narrow tiles: tile ct of this CTA from the CTA's tile list (its tiles
// t_first, t_first + 1, ...: x = expert | rows << 22, y = first slot; x < 0
// when invalid) or, past the list, straight from the plan. Active expert
// a = ct / MT owns tiles a * MT .. a * MT + MT - 1, one per weight tile.
template <int NT, int TLIST>
__device__ __forceinline__ bool tile_at_list(int ct, int MT, const int2 *s_list, int t_first,
                                             const MoeGemmArgs &args, Tile &t) {
    const int a = ct / MT, mg = ct - a * MT;
    const int i = ct - t_first;
    int e, sb, cnt;
    if (i >= 0 && i < TLIST) {
        const int2 v = s_list[i];
        if (v.x < 0) return false;
        e = v.x & 0x3FFFFF;
        cnt = v.x >> 22;
        sb = v.y;
    } else {
        e = args.active[1 + a];
        if (e < 0 || e >= args.E) return false;
        sb = args.offsets[e];
        cnt = args.offsets[e + 1] - sb;
        if (sb < 0 || sb + cnt > args.n_rows) return false;
    }
    t.e = e;
    t.mt = mg;
    t.s0 = sb;
    t.n = cnt;
    t.nmma = (cnt + 15) & ~15;
    t.tt = a;
    return cnt > 0 && cnt <= NT;
}

// Position of (B row n < 256, 32-wide K block c) inside the 1 KB activation
// scale block of one chunk: 32 lanes x 8 columns, lane n % 32 column n / 32,
// stored as the K-major core matrices (8 rows x 16 bytes) that
// tcgen05.cp.128x256b reads: [lane / 8][column / 4][lane % 8][16 bytes].
__device__ __forceinline__ int bsf_off(int n, int c) {
    const int i = n & 31, j = n >> 5;
    return (i >> 3) * 256 + (j >> 2) * 128 + (i & 7) * 16 + (j & 3) * 4 + c;
}

// Stream-K split: the CTA whose stage range [U b / G, U (b + 1) / G) holds
// stage u (the largest b with floor(U b / G) <= u).
__device__ __forceinline__ int cta_of(long long U, long long u) {
    return (int)(((u + 1) * gridDim.x + U - 1) / U - 1);
}

// The four epilogue warps (128 threads) meet at named barrier 1.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

}  // namespace

template <int MODE, int NT, int AF>
__global__ void __launch_bounds__(Cfg<MODE, NT, AF>::THREADS, 1) moe_grouped_gemm_kernel(
    const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapA2,
    const MoeGemmArgs args) {
    using C = Cfg<MODE, NT, AF>;
    constexpr bool FP4 = C::FP4, BF16 = C::BF16;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem =
        (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint64_t *full = (uint64_t *)(smem + C::BAR_BASE);  // both operands of stage s landed
    uint64_t *empty = full + C::N_FULL;                  // stage s consumed
    uint64_t *tfull = empty + C::N_EMPTY;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;  // per issuer: its MMAs in flight, waited on when giving up
    uint32_t *tmem_slot = (uint32_t *)(drain + C::NSPLIT);
    int *abort_flag = (int *)(tmem_slot + 1);
    int *s_issued = abort_flag + 1;  // stages filled by the weight [0] / activation [1] producer
    volatile int *sk_last = s_issued + 2;  // epilogue: this CTA holds a split tile's last part
    int *s_prefix = (int *)(smem + C::PREFIX_BASE);
    int *s_expert = (int *)(smem + C::EXPERT_BASE);
    int2 *s_seg = (int2 *)(smem + C::SEG_BASE);
    int2 *s_list = (int2 *)(smem + C::LIST_BASE);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = args.E;
    int n_active = args.active[0];
    if (n_active < 0 || n_active > E) n_active = 0;
    // The CTA's work. Wide: whole tiles ct = blockIdx.x + i * gridDim.x.
    // Narrow (stream-K): the stages of all tiles in order form one sequence,
    // and CTA b takes the contiguous range [U b / G, U (b + 1) / G) of it, so
    // every CTA streams the same weight bytes whatever the tile count. A
    // tile split between CTAs is finished by the last part to arrive: gate/up
    // parts meet in global memory (args.sk_part), down parts each add their
    // own share to the output rows.
    const int NST = (args.KC + C::KS - 1) / C::KS;  // stages per tile
    const long long U = C::NARROW ? (long long)n_active * args.MT * NST : 0;
    const long long u_begin = U * blockIdx.x / gridDim.x;
    const long long u_end = U * (blockIdx.x + 1) / gridDim.x;
    const int t_first = C::NARROW ? (int)(u_begin / NST) : 0;  // this CTA's first tile
    if (C::NARROW) {  // this CTA's tiles: t_first, t_first + 1, .. (tile of stage u_end - 1)
        const long long n_tiles = u_end > u_begin ? (u_end - 1) / NST + 1 : 0;
        for (int i = tid; i < C::TLIST; i += C::THREADS) {
            const long long ct = (long long)t_first + i;
            int2 v = make_int2(-1, 0);
            if (ct < n_tiles) {
                const int a = (int)(ct / args.MT);
                const int e = args.active[1 + a];
                if (e >= 0 && e < E) {
                    const int sb = args.offsets[e], cnt = args.offsets[e + 1] - sb;
                    if (sb >= 0 && cnt > 0 && cnt <= NT && sb + cnt <= args.n_rows)
                        v = make_int2(e | (cnt << 22), sb);
                }
                if (v.x < 0) moe_flag(args.status, MOE_ERR_BAD_INDEX);
            }
            s_list[i] = v;
        }
    }
    for (int i = tid; C::NTAB && i <= n_active; i += C::THREADS) s_prefix[i] = args.tt_prefix[i];
    for (int a = tid; C::NTAB && a < n_active; a += C::THREADS) {
        const int e = args.active[1 + a];
        int sb = 0, cnt = 0;
        if (e >= 0 && e < E) {
            sb = args.offsets[e];
            cnt = args.offsets[e + 1] - sb;
        }
        const bool ok = e >= 0 && e < E && sb >= 0 && cnt > 0 && sb + cnt <= args.n_rows;
        if (!ok) moe_flag(args.status, MOE_ERR_BAD_INDEX);
        s_expert[a] = ok ? e : -1;
        s_seg[a] = make_int2(sb, ok ? cnt : 0);
    }
    if (tid == 0) {
        *abort_flag = 0;
        s_issued[0] = s_issued[1] = 0;
        for (int s = 0; s < C::SA; ++s) {
            tc::mbar_init(&full[s], 2);  // both producers arrive
            tc::mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < C::NSPLIT; ++i) tc::mbar_init(&drain[i], 1);
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], C::NSPLIT);  // every issuer commits its share
            tc::mbar_init(&tempty[b], 4);
        }
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    // Launched with programmatic dependent launch: everything so far read the
    // plan only, which is complete (it is two launches back); the next kernel
    // may start on SMs this grid leaves, and only the activation producer
    // waits below for the previous kernel's output.
    grid_dep_launch();
    const uint32_t tmem = *tmem_slot;
    const int MT = args.MT, KC = args.KC;
    const int total_tiles =
        n_active <= 0 ? 0 : (C::NARROW ? n_active * MT : s_prefix[n_active] * MT);
    auto get_tile = [&](int ct, int &cur, Tile &t) -> bool {
        if constexpr (C::NARROW)
            return tile_at_list<NT, C::TLIST>(ct, MT, s_list, t_first, args, t);
        else
            return tile_at<NT, MODE == MOE_GEMM_GATEUP>(ct, n_active, MT, s_prefix, s_expert, s_seg,
                                                        cur, t);
    };
    // Next piece of this CTA's work: tile sg.tile, stages [sg.s0, sg.s1) of
    // it (all of them unless a narrow tile is split between CTAs). Every role
    // walks the same sequence; `u` starts at seg_start. A narrow CTA's range
    // is at most a partial first tile, whole tiles and a partial last tile;
    // it takes the partial pieces first, so that joining a split tile's
    // parts (a few round trips to L2) overlaps the whole tiles' streaming
    // instead of adding to the end of the launch.
    const int f_tile = (int)(u_begin / NST), l_tile = (int)((u_end - 1) / NST);
    const int f_s0 = (int)(u_begin - (long long)f_tile * NST);
    const int l_s1 = (int)(u_end - (long long)l_tile * NST);
    const int f_s1 = l_tile == f_tile ? l_s1 : NST;
    const bool f_part = u_end > u_begin && (f_s0 != 0 || f_s1 != NST);
    const bool l_part = u_end > u_begin && l_tile != f_tile && l_s1 != NST;
    const int w_first = f_part ? f_tile + 1 : f_tile;  // whole tiles w_first .. w_last
    const int w_last = u_end > u_begin ? (l_part ? l_tile - 1 : l_tile) : -1;
    const long long seg_start = C::NARROW ? 0 : (long long)blockIdx.x;
    auto seg_next = [&](long long &u, Seg &sg) -> bool {
        if constexpr (C::NARROW) {
            int i = (int)u++;  // position in this CTA's order
            if (f_part && i-- == 0) {
                sg.tile = f_tile; sg.s0 = f_s0; sg.s1 = f_s1;
                return true;
            }
            if (l_part && i-- == 0) {
                sg.tile = l_tile; sg.s0 = 0; sg.s1 = l_s1;
                return true;
            }
            if (w_first + i > w_last) return false;
            sg.tile = w_first + i;
            sg.s0 = 0;
            sg.s1 = NST;
        } else {
            if (u >= total_tiles) return false;
            sg.tile = (int)u;
            sg.s0 = 0;
            sg.s1 = NST;
            u += gridDim.x;
        }
        return true;
    };
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
            int cur = 0;
            long long u = seg_start;
            Seg sg;
            while (ok && seg_next(u, sg)) {
                Tile t;
                if (!get_tile(sg.tile, cur, t)) {
                    moe_flag(args.status, MOE_ERR_BAD_INDEX);
                    continue;
                }
                int we = t.e;  // weight slot of the expert
                if (args.w_index) {
                    we = args.w_index[t.e];
                    if (we < 0 || we >= args.n_wexp) {  // not resident: flag, stay in bounds
                        moe_flag(args.status, MOE_ERR_BAD_INDEX);
                        we = 0;
                    }
                }
                const int row0 = we * args.M + t.mt * C::MROWS;
                const size_t atom0 = ((size_t)we * MT + t.mt) * ((KC + ATOM_BLOCKS - 1) / ATOM_BLOCKS);
                const int kend = min(KC, sg.s1 * C::KS);
                for (int kc = sg.s0 * C::KS; kc < kend; kc += C::KS) {
                    const int s = it % C::SA, round = it / C::SA;
                    const int nsub = min(C::KS, KC - kc);
                    if (round > 0 && !tc::mbar_wait(&empty[s], (round - 1) & 1, LIMIT, abort_p)) {
                        fail();
                        ok = false;
                        break;
                    }
                    unsigned char *st = smem + s * C::A_STAGE;
                    if constexpr (FP4) {
                        // one packed 128-byte row per weight row holds the stage's two
                        // K blocks (a lone last block: the box's second half reads past
                        // the row end, which the TMA fills with zeros)
                        tc::mbar_arrive_expect_tx(&full[s],
                                                  (uint32_t)(C::A_TILE + C::SCALE_REP_A * SF_BYTES));
                        ++it;  // a fill of this stage is now in flight
                        tc::tma_load_2d(st, &mapA, &full[s], kc * (BK / 2), row0, pol_w);
                        if (MODE == MOE_GEMM_GATEUP)  // up rows fill lanes 64..127
                            tc::tma_load_2d(st + 64 * 128, &mapA2, &full[s], kc * (BK / 2), row0,
                                            pol_w);
                    } else if constexpr (BF16) {
                        // one 128 x 64 bf16 tile (128-byte rows) per K block
                        tc::mbar_arrive_expect_tx(&full[s], (uint32_t)(nsub * A_BYTES));
                        ++it;  // a fill of this stage is now in flight
                        for (int sub = 0; sub < nsub; ++sub) {
                            unsigned char *sa = st + sub * A_BYTES;
                            tc::tma_load_2d(sa, &mapA, &full[s], (kc + sub) * 64, row0, pol_w);
                            if (MODE == MOE_GEMM_GATEUP)  // up rows fill lanes 64..127
                                tc::tma_load_2d(sa + 64 * 128, &mapA2, &full[s], (kc + sub) * 64,
                                                row0, pol_w);
                        }
                    } else {
                        tc::mbar_arrive_expect_tx(
                            &full[s], (uint32_t)(nsub * A_TX + C::SCALE_REP_A * SF_BYTES));
                        ++it;  // a fill of this stage is now in flight
                        for (int sub = 0; sub < nsub; ++sub) {
                            unsigned char *sa = st + sub * A_BYTES;
                            tc::tma_load_2d(sa, &mapA, &full[s], (kc + sub) * BK, row0, pol_w);
                            if (MODE == MOE_GEMM_GATEUP)  // up rows fill lanes 64..127
                                tc::tma_load_2d(sa + 64 * BK, &mapA2, &full[s], (kc + sub) * BK,
                                                row0, pol_w);
                        }
                    }
                    // the scale block holding this stage's K block(s)
                    const uint8_t *sf = args.a_atoms + (atom0 + kc / ATOM_BLOCKS) * SF_BYTES;
                    for (int qd = 0; qd < C::SCALE_REP_A; ++qd)
                        tc::bulk_copy_g2s(st + C::A_SF + qd * SF_BYTES, sf, SF_BYTES, &full[s], pol_w);
                }
            }
            s_issued[0] = it;
        }
    } else if (warp == 1) {
        // ------------------------------------------ activation producer (one thread)
        if (lane == 0) {
            grid_dep_wait();  // the activation (or h) tiles come from the previous kernel
            const uint64_t pol_x = tc::policy_evict_last();
            int it = 0;
            bool ok = true;
            int cur = 0;
            long long u = seg_start;
            Seg sg;
            while (ok && seg_next(u, sg)) {
                Tile t;
                if (!get_tile(sg.tile, cur, t)) continue;
                // [hi; lo] rows per K block, or (FP4) one packed row per token per stage
                const uint32_t tile_bytes =
                    (uint32_t)((FP4 || BF16) ? t.nmma * 128 : 2 * t.nmma * BK);
                const size_t blk0 = (size_t)t.tt * KC;
                const size_t chunk0 = (size_t)t.tt * ((KC + 1) / 2);  // FP4: 256-wide K chunks
                const int kend = min(KC, sg.s1 * C::KS);
                for (int kc = sg.s0 * C::KS; kc < kend; kc += C::KS) {
                    const int s = it % C::SB, round = it / C::SB;
                    const int nsub = min(C::KS, KC - kc);
                    if (round > 0 && !tc::mbar_wait(&empty[s], (round - 1) & 1, LIMIT, abort_p)) {
                        fail();
                        ok = false;
                        break;
                    }
                    unsigned char *st = smem + C::B_BASE + s * C::B_STAGE;
                    if constexpr (FP4) {
                        tc::mbar_arrive_expect_tx(
                            &full[s], tile_bytes + (uint32_t)nsub * C::SCALE_REP_B * BSF_BYTES);
                        tc::bulk_copy_g2s(st, args.b_tiles + (chunk0 + kc / 2) * MOE_GEMM_BTILE,
                                          tile_bytes, &full[s], pol_x);
                    } else {
                        tc::mbar_arrive_expect_tx(
                            &full[s], (uint32_t)nsub * (tile_bytes + C::SCALE_REP_B * BSF_BYTES));
                    }
                    ++it;
                    for (int sub = 0; sub < nsub; ++sub) {
                        const size_t blk = blk0 + kc + sub;
                        if (!FP4)
                            tc::bulk_copy_g2s(st + sub * C::B_BYTES, args.b_tiles + blk * MOE_GEMM_BTILE,
                                              tile_bytes, &full[s], pol_x);
                        const uint8_t *ss = args.b_atoms + blk * BSF_BYTES;
                        for (int qd = 0; qd < C::SCALE_REP_B; ++qd)
                            tc::bulk_copy_g2s(st + C::B_SF + (sub * C::SCALE_REP_B + qd) * BSF_BYTES,
                                              ss, BSF_BYTES, &full[s], pol_x);
                    }
                }
            }
            s_issued[1] = it;
        }
    } else if (warp == 2 || warp >= 7) {
        // ------------------------------------------ MMA issuer(s), one warp each
        // The whole warp walks the issue loop: the waits, shared-memory
        // addresses and descriptors are the same in every lane, so they stay
        // in the warp-uniform registers the tcgen05 instructions read, and
        // lane 0 issues the instructions. (Run by lane 0 alone, the loop moved
        // every operand into uniform registers anew for each instruction,
        // about 80 cycles apiece, and a stage issues 9 to 13 of them.) With
        // NSPLIT issuers, issuer `split` takes the piece's stages j with
        // j % NSPLIT == split into accumulator `split` of the buffer.
        const int split = warp == 2 ? 0 : warp - 6;
        const bool leader = lane == 0;
        // a wait in every lane, decided for the warp: it fails if any lane's ran out
        auto wait_all = [&](uint64_t *bar, uint32_t parity) -> bool {
            return __all_sync(0xFFFFFFFFu, tc::mbar_wait(bar, parity, LIMIT, abort_p));
        };
        int it = 0, lt = 0, mine = 0;
        bool ok = true;
        uint64_t *last = nullptr;
        uint32_t last_par = 0;
        int cur = 0;
        // Test hook (off unless the host asks for it): the first issuer waits
        // on its drain barrier, which nothing signals before the wind-down, so
        // the wait runs out and the CTA takes the timeout path below with
        // operand copies in flight.
        if (args.inject == MOE_INJECT_GEMM_STALL && split == 0 && !wait_all(&drain[0], 0)) {
            if (leader) fail();
            ok = false;
        }
        long long u = seg_start;
        Seg sg;
        while (ok && seg_next(u, sg)) {
            Tile t;
            if (!get_tile(sg.tile, cur, t)) continue;
            const int buf = lt & 1, use = lt >> 1;
            ++lt;
            if (use > 0 && !wait_all(&tempty[buf], (use - 1) & 1)) {
                if (leader) fail();
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t acc = tmem + buf * C::BUF_COLS + split * C::ACC_COLS;
            // E4M3 path: scale byte k of each column for K step k (32 wide);
            // FP4: scale bytes 2 k2, 2 k2 + 1 for K step k2 (64 wide)
            uint32_t idesc[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                idesc[k] = BF16 ? tc::idesc_bf16(128, t.nmma)
                           : FP4 ? tc::idesc_mxf4(128, t.nmma, 2 * (k & 1), 2 * (k & 1))
                                 : tc::idesc_mxf8f6f4(tc::FMT_E2M1, tc::FMT_E4M3, 128,
                                                      2 * t.nmma, k, k);
            bool first = true;
            const int kend = min(KC, sg.s1 * C::KS);
            for (int kc = sg.s0 * C::KS, j = 0; kc < kend; kc += C::KS, ++it, ++j) {
                if (C::NSPLIT > 1 && j % C::NSPLIT != split) continue;  // another issuer's stage
                const int s = it % C::SA, round = it / C::SA;
                const int nsub = min(C::KS, KC - kc);
                // With two issuers the slot's previous fill may have been the
                // other issuer's, still in flight: a parity wait on full[s]
                // could then match the phase before it. The slot's release of
                // round - 1 comes after that fill landed and before the
                // producers refill it, so once it is seen the full wait can only
                // mean this round (and it costs nothing: the fill of this round
                // waits for that release anyway).
                if (C::NSPLIT > 1 && round > 0 && !wait_all(&empty[s], (round - 1) & 1)) {
                    if (leader) fail();
                    ok = false;
                    break;
                }
                if (!wait_all(&full[s], round & 1)) {
                    if (leader) fail();
                    ok = false;
                    break;
                }
                const uint32_t a_s = tc::smem_u32(smem + s * C::A_STAGE);
                const uint32_t b_s = tc::smem_u32(smem + C::B_BASE + s * C::B_STAGE);
                const uint32_t slot =
                    tmem + C::SF_TMEM_COL + (uint32_t)(2 * split + (mine & 1)) * C::SF_SLOT;
                ++mine;
                // descriptors of the stage (offsets in 16-byte units are added
                // to the start-address field, which cannot carry over: shared
                // memory addresses stay below 256 KB)
                const uint64_t ad = tc::sdesc_sw128(a_s), bd = tc::sdesc_sw128(b_s);
                const uint64_t asf4 = tc::sdesc_plain_128x32(a_s + C::A_SF);
                uint64_t asf1[C::KS], bsf[C::KS];
#pragma unroll
                for (int sub = 0; sub < C::KS; ++sub) {
                    asf1[sub] = tc::sdesc_plain_32x16_groups256(a_s + C::A_SF + 128 * ((kc + sub) & 1));
                    const uint32_t b_sf = b_s + C::B_SF + sub * C::SCALE_REP_B * BSF_BYTES;
                    bsf[sub] = C::SCALE_REP_B == 4 ? tc::sdesc_plain_128x32(b_sf)
                                                   : tc::sdesc_plain_32x16_groups256(b_sf);
                }
                if (leader) {
                    if (C::SCALE_REP_A == 4)  // both blocks' weight scales: columns slot .. slot + 7
                        tc::tmem_cp_128x256b(slot, asf4);
#pragma unroll
                    for (int sub = 0; sub < C::KS; ++sub) {
                        if (sub >= nsub) break;
                        const uint32_t sfa = slot + 4 * sub, sfb = slot + 4 * C::KS + C::BSF_COLS * sub;
                        if (C::SCALE_REP_A == 1)  // K block kc + sub: its half of the scale block
                            tc::tmem_cp_32x128b_warpx4(sfa, asf1[sub]);
                        if (C::SCALE_REP_B == 4)
                            tc::tmem_cp_128x256b(sfb, bsf[sub]);
                        else if (C::SCALE_REP_B == 1)  // B rows 0..127 (columns 0..3)
                            tc::tmem_cp_32x128b_warpx4(sfb, bsf[sub]);
                        if constexpr (BF16) {
                            // K block sub: 64 bf16 per row, four MMAs of 16 K each
                            const uint64_t as = ad + (uint64_t)((sub * A_BYTES) >> 4);
                            const uint64_t bs = bd + (uint64_t)((sub * C::B_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc::mma_bf16(acc, as + 2 * k, bs + 2 * k, idesc[0],
                                             (!first || sub > 0 || k > 0) ? 1u : 0u);
                        } else if constexpr (FP4) {
                            // K block sub is bytes 64 sub .. 64 sub + 63 of every packed
                            // row; two MMAs of 64 K each
#pragma unroll
                            for (int k2 = 0; k2 < 2; ++k2)
                                tc::mma_mxf4(acc, ad + 4 * sub + 2 * k2, bd + 4 * sub + 2 * k2,
                                             idesc[k2], sfa, sfb,
                                             (!first || sub > 0 || k2 > 0) ? 1u : 0u);
                        } else {
                            const uint64_t as = ad + (uint64_t)((sub * A_BYTES) >> 4);
                            const uint64_t bs = bd + (uint64_t)((sub * C::B_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                tc::mma_mxf8f6f4(acc, as + 2 * k, bs + 2 * k, idesc[k], sfa, sfb,
                                                 (!first || sub > 0 || k > 0) ? 1u : 0u);
                        }
                    }
                    tc::mma_commit(&empty[s]);  // the stage is free once these MMAs are done
                }
                first = false;
                last = &empty[s];
                last_par = round & 1;
            }
            if (!ok) break;
            if (leader) tc::mma_commit(&tfull[buf]);
            __syncwarp();
        }
        // the last stage release must land before the CTA can exit
        if (ok && last && !wait_all(last, last_par) && leader) fail();
        // giving up: this warp's MMAs must finish before tensor memory is
        // freed (their operands are in shared memory, so they do)
        if (leader && (!ok || *abort_p)) tc::drain_mmas(&drain[split], LIMIT);
        __syncwarp();
    } else {
        // ------------------------------------------ epilogue (warps 3..6)
        // (warp 7, when present, is the second MMA issuer above)
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const uint64_t pol_acc = tc::policy_evict_last();
        int lt = 0, cur = 0;
        long long u = seg_start;
        Seg sg;
        while (seg_next(u, sg)) {
            Tile t;
            if (!get_tile(sg.tile, cur, t))
                continue;
            const int buf = lt & 1, use = lt >> 1;
            ++lt;
            // GEMM2: the tile's token rows and routing weights, read before the
            // accumulator is ready (column lane + 32 i of the tile in pf[i], pw[i])
            int pf[NT / 32 + 1];
            float pw[NT / 32 + 1];
            if (MODE == MOE_GEMM_DOWN && !args.y) {
#pragma unroll
                for (int i = 0; i <= NT / 32; ++i) {
                    const int col = lane + 32 * i;
                    pf[i] = -1;
                    pw[i] = 0.f;
                    if (col < t.n) {
                        const int fl = args.perm[t.s0 + col];
                        if (fl < 0 || fl >= args.n_rows) {
                            moe_flag(args.status, MOE_ERR_BAD_INDEX);
                        } else {
                            pf[i] = fl;
                            pw[i] = args.topk_w[fl];
                        }
                    }
                }
            }
            // a long wait (the tile's MMAs): sleep in try_wait rather than
            // spin, leaving issue slots to the producer and issuer warps. The
            // four warps then decide together, so none of them is left at a
            // later epilogue barrier by a warp that gave up.
            const bool got = tc::mbar_wait_sleep(&tfull[buf], use & 1, LIMIT, abort_p);
            if (!tc::bar_and(1, 128, got)) {
                if (!got && lane == 0) fail();
                break;
            }
            tc::tc_fence_after();
            const uint32_t acc = tmem + lane_base + buf * C::BUF_COLS;
            // issuer i's accumulator holds something only if the piece has > i stages
            const int nacc = min(C::NSPLIT, sg.s1 - sg.s0);
            for (int c0 = 0; c0 < t.n; c0 += 16) {
                // columns c0 .. c0 + 15: the hi and lo halves added (one term: as is)
                constexpr bool ONE = C::TERMS == 1;
                uint32_t rh[16], rl[16];
                float v[16];
                tc::tmem_ld_32x32b_x16(acc + c0, rh);
                if (!ONE) tc::tmem_ld_32x32b_x16(acc + t.nmma + c0, rl);
                tc::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    v[j] = __uint_as_float(rh[j]) + (ONE ? 0.f : __uint_as_float(rl[j]));
#pragma unroll
                for (int i = 1; i < C::NSPLIT; ++i) {
                    if (i >= nacc) break;
                    tc::tmem_ld_32x32b_x16(acc + i * C::ACC_COLS + c0, rh);
                    if (!ONE) tc::tmem_ld_32x32b_x16(acc + i * C::ACC_COLS + t.nmma + c0, rl);
                    tc::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        v[j] += __uint_as_float(rh[j]) + (ONE ? 0.f : __uint_as_float(rl[j]));
                }
                if constexpr (C::NARROW && MODE == MOE_GEMM_GATEUP) {
                    // A tile split between CTAs (one 16-column chunk): each part
                    // stores its sums in its slot and counts itself in; the last
                    // one adds every part in CTA order (the same sums whichever
                    // CTA is last) and finishes the tile.
                    const int c_first = cta_of(U, (long long)sg.tile * NST);
                    const int c_last = cta_of(U, (long long)sg.tile * NST + NST - 1);
                    if (c_first != c_last) {
                        // the parts: CTAs in [c_first, c_last] with a non-empty range
                        // (fewer stages than CTAs leave some ranges empty)
                        auto has_part = [&](int c) {
                            return U * (c + 1) / gridDim.x > U * c / gridDim.x;
                        };
                        int n_parts = 0;
                        for (int c = c_first; c <= c_last; ++c) n_parts += has_part(c) ? 1 : 0;
                        const int row = q * 32 + lane;
                        float *mine = args.sk_part +
                                      ((size_t)blockIdx.x * 2 + (sg.tile == t_first ? 0 : 1)) * (16 * 128);
#pragma unroll
                        for (int j = 0; j < 16; ++j) mine[j * 128 + row] = v[j];
                        __threadfence();
                        epi_sync();
                        if (warp == 3 && lane == 0)
                            *sk_last = atomicAdd(&args.sk_count[sg.tile], 1) == n_parts - 1;
                        epi_sync();
                        if (!*sk_last) break;  // another part finishes the tile
                        __threadfence();
                        float sum[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) sum[j] = 0.f;
                        for (int c = c_first; c <= c_last; ++c) {
                            if (!has_part(c)) continue;
                            // slot 0 holds a CTA's first tile, slot 1 its last
                            const int slot =
                                sg.tile == (int)(U * c / gridDim.x / NST) ? 0 : 1;
                            const float *part = args.sk_part + ((size_t)c * 2 + slot) * (16 * 128);
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                sum[j] += c == (int)blockIdx.x ? v[j] : __ldcg(part + j * 128 + row);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = sum[j];
                    }
                }
                if (MODE == MOE_GEMM_GATEUP) {
                    // Lanes 0..63 hold gate rows f0 + r, lanes 64..127 the same up rows.
                    // Gate warps finish columns 0..7 of the chunk, up warps 8..15; each
                    // hands the other half to its partner through shared memory.
                    float *stg = (float *)(smem + C::EPI_BASE);  // [16 columns][64 rows]
                    const bool gate = q < 2;
                    const int rr = (q & 1) * 32 + lane;          // row within the 64
#pragma unroll
                    for (int j = 0; j < 8; ++j) stg[(gate ? j + 8 : j) * 64 + rr] = v[gate ? j + 8 : j];
                    epi_sync();
                    const int F = args.M;
                    const int f = t.mt * 64 + rr;  // intermediate row of this lane
                    const size_t at_base = ((size_t)t.tt * (F / 128) + f / 128) * BSF_BYTES;
                    const int cblk = (f & 127) >> 5;
                    // Eight independent columns, each step over all eight before the
                    // next, so that reductions and conversions overlap instead of
                    // forming one long chain per column. SiLU in fast math: its
                    // ~1e-6 relative error is far below the E4M3 split that follows.
                    float h[8], rr8[8];
                    int sh[8], sl[8];
                    uint32_t hb[8], lb[8];
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = gate ? jj : jj + 8;
                        const float g = gate ? v[j] : stg[j * 64 + rr];
                        const float u = gate ? stg[j * 64 + rr] : v[j];
                        h[jj] = __fdividef(g, 1.f + __expf(-g)) * u;
                    }
                    if constexpr (BF16) {
                        // h in bf16 (round to nearest even) as GEMM2's B tile of K
                        // block f / 64: row r, bytes 2 (f % 64) .. of its 128-byte row,
                        // pre-swizzled; lanes f and f + 1 share one 4-byte store
                        uint8_t *hblk = args.h_tiles + ((size_t)t.tt * (F / 64) + f / 64) * MOE_GEMM_BTILE;
                        const int bo = (f & 63) * 2;  // byte of the row
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const uint32_t hv = f32_to_bf16_bits(h[jj]);
                            const uint32_t hn = __shfl_down_sync(0xFFFFFFFFu, hv, 1);
                            const int j = gate ? jj : jj + 8;
                            const int r = c0 + j;
                            if (r < t.n && (lane & 1) == 0)
                                *(uint32_t *)(hblk + r * 128 + (((bo >> 4) ^ (r & 7)) << 4) + (bo & 15)) =
                                    hv | (hn << 16);
                        }
                    } else if constexpr (FP4) {
                        // one MXFP4 term over this warp's 32 rows (one MX block along
                        // F): the scale from the block maximum, each value to the
                        // nearest E2M1 code; lanes f and f + 1 share a byte of the
                        // packed row (f even in the low nibble)
                        uint32_t nib[8];
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            sh[jj] = mx4::scale_exp(__uint_as_float(
                                __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h[jj])))));
                            nib[jj] = mx4::to_e2m1x2(h[jj] * mx8::exp2i(-sh[jj]), 0.f) & 0xFu;
                        }
                        uint8_t *hblk = args.h_tiles +
                                        ((size_t)t.tt * ((F / 128 + 1) / 2) + f / 256) * MOE_GEMM_BTILE;
                        const int bi = (f & 255) >> 1;  // byte of the packed row
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) {
                            const uint32_t up_nib = __shfl_down_sync(0xFFFFFFFFu, nib[jj], 1);
                            const int j = gate ? jj : jj + 8;
                            const int r = c0 + j;
                            if (r < t.n && (lane & 1) == 0)
                                hblk[r * 128 + (((bi >> 4) ^ (r & 7)) << 4) + (bi & 15)] =
                                    (uint8_t)(nib[jj] | (up_nib << 4));
                            if (r < t.n && lane == 0)
                                args.h_atoms[at_base + bsf_off(r, cblk)] = (uint8_t)(sh[jj] + 127);
                        }
                    } else {
                    // two-term E4M3 split over this warp's 32 rows (one MX block along F)
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        sh[jj] = mx8::scale_exp(__uint_as_float(
                            __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(h[jj])))));
#pragma unroll
                    for (int jj = 0; jj < 8; jj += 2) {
                        const uint32_t p = mx8::to_e4m3x2(h[jj] * mx8::exp2i(-sh[jj]),
                                                          h[jj + 1] * mx8::exp2i(-sh[jj + 1]));
                        const float2 back = mx8::from_e4m3x2(p);
                        hb[jj] = p & 0xFF;
                        hb[jj + 1] = (p >> 8) & 0xFF;
                        rr8[jj] = h[jj] - back.x * mx8::exp2i(sh[jj]);
                        rr8[jj + 1] = h[jj + 1] - back.y * mx8::exp2i(sh[jj + 1]);
                    }
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj)
                        sl[jj] = mx8::scale_exp(__uint_as_float(
                            __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(fabsf(rr8[jj])))));
#pragma unroll
                    for (int jj = 0; jj < 8; jj += 2) {
                        const uint32_t p = mx8::to_e4m3x2(rr8[jj] * mx8::exp2i(-sl[jj]),
                                                          rr8[jj + 1] * mx8::exp2i(-sl[jj + 1]));
                        lb[jj] = p & 0xFF;
                        lb[jj + 1] = (p >> 8) & 0xFF;
                    }
                    uint8_t *hblk =
                        args.h_tiles + ((size_t)t.tt * (F / 128) + f / 128) * MOE_GEMM_BTILE;
                    const int cb = f & 127;
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = gate ? jj : jj + 8;
                        if (c0 + j < t.n) {
                            // GEMM2 B tile of chunk f / 128: rows r (hi) and nmma + r (lo),
                            // byte f % 128 of the row, pre-swizzled
                            const int r = c0 + j, rlo = t.nmma + r;
                            hblk[r * 128 + (((cb >> 4) ^ (r & 7)) << 4) + (cb & 15)] = (uint8_t)hb[jj];
                            hblk[rlo * 128 + (((cb >> 4) ^ (rlo & 7)) << 4) + (cb & 15)] =
                                (uint8_t)lb[jj];
                            if (lane == 0) {
                                // GEMM2 chunk f / 128, block (f % 128) / 32; B rows hi r, lo nmma + r
                                args.h_atoms[at_base + bsf_off(c0 + j, cblk)] = (uint8_t)(sh[jj] + 127);
                                args.h_atoms[at_base + bsf_off(t.nmma + c0 + j, cblk)] =
                                    (uint8_t)(sl[jj] + 127);
                            }
                        }
                    }
                    }  // two-term split
                    epi_sync();
                } else if (args.y && args.y_bf16) {
                    // the rows' unweighted values in bf16: the four warps' 128
                    // rows of columns c0 .. c0 + 15 meet in shared memory (bf16,
                    // two buffers used in turn, so one barrier per 16 columns),
                    // then each thread writes 32 contiguous bytes of one token
                    // row, y[slot][mt * 128 + 16 p ..] (whole 128-byte lines;
                    // bf16 stored straight from the lanes made 64-byte half
                    // lines, measured slower than fp32 rows)
                    uint16_t *yb = (uint16_t *)args.y;
                    uint16_t *stg = (uint16_t *)(smem + C::EPI_BASE) + ((c0 >> 4) & 1) * (16 * 128);
#pragma unroll
                    for (int j = 0; j < 16; ++j) stg[j * 128 + q * 32 + lane] = f32_to_bf16_bits(v[j]);
                    epi_sync();
                    const int e = (warp - 3) * 32 + lane, j = e >> 3, p = e & 7;
                    if (c0 + j < t.n) {
                        const uint4 *src = (const uint4 *)(stg + j * 128 + p * 16);
                        uint4 *dst = (uint4 *)(yb + (size_t)(t.s0 + c0 + j) * args.Dout +
                                               t.mt * 128 + p * 16);
                        dst[0] = src[0];
                        dst[1] = src[1];
                    }
                } else if (args.y) {
                    // fp32 rows straight from the lanes, one 128-byte line per
                    // warp and column (token row): y[slot][mt * 128 + 32 q + lane]
                    float *yd = (float *)args.y + (size_t)t.s0 * args.Dout + t.mt * 128 + q * 32 + lane;
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < t.n) yd[(size_t)(c0 + j) * args.Dout] = v[j];
                } else {
                    // weighted values -> warp staging [16 columns][32 rows], then each
                    // lane adds 4 consecutive rows of one column with one vector reduction
                    float *stg = (float *)(smem + C::EPI_BASE) + (warp - 3) * 16 * 32;
                    // columns c0 .. c0 + 15 live in pf/pw[c0 / 32] of lanes c0 % 32 + j
                    const int ci = c0 >> 5, cl = c0 & 31;
                    int fl = pf[0];
                    float wv = pw[0];
#pragma unroll
                    for (int i = 1; i <= NT / 32; ++i)
                        if (ci == i) {
                            fl = pf[i];
                            wv = pw[i];
                        }
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        stg[j * 32 + lane] = __shfl_sync(0xFFFFFFFFu, wv, cl + j) * v[j];
                    __syncwarp();
                    const int d0 = t.mt * 128 + q * 32;
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int i = lane + 32 * u;  // float4 index: column i/8, rows 4*(i%8)..+3
                        const int j = i >> 3, g = i & 7;
                        const int flj = __shfl_sync(0xFFFFFFFFu, fl, cl + j);
                        if (c0 + j < t.n && flj >= 0) {
                            const float4 w4 = *(const float4 *)(stg + j * 32 + 4 * g);
                            float *dst = args.acc + (size_t)(flj / args.k) * args.Dout + d0 + 4 * g;
                            // evict_last: the accumulator rows stay in L2 while
                            // the weights stream through it (evict_first)
                            asm volatile(
                                "red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst),
                                "f"(w4.x), "f"(w4.y), "f"(w4.z), "f"(w4.w), "l"(pol_acc)
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

    // Wind-down after a timeout: every operand copy this CTA issued must land
    // before its shared memory is released. A stage filled in round r has
    // completed its full barrier phase r once both producers' arrivals and
    // bytes are in. The producers stop at most one round apart on a stage
    // (a fill of round r waited for the release of round r - 1, which needed
    // both fills of that round), so where only one of them filled the last
    // round, the missing arrival is made here and the wait then ends when the
    // issued bytes have landed.
    __syncthreads();
    if (*abort_p && tid == 0) {
        int never = 0;
        const int na = s_issued[0], nb = s_issued[1];
        for (int s = 0; s < C::SA; ++s) {
            const int ra = na > s ? (na - s + C::SA - 1) / C::SA : 0;  // rounds of slot s filled
            const int rb = nb > s ? (nb - s + C::SA - 1) / C::SA : 0;
            const int r = max(ra, rb);
            if (r == 0 || ra - rb > 1 || rb - ra > 1) continue;
            if (ra != rb) tc::mbar_arrive(&full[s]);
            tc::mbar_wait(&full[s], (uint32_t)((r - 1) & 1), LIMIT / 100 + 100000, &never);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Weight scales re-laid for the tensor cores: one 1 KB block per (expert,
// weight tile, pair of 128-wide K blocks), in the layout a 128x256b
// tcgen05.cp reads for one TMEM lane quadrant (8-row x 16-byte core
// matrices): lane l (0..31), 32-bit column j (0..7) at byte
// (l / 8) * 256 + (j / 4) * 128 + (l % 8) * 16 + (j % 4) * 4. Column j holds
// the four 32-wide block scales of tile row 32 * (j % 4) + l in K block
// 2 * pair + j / 4 (zero past the last block). For the gate/up GEMM a tile's
// rows 0..63 are gate rows mt*64 .. and rows 64..127 the same up rows; for
// the down GEMM a tile is 128 consecutive rows. One thread per 4-byte word.
__device__ __forceinline__ uint32_t atom_word(int64_t e, int mt, int pair, int wi, int M, int K,
                                              int mrows, const uint8_t *__restrict__ s,
                                              const uint8_t *__restrict__ s2) {
    const int KC = K / BK, ksb = K / 32;
    const int l = (wi / 64) * 8 + (wi % 32) / 4;   // lane
    const int j = ((wi % 64) / 32) * 4 + wi % 4;   // column
    const int m = 32 * (j % 4) + l;                // tile row
    const int kc = ATOM_BLOCKS * pair + j / 4;
    if (kc >= KC) return 0u;
    const uint8_t *src;
    if (s2 && m >= 64) src = s2 + ((e * M + (int64_t)mt * mrows + (m - 64)) * ksb + kc * 4);
    else src = s + ((e * M + (int64_t)mt * mrows + m) * ksb + kc * 4);
    return *(const uint32_t *)src;
}

__global__ void __launch_bounds__(256) moe_prepare_atoms_kernel(int64_t words, int M, int K,
                                                                int mrows, const uint8_t *__restrict__ s,
                                                                const uint8_t *__restrict__ s2,
                                                                uint32_t *__restrict__ out) {
    int64_t w = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (w >= words) return;
    const int MT = M / mrows, NP = (K / BK + ATOM_BLOCKS - 1) / ATOM_BLOCKS;
    const int64_t blk = w / 256;
    const int pair = (int)(blk % NP);
    const int64_t em = blk / NP;  // e * MT + mt
    out[w] = atom_word(em / MT, (int)(em % MT), pair, (int)(w % 256), M, K, mrows, s, s2);
}

// The same blocks for the experts just copied into slots miss_slot[0 .. *n_miss)
// (expert streaming), read from and written for those slots only.
__global__ void __launch_bounds__(256) moe_prepare_atoms_slots_kernel(
    int M, int K, int mrows, const uint8_t *__restrict__ s, const uint8_t *__restrict__ s2,
    uint32_t *__restrict__ out, const int *__restrict__ n_miss, const int32_t *__restrict__ miss_slot) {
    const int MT = M / mrows, NP = (K / BK + ATOM_BLOCKS - 1) / ATOM_BLOCKS;
    const int64_t per = (int64_t)MT * NP * 256;  // words per expert
    const int64_t total = per * (*n_miss);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int m = (int)(i / per);
        const int64_t w = i - (int64_t)m * per;
        const int64_t slot = miss_slot[m];
        const int64_t blk = w / 256;
        const int pair = (int)(blk % NP), mt = (int)(blk / NP);
        out[slot * per + w] = atom_word(slot, mt, pair, (int)(w % 256), M, K, mrows, s, s2);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
size_t moe_prepared_atoms_bytes(int E, int M, int K, int mrows) {
    const int KC = K / BK, NP = (KC + ATOM_BLOCKS - 1) / ATOM_BLOCKS;
    return (size_t)E * (M / mrows) * NP * SF_BYTES;
}

cudaError_t moe_launch_prepare_atoms_slots(int M, int K, int mrows, const uint8_t *s,
                                           const uint8_t *s2, uint8_t *out, const int *n_miss,
                                           const int32_t *miss_slot, int nsm, cudaStream_t st) {
    moe_prepare_atoms_slots_kernel<<<nsm * 4, 256, 0, st>>>(M, K, mrows, s, s2, (uint32_t *)out,
                                                            n_miss, miss_slot);
    return cudaGetLastError();
}

cudaError_t moe_launch_prepare_atoms(int E, int M, int K, int mrows, const uint8_t *s,
                                     const uint8_t *s2, uint8_t *out, cudaStream_t st) {
    const int64_t words = (int64_t)(moe_prepared_atoms_bytes(E, M, K, mrows) / 4);
    moe_prepare_atoms_kernel<<<(unsigned)((words + 255) / 256), 256, 0, st>>>(
        words, M, K, mrows, s, s2, (uint32_t *)out);
    return cudaGetLastError();
}

namespace {
// One persistent CTA per SM (grid = max_ctas, the SM count): the kernel's
// shared memory admits exactly one CTA per SM.
template <int MODE, int NT, int AF>
cudaError_t launch_gemm_t(const CUtensorMap *mA, const CUtensorMap *mA2, const MoeGemmArgs *args,
                          int max_ctas, cudaStream_t st) {
    using C = Cfg<MODE, NT, AF>;
    auto kern = moe_grouped_gemm_kernel<MODE, NT, AF>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (err != cudaSuccess) return err;
    if (max_ctas < 1) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(max_ctas), dim3(C::THREADS), (size_t)C::SMEM, st, *mA, *mA2,
                      *args);
}

template <int AF>
cudaError_t launch_gemm_fmt(int mode, const CUtensorMap *mA, const CUtensorMap *mA2,
                            const MoeGemmArgs *args, int max_rows, int grid, cudaStream_t st) {
    constexpr int NN = MOE_GEMM_NT_NARROW;
    // the narrow gate/up GEMM meets split tiles in sk_part (2 slots per CTA)
    if (max_rows <= NN && mode == MOE_GEMM_GATEUP && (!args->sk_part || !args->sk_count))
        return cudaErrorInvalidValue;
    if (max_rows <= NN)
        return mode == MOE_GEMM_GATEUP
                   ? launch_gemm_t<MOE_GEMM_GATEUP, NN, AF>(mA, mA2, args, grid, st)
                   : launch_gemm_t<MOE_GEMM_DOWN, NN, AF>(mA, mA2, args, grid, st);
    return mode == MOE_GEMM_GATEUP
               ? launch_gemm_t<MOE_GEMM_GATEUP, NTMAX, AF>(mA, mA2, args, grid, st)
               : launch_gemm_t<MOE_GEMM_DOWN, NTMAX, AF>(mA, mA2, args, grid, st);
}
}  // namespace

cudaError_t moe_launch_gemm(int mode, const CUtensorMap *mA, const CUtensorMap *mA2,
                            const MoeGemmArgs *args, int max_rows, int grid, int af,
                            cudaStream_t st) {
    switch (af) {
        case MOE_AF_E4M3X2: return launch_gemm_fmt<MOE_AF_E4M3X2>(mode, mA, mA2, args, max_rows, grid, st);
        case MOE_AF_MXF4: return launch_gemm_fmt<MOE_AF_MXF4>(mode, mA, mA2, args, max_rows, grid, st);
        case MOE_AF_BF16: return launch_gemm_fmt<MOE_AF_BF16>(mode, mA, mA2, args, max_rows, grid, st);
        default: return cudaErrorInvalidValue;
    }
}
