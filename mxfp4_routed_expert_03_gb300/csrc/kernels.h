// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/moe.h"

#define MOE_PLAN_CHUNK 64

// Optional events bracketing one kernel (see moe_profile_kernel).
struct MoeProf {
    int which;
    cudaEvent_t start, stop;
    void before(int k, cudaStream_t st) const {
        if (which == k && start) cudaEventRecord(start, st);
    }
    void after(int k, cudaStream_t st) const {
        if (which == k && stop) cudaEventRecord(stop, st);
    }
};
static inline bool moe_plan_is_small(int T) { return T <= 64; }

// route.cu
size_t moe_plan_ws_bytes(int T, int E);
cudaError_t moe_launch_plan(int T, int E, int k, const float *logits, const moe_plan_buf *p,
                            void *ws, int *status, cudaStream_t st);

// decode.cu
int moe_decode_per_lane(int K);
size_t moe_decode_ws_bytes(int T, int D, int F, int k);
// shared_out: optional fp32 [T][D] added to every token's combine (NULL: none).
// fp8: the weights are FP8 (E4M3FN codes [N][K], fp32 scales per 128 x 128
// block) instead of MXFP4.
// out[t] = bf16(sum_j topk_w[t][j] * y[inv[t k + j]] (+ shared[t])), j ascending:
// the deterministic combine of per-slot expert rows y [n_rows][D], fp32
// (moe_decode) or, with the _bf16 form, bf16 (moe_forward's FP4 mode).
cudaError_t moe_launch_combine_slots(int T, int D, int k, int n_rows, const float *topk_w,
                                     const int32_t *inv, const float *y, const float *shared,
                                     uint16_t *out, int *status, cudaStream_t st);
cudaError_t moe_launch_combine_slots_bf16(int T, int D, int k, int n_rows, const float *topk_w,
                                          const int32_t *inv, const uint16_t *y,
                                          const float *shared, uint16_t *out, int *status,
                                          cudaStream_t st);
cudaError_t moe_launch_decode(int T, int D, int F, int E, int k, const uint16_t *x,
                              const moe_plan_buf *p, const moe_weights *w, int fp8,
                              const float *shared_out, uint16_t *out, void *ws, int *status,
                              const MoeProf &prof, cudaStream_t st);

// noalloc.cu: fixed scratch of moe_decode_noalloc
#define MOE_NOALLOC_MAX_ROWS 256     // tokens x top_k
#define MOE_NOALLOC_MAX_DFF 2048
#define MOE_NOALLOC_MAX_DMODEL 8192
size_t moe_noalloc_scratch_bytes();
cudaError_t moe_noalloc_scratch(void **ptr);

// quant.cu
cudaError_t moe_launch_quant_x(int T, int D, const uint16_t *x, uint8_t *q_hi, uint8_t *q_lo,
                               uint8_t *s_hi, uint8_t *s_lo, cudaStream_t st);
cudaError_t moe_launch_schedule(int E, int ntmax, const int32_t *offsets, const int32_t *active,
                                int32_t *tt_prefix, int *status, cudaStream_t st);
// T <= MOE_GEMM_NT_NARROW: quantise + gather + identity schedule (+ zero acc
// when acc is not null, and sk_count[0 .. n_sk), the grouped GEMMs'
// split-tile counters) in one launch.
cudaError_t moe_launch_prep_small(int T, int E, int k, int D, const int32_t *offsets,
                                  const int32_t *perm, const int32_t *active, const uint16_t *x,
                                  int32_t *tt_prefix, uint8_t *tiles, uint8_t *atoms, float *acc,
                                  int *sk_count, int n_sk, int *status, cudaStream_t st);
// The FP4 x FP4 mode's counterparts: one MXFP4 term per activation, in the
// FP4 tile layout (see moe_launch_gemm).
cudaError_t moe_launch_prep_small_fp4(int T, int E, int k, int D, const int32_t *offsets,
                                      const int32_t *perm, const int32_t *active,
                                      const uint16_t *x, int32_t *tt_prefix, uint8_t *tiles,
                                      uint8_t *atoms, float *acc, int *sk_count, int n_sk,
                                      int *status, cudaStream_t st);
// Larger batches: every token's row once to MXFP4 (q [T][D/2], biased scale
// bytes s [T][D/32]), then the token tiles gathered from them.
cudaError_t moe_launch_quant_x_fp4(int T, int D, const uint16_t *x, uint8_t *q, uint8_t *s,
                                   cudaStream_t st);
cudaError_t moe_launch_gather_x_fp4(int max_tt, int E, int k, int n_rows, int D,
                                    const int32_t *offsets, const int32_t *perm,
                                    const int32_t *active, const int32_t *tt_prefix,
                                    const uint8_t *q, const uint8_t *s, uint8_t *tiles,
                                    uint8_t *atoms, int *status, cudaStream_t st);
cudaError_t moe_launch_finalize(int T, int D, const float *acc, uint16_t *out, cudaStream_t st);
cudaError_t moe_launch_gather_x(int max_tt, int E, int k, int n_rows, int D, int ntmax,
                                const int32_t *offsets, const int32_t *perm, const int32_t *active,
                                const int32_t *tt_prefix, const uint8_t *q_hi, const uint8_t *q_lo,
                                const uint8_t *s_hi, const uint8_t *s_lo, uint8_t *tiles,
                                uint8_t *atoms, int *status, cudaStream_t st);

// fp8.cu: the FP8 lane's prefill side (bf16 copy of the experts, bf16 tiles)
cudaError_t moe_launch_fp8_dequant(int E, int N, int K, const uint8_t *codes, const float *scales,
                                   uint16_t *out, cudaStream_t st);
cudaError_t moe_launch_prep_small_bf16(int T, int E, int k, int D, const int32_t *offsets,
                                       const int32_t *perm, const int32_t *active,
                                       const uint16_t *x, int32_t *tt_prefix, uint8_t *tiles,
                                       float *acc, int *sk_count, int n_sk, int *status,
                                       cudaStream_t st);
cudaError_t moe_launch_gather_x_bf16(int max_tt, int E, int k, int n_rows, int D,
                                     const int32_t *offsets, const int32_t *perm,
                                     const int32_t *active, const int32_t *tt_prefix,
                                     const uint16_t *x, uint8_t *tiles, int *status,
                                     cudaStream_t st);

// grouped_gemm.cu
#include <cuda.h>
#define MOE_GEMM_GATEUP 0
#define MOE_GEMM_DOWN 1
#define MOE_GEMM_NTMAX 112
#define MOE_GEMM_NT_NARROW 16  // token rows per tile of the narrow variant
#define MOE_GEMM_BTILE (2 * MOE_GEMM_NTMAX * 128)  // bytes of one activation B tile block

struct MoeGemmArgs {
    int E, k, n_rows;        // experts, top-k, T*k
    int M, MT, K, KC;        // weight rows per expert (F or D), M/128, reduction length, K/128
    int Dout;                // row stride of the fp32 output accumulator (d_model)
    const int32_t *offsets, *perm, *active, *tt_prefix;
    const float *topk_w;
    const int32_t *w_index;  // weight slot of expert e (expert streaming), or NULL: e itself
    int n_wexp;              // experts held by the weight arrays (bound for w_index values)
    const uint8_t *a_atoms;  // weight scale blocks [E][weight tiles][K/256][1 KB]
    const uint8_t *b_tiles;  // activation B tiles [token tile][K/128][2*NTMAX rows][128 B]:
                             // rows [0, nmma) the hi term, [nmma, 2 nmma) the lo term,
                             // each 128-byte row pre-swizzled (16-byte chunk c at c ^ row % 8)
    const uint8_t *b_atoms;  // their scales [token tile][K/128][1 KB] (see bsf_off)
    uint8_t *h_tiles;        // GEMM1 output: h as GEMM2's B tiles [token tile][M/128][...]
    uint8_t *h_atoms;        // GEMM1 output: h scales [token tile][M/128][1 KB]
    float *acc;                        // GEMM2 output
    // Narrow variant (stream-K split of the stages over the CTAs): gate/up
    // tiles split between CTAs meet here. sk_part: per CTA two slots of
    // 16 x 128 fp32 partial sums (its first and its last tile); sk_count:
    // per weight tile the parts that arrived, zero before the launch.
    float *sk_part;
    int *sk_count;
    // Wide down GEMM, when not null: each routed row's unweighted output goes
    // to y[slot][0 .. Dout) (slot: its position in perm order) with plain
    // stores of whole 128-byte lines, for the deterministic combine; acc is
    // then unused. y_bf16: bf16 rows (rounded to nearest even) staged through
    // shared memory, else fp32 rows stored straight from the lanes.
    void *y;
    int y_bf16;
    int *status;
    long long timeout_cycles;
    int inject;              // MOE_INJECT_NONE, or a test hook (see moe_set_fault_injection)
};

size_t moe_prepared_atoms_bytes(int E, int M, int K, int mrows);
cudaError_t moe_launch_prepare_atoms(int E, int M, int K, int mrows, const uint8_t *s,
                                     const uint8_t *s2, uint8_t *out, cudaStream_t st);
// Arithmetic formats of the grouped GEMMs (af):
//  MOE_AF_E4M3X2  MXFP4 weights (8-bit containers) x two-term E4M3 activations,
//                 kind::mxf8f6f4; K blocks of 128
//  MOE_AF_MXF4    the FP4 x FP4 mode: packed MXFP4 weights x one MXFP4 term,
//                 kind::mxf4; activation tiles hold one 128-byte row per token
//                 per 256-wide K chunk (chunk c of token tile tt at block
//                 tt * ceil(K / 256) + c of b_tiles / h_tiles), scale blocks
//                 as for the two-term format, hi rows only
//  MOE_AF_BF16    bf16 weights x bf16 activations, kind::f16, no scales; K
//                 blocks of 64 (one 128-byte row per token and block, block
//                 kb of token tile tt at tt * (K / 64) + kb); args.KC = K / 64
#define MOE_AF_E4M3X2 0
#define MOE_AF_MXF4 1
#define MOE_AF_BF16 2
// max_rows: bound on any expert's routed rows (T for distinct top-k experts);
// at most MOE_GEMM_NT_NARROW selects the narrow-tile variant.
cudaError_t moe_launch_gemm(int mode, const CUtensorMap *mA, const CUtensorMap *mA2,
                            const MoeGemmArgs *args, int max_rows, int grid, int af,
                            cudaStream_t st);

// stream.cu: expert streaming (HBM slot cache in front of host memory)
struct MoeStreamHdr {
    int clock;       // calls so far
    int last_miss;   // misses of the last call (entries of miss_e / miss_s)
    int pad[2];
    unsigned long long hits, misses;  // totals over all calls
};
struct MoeStreamView {
    MoeStreamHdr *hdr;
    int32_t *slot_of;    // [E] slot holding expert e, or -1
    int32_t *expert_of;  // [S] expert held by slot s, or -1
    int32_t *stamp;      // [S] clock of the slot's last use (0: never)
    int32_t *miss_e, *miss_s;  // [S] the last call's missing experts and their slots
};
struct MoeStreamCopy {  // gate_q, gate_s, up_q, up_s, down_q, down_s
    const uint8_t *host[6];
    uint8_t *slot[6];
    int64_t bytes[6];  // per expert, multiples of 16
};
size_t moe_stream_state_size(int E, int S);
MoeStreamView moe_stream_view(void *state, int E, int S);
cudaError_t moe_launch_stream_init(int E, int S, void *state, cudaStream_t st);
cudaError_t moe_launch_stream_lru(int E, int S, const int32_t *active, void *state, int *status,
                                  cudaStream_t st);
cudaError_t moe_launch_stream_copy(int E, int S, void *state, const MoeStreamCopy *c, int nsm,
                                   cudaStream_t st);
// store.cu: decode of compressed-store experts into cache slots. Items are the
// pairs (experts[m], slots[m]), m < count, where count is *n_dev when n_dev is
// set (clamped to [0, max_items]) and n_host otherwise.
struct MoeStoreJob {
    const uint8_t *blob;
    int64_t blob_bytes;
    const moe_tile_rec *tiles;
    const uint16_t *tables;
    int E, tpe, n_slots;
    int64_t bytes[6];  // per expert and array
    int first[7];      // first tile of each array within an expert
    uint8_t *dst[6];   // slot arrays (n_slots experts each)
    const int32_t *experts, *slots;
    const int32_t *n_dev;
    int n_host, max_items;
    int *status;
};
// Fills bytes/first/tpe from the layer shape; false on a bad shape.
bool moe_store_job_shape(int D, int F, MoeStoreJob &j);
cudaError_t moe_launch_store_decode(const MoeStoreJob &j, int nsm, cudaStream_t st);
// grouped_gemm.cu: prepared scale blocks of the slots listed in miss_s[0 .. *n_miss)
cudaError_t moe_launch_prepare_atoms_slots(int M, int K, int mrows, const uint8_t *s,
                                           const uint8_t *s2, uint8_t *out, const int *n_miss,
                                           const int32_t *miss_slot, int nsm, cudaStream_t st);

// dense_gemm.cu: bf16 tcgen05 GEMMs of the router and the shared expert
#define MOE_DENSE_ROUTER 0  // 3 bf16 terms of W_r, fp32 store out_f32[t][m] (m < M)
#define MOE_DENSE_SWIGLU 1  // gate/up (64 + 64 rows per tile), bf16 store out_bf16[t][f]
#define MOE_DENSE_STORE 2   // 1 term, fp32 store out_f32[t][m] (m < M)
#define MOE_DENSE_NTILE 192  // tokens per tile

struct MoeDenseArgs {
    int M;          // output rows (experts, d_ff or d_model)
    int N;          // tokens
    int K;          // reduction length, a multiple of 64
    int ldo;        // row stride of the output (elements)
    float *out_f32;
    uint16_t *out_bf16;
    int *status;
    long long timeout_cycles;
};

cudaError_t moe_launch_split3(int64_t n, const float *w, uint16_t *t0, uint16_t *t1, uint16_t *t2,
                              cudaStream_t st);
int moe_dense_tiles(int epi, int M, int N);
cudaError_t moe_launch_dense(int epi, const CUtensorMap *a0, const CUtensorMap *a1,
                             const CUtensorMap *a2, const CUtensorMap *b,
                             const MoeDenseArgs *args, int grid, cudaStream_t st);
