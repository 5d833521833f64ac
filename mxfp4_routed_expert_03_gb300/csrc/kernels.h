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
cudaError_t moe_launch_decode(int T, int D, int F, int E, int k, const uint16_t *x,
                              const moe_plan_buf *p, const moe_weights *w, uint16_t *out,
                              void *ws, int *status, const MoeProf &prof, cudaStream_t st);

// quant.cu
cudaError_t moe_launch_quant_x(int T, int D, const uint16_t *x, uint8_t *q_hi, uint8_t *q_lo,
                               uint8_t *s_hi, uint8_t *s_lo, cudaStream_t st);
cudaError_t moe_launch_schedule(int E, int ntmax, const int32_t *offsets, const int32_t *active,
                                int32_t *tt_prefix, int *status, cudaStream_t st);
cudaError_t moe_launch_finalize(int T, int D, const float *acc, uint16_t *out, cudaStream_t st);
cudaError_t moe_launch_gather_x(int max_tt, int E, int k, int n_rows, int D, int ntmax,
                                const int32_t *offsets, const int32_t *perm, const int32_t *active,
                                const int32_t *tt_prefix, const uint8_t *q_hi, const uint8_t *q_lo,
                                const uint8_t *s_hi, const uint8_t *s_lo, uint8_t *g_hi,
                                uint8_t *g_lo, uint8_t *atoms_hi, uint8_t *atoms_lo, int *status,
                                cudaStream_t st);

// grouped_gemm.cu
#include <cuda.h>
#define MOE_GEMM_GATEUP 0
#define MOE_GEMM_DOWN 1
#define MOE_GEMM_NTMAX 112

struct MoeGemmArgs {
    int E, k, n_rows;        // experts, top-k, T*k
    int M, MT, K, KC;        // weight rows per expert (F or D), M/128, reduction length, K/128
    int Dout;                // row stride of the fp32 output accumulator (d_model)
    const int32_t *offsets, *perm, *active, *tt_prefix;
    const float *topk_w;
    const uint8_t *a_atoms, *a2_atoms;  // weight scales as 512-byte atoms [E][M/128][K/128]
    const uint8_t *b_atoms_hi, *b_atoms_lo;  // activation scale atoms [token tile][K/128]
    uint8_t *h_hi, *h_lo;                    // GEMM1 outputs: h terms, slot order [T*k][M]
    uint8_t *h_atoms_hi, *h_atoms_lo;        // GEMM1 outputs: h scale atoms [token tile][M/128]
    float *acc;                        // GEMM2 output
    int *status;
    long long timeout_cycles;
};

size_t moe_gemm_smem_bytes(int mode);
cudaError_t moe_launch_prepare_atoms(int E, int M, int K, const uint8_t *s, uint8_t *out,
                                     cudaStream_t st);
cudaError_t moe_launch_gemm(int mode, const CUtensorMap *mA, const CUtensorMap *mA2,
                            const CUtensorMap *mBhi, const CUtensorMap *mBlo,
                            const MoeGemmArgs *args, int grid, cudaStream_t st);
