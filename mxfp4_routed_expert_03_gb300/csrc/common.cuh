// Shared device helpers of the routed-expert FFN library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#define MOE_MAX_TOPK 32
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_DMODEL 16384
#define MOE_MAX_DFF 8192

// Record the first device-side error; later errors keep the first one.
__device__ __forceinline__ void moe_flag(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

// fp32 -> bf16 bits, round to nearest even (NaN kept quiet).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

// 2^(b - 127) for an E8M0 scale byte b (255 -> NaN).
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    if (b == 255u) return __uint_as_float(0x7FC00000u);
    if (b == 0u) return __uint_as_float(0x00400000u);  // 2^-127 (fp32 subnormal)
    return __uint_as_float(b << 23);
}

// Programmatic dependent launch. A kernel launched with launch_pdl may start
// while its predecessor in the stream is still running (once every CTA of the
// predecessor has called grid_dep_launch or exited). grid_dep_wait blocks the
// calling thread until the predecessor has completed and its memory is
// visible; before it, a kernel may touch only what no running kernel writes.
// The library keeps one rule that makes this safe for its chains: a kernel
// whose predecessor may still run calls grid_dep_wait before it reads that
// predecessor's output, and calls grid_dep_launch only after its own wait or,
// in the grouped GEMMs, after reading nothing but the plan and the weights;
// so when a kernel starts, every kernel two or more launches back has
// completed. Both are no-ops in an ordinary launch.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Host: launch `kern` with programmatic dependent launch allowed (see
// grid_dep_wait). Every kernel of a chain asks for the largest shared-memory
// carve-out: an SM's L1 / shared split changes only when the SM is idle, so
// a small kernel's CTA left on an SM in the default split keeps the next
// kernel's large-shared-memory CTA (the grouped GEMMs) off that SM until it
// exits, even where both fit.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args... args) {
    cudaError_t err = cudaFuncSetAttribute((const void *)kern,
                                           cudaFuncAttributePreferredSharedMemoryCarveout,
                                           (int)cudaSharedmemCarveoutMaxShared);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}
