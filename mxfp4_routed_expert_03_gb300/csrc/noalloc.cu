// Fixed scratch for moe_decode_noalloc: a file-scope device array, so callers
// that cannot allocate device memory can still run the decode path.
//
// The array holds the decode path's intermediate buffers (f16 h with its
// exponents and the per-slot fp32 expert outputs) for up to
// MOE_NOALLOC_MAX_ROWS routed rows (tokens x top_k) of a layer with
// d_ff <= MOE_NOALLOC_MAX_DFF and d_model <= MOE_NOALLOC_MAX_DMODEL. Every GPU
// that loads the library keeps it for the life of the process. All calls
// share it, so calls whose kernels overlap on the GPU race on it.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// Same region sizes the decode launcher carves (h16, exponents, y), at the
// largest shape the array accepts.
constexpr size_t kScratchBytes =
    round256((size_t)MOE_NOALLOC_MAX_ROWS * MOE_NOALLOC_MAX_DFF * 2) +
    round256((size_t)MOE_NOALLOC_MAX_ROWS * MOE_NOALLOC_MAX_DFF / 32) +
    round256((size_t)MOE_NOALLOC_MAX_ROWS * MOE_NOALLOC_MAX_DMODEL * sizeof(float));

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];  // device address of g_decode_scratch, per device
std::mutex g_scratch_mu;

}  // namespace

size_t moe_noalloc_scratch_bytes() { return kScratchBytes; }

// Device address of the fixed scratch on the current device. The first call on
// a device looks it up (cudaGetSymbolAddress, with that device current); in
// host code the array's name is not a device address and must not be passed
// to a kernel. Returns cudaSuccess or the lookup's error.
cudaError_t moe_noalloc_scratch(void **ptr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = p;
    }
    *ptr = g_scratch_addr[dev];
    return cudaSuccess;
}
