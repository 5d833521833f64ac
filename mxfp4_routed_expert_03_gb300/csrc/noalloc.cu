// Fixed scratch for moe_decode_noalloc: a file-scope device array, so callers
// that cannot allocate device memory can still run the decode path.
//
// The array holds the decode path's intermediate buffers (f16 h with its
// exponents and the per-slot fp32 expert outputs) for up to
// MOE_NOALLOC_MAX_ROWS routed rows (tokens x top_k) of a layer with
// d_ff <= MOE_NOALLOC_MAX_DFF and d_model <= MOE_NOALLOC_MAX_DMODEL. Every GPU
// that loads the library keeps it for the life of the process. All calls
// share it, so calls whose kernels overlap on the GPU race on it.
#include <cuda.h>

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

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
// Device address of g_decode_scratch per device, with the context it was
// looked up in: a device reset (or the primary context being torn down and
// created again) gives the device a new context, where the old address is
// stale, so the address is looked up again whenever the context changes.
struct ScratchAddr {
    CUcontext ctx;
    void *ptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

typedef CUresult (*ctx_get_current_fn)(CUcontext *);

// cuCtxGetCurrent, looked up through the runtime (the library does not link
// the driver library directly).
ctx_get_current_fn ctx_get_current() {
    static ctx_get_current_fn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (ctx_get_current_fn)p;
    }
    return fn;
}

}  // namespace

size_t moe_noalloc_scratch_bytes() { return kScratchBytes; }

// Device address of the fixed scratch on the current device. The first call on
// a device (and the first after its context changed) looks it up with
// cudaGetSymbolAddress, with that device current; in host code the array's
// name is only a host-side stand-in, never a device address, and must not be
// passed to a kernel. Returns cudaSuccess or the lookup's error.
cudaError_t moe_noalloc_scratch(void **ptr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // the context current on this thread (none yet on a thread that has not
    // used the device: the lookup below then binds the device's primary one)
    ctx_get_current_fn get = ctx_get_current();
    CUcontext ctx = nullptr;
    if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &a = g_scratch_addr[dev];
    if (!a.ptr || !ctx || a.ctx != ctx) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (err != cudaSuccess) return err;
        if (get && get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
        a.ctx = ctx;  // null: looked up again on the next call
        a.ptr = p;
    }
    *ptr = a.ptr;
    return cudaSuccess;
}
