// Expert streaming: a per-layer HBM slot cache in front of experts kept in
// host memory (the pages' routed-expert store with its per-layer online LRU
// slot cache: Moonshine README, "How the engine works"; Moonshine GitHub
// README, "Decode"). The cache is managed on the device so that a call needs
// no host round trip: one CTA applies the replacement rule to the plan's
// active experts, a grid-stride kernel copies the missing experts from host
// memory (GPU reads over NVLink-C2C on Grace) into their slots, and the
// grouped GEMMs then address weights through slot_of[].
//
// Replacement rule: each call advances a clock; resident active experts stamp
// their slot with it (hits); missing experts, in increasing expert index,
// take the slots not stamped by this call in increasing (stamp, slot) order
// (empty slots carry stamp 0), evicting whatever those slots held.
#include "common.cuh"
#include "kernels.h"

#define FULL_MASK 0xFFFFFFFFu

size_t moe_stream_state_size(int E, int S) {
    const size_t b = sizeof(MoeStreamHdr) + sizeof(int32_t) * ((size_t)E + 4 * (size_t)S);
    return (b + 255) / 256 * 256;
}

MoeStreamView moe_stream_view(void *state, int E, int S) {
    MoeStreamView v;
    v.hdr = (MoeStreamHdr *)state;
    int32_t *p = (int32_t *)((unsigned char *)state + sizeof(MoeStreamHdr));
    v.slot_of = p;
    v.expert_of = p + E;
    v.stamp = v.expert_of + S;
    v.miss_e = v.stamp + S;
    v.miss_s = v.miss_e + S;
    return v;
}

namespace {

__global__ void moe_stream_init_kernel(int E, int S, MoeStreamView v) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i == 0) {
        v.hdr->clock = 0;
        v.hdr->last_miss = 0;
        v.hdr->hits = 0;
        v.hdr->misses = 0;
    }
    if (i < E) v.slot_of[i] = -1;
    if (i < S) {
        v.expert_of[i] = -1;
        v.stamp[i] = 0;
        v.miss_e[i] = -1;
        v.miss_s[i] = -1;
    }
}

// Exclusive block scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_scan_1024(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(FULL_MASK, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const int t = warp_tot[lane];
        int ti = t;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(FULL_MASK, ti, off);
            if (lane >= off) ti += o;
        }
        warp_tot[lane] = ti - t;
        if (lane == 31) warp_tot[32] = ti;
    }
    __syncthreads();
    const int r = warp_tot[wid] + inc - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

// One CTA of 1024 threads (E <= 1024, S <= 1024).
__global__ void __launch_bounds__(1024) moe_stream_lru_kernel(int E, int S,
                                                              const int32_t *__restrict__ active,
                                                              MoeStreamView v, int *status) {
    __shared__ unsigned long long s_key[1024];
    __shared__ int s_tot[33];
    __shared__ int s_clock, s_hits, s_bad;
    const int tid = threadIdx.x;
    int n = active[0];
    if (tid == 0) {
        s_clock = v.hdr->clock + 1;
        v.hdr->clock = s_clock;
        s_hits = 0;
        s_bad = 0;
    }
    if (n < 0 || n > E) {
        if (tid == 0) moe_flag(status, MOE_ERR_BAD_INDEX);
        n = 0;
    }
    __syncthreads();
    const int clock = s_clock;
    // hits: resident active experts stamp their slots
    int e = -1, miss = 0;
    if (tid < n) {
        e = active[1 + tid];
        if (e < 0 || e >= E) {
            moe_flag(status, MOE_ERR_BAD_INDEX);
            e = -1;
        } else {
            const int s = v.slot_of[e];
            if (s >= 0 && s < S && v.expert_of[s] == e) {
                v.stamp[s] = clock;
                atomicAdd(&s_hits, 1);
            } else {
                miss = 1;
            }
        }
    }
    __syncthreads();
    // candidate slots, oldest first: key (stamp, slot); stamped-now slots last
    unsigned long long key = ~0ull;
    if (tid < S) {
        const int st = v.stamp[tid];
        if (st != clock) key = ((unsigned long long)(uint32_t)st << 32) | (uint32_t)tid;
    }
    s_key[tid] = key;
    __syncthreads();
    for (int size = 2; size <= 1024; size <<= 1) {  // bitonic sort, ascending
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int j = tid ^ stride;
            if (j > tid) {
                const unsigned long long a = s_key[tid], b = s_key[j];
                const bool up = (tid & size) == 0;
                if ((a > b) == up) {
                    s_key[tid] = b;
                    s_key[j] = a;
                }
            }
            __syncthreads();
        }
    }
    // misses in increasing expert index (the active list is ascending) take
    // the oldest candidates in order
    int total = 0;
    const int rank = block_scan_1024(miss, s_tot, total);
    if (miss) {
        const unsigned long long k = s_key[rank];
        if (k == ~0ull) {
            atomicExch(&s_bad, 1);
        } else {
            const int s = (int)(k & 0xFFFFFFFFull);
            const int old = v.expert_of[s];
            if (old >= 0 && old < E) v.slot_of[old] = -1;
            v.expert_of[s] = e;
            v.slot_of[e] = s;
            v.stamp[s] = clock;
            v.miss_e[rank] = e;
            v.miss_s[rank] = s;
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (s_bad) moe_flag(status, MOE_ERR_UNSUPPORTED);  // more active experts than slots
        v.hdr->last_miss = s_bad ? 0 : total;
        v.hdr->hits += (unsigned long long)s_hits;
        v.hdr->misses += (unsigned long long)(s_bad ? 0 : total);
    }
}

// Copies the last call's missing experts from host memory into their slots:
// the six arrays of each expert, 16 bytes per thread step, grid-stride.
__global__ void __launch_bounds__(256) moe_stream_copy_kernel(MoeStreamView v, MoeStreamCopy c) {
    const int n_miss = v.hdr->last_miss;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
#pragma unroll 1
    for (int a = 0; a < 6; ++a) {
        const int64_t chunks = c.bytes[a] / 16;
        const int64_t total = chunks * n_miss;
        for (int64_t i = t0; i < total; i += stride) {
            const int m = (int)(i / chunks);
            const int64_t q = i - (int64_t)m * chunks;
            const int e = v.miss_e[m], s = v.miss_s[m];
            const uint4 *src = (const uint4 *)(c.host[a] + (size_t)e * c.bytes[a]) + q;
            uint4 *dst = (uint4 *)(c.slot[a] + (size_t)s * c.bytes[a]) + q;
            *dst = *src;
        }
    }
}

}  // namespace

cudaError_t moe_launch_stream_init(int E, int S, void *state, cudaStream_t st) {
    const int n = E > S ? E : S;
    moe_stream_init_kernel<<<(n + 255) / 256, 256, 0, st>>>(E, S, moe_stream_view(state, E, S));
    return cudaGetLastError();
}

cudaError_t moe_launch_stream_lru(int E, int S, const int32_t *active, void *state, int *status,
                                  cudaStream_t st) {
    moe_stream_lru_kernel<<<1, 1024, 0, st>>>(E, S, active, moe_stream_view(state, E, S), status);
    return cudaGetLastError();
}

cudaError_t moe_launch_stream_copy(int E, int S, void *state, const MoeStreamCopy *c, int nsm,
                                   cudaStream_t st) {
    moe_stream_copy_kernel<<<nsm * 8, 256, 0, st>>>(moe_stream_view(state, E, S), *c);
    return cudaGetLastError();
}
