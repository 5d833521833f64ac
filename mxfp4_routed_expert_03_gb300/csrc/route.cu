// Routing: per-token top-k with softmax weights (K1) and the per-expert route
// plan (K2: histogram, exclusive scan, stable counting-sort scatter).
//
// Each token selects top_k of n_experts experts (MoonTail, intro; Moonshine
// README, "How the engine works"). All rows selecting each expert are then
// grouped and only the experts with rows are touched (Moonshine README,
// "How the engine works", prefill paragraph; Moonshine GitHub README,
// "Prefill"). Order: descending logit, ties to the lower expert index; the
// weights are the softmax over the selected logits. The plan orders the flat
// indices t*k+j by (expert, flat index), so it is unique and bit-exact.
#include "common.cuh"
#include "kernels.h"

#define FULL_MASK 0xFFFFFFFFu

namespace {

// Order-preserving 32-bit key of a logit: a larger key is a larger value;
// -0 and +0 share a key (they compare equal). NaN is mapped to -inf first.
__device__ __forceinline__ uint32_t logit_key(float v) {
    const uint32_t u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// Keys of one warp's k largest: lane l holds key[i] of position l + 32 i
// (i < NK); positions order equal keys. Returns in lane j < k the j-th
// selection's position and key (descending key, ties to the lower
// position). `scratch` is k entries of warp-private shared memory.
//
// Selection by threshold rather than k rounds of arg-max: a bitwise search
// finds the k-th largest key t (the largest x with at least k keys >= x),
// stopping early once exactly k keys are >= the prefix found so far; every
// key > t is selected, and of the keys equal to t the lowest positions fill
// the remaining places. The k winners are then ranked by (key, position).
// The per-lane counts are summed in independent partial sums: a single
// dependent chain over a lane's keys made each of the 32 steps several
// hundred cycles.
template <int NK>
__device__ __forceinline__ void warp_select(const uint32_t (&key)[NK], int k, int lane,
                                            uint2 *scratch, int &pos_out, uint32_t &key_out) {
    uint32_t thr = 0u;
    for (int b = 31; b >= 0; --b) {
        const uint32_t cand = thr | (1u << b);
        int c[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < NK; ++i) c[i & 3] += key[i] >= cand ? 1 : 0;
        const int tot =
            (int)__reduce_add_sync(FULL_MASK, (unsigned)((c[0] + c[1]) + (c[2] + c[3])));
        if (tot >= k) {
            thr = cand;
            if (tot == k) break;  // the keys >= thr are the selection
        }
    }
    uint32_t sel = 0u;
    int gt = 0;
#pragma unroll
    for (int i = 0; i < NK; ++i)
        if (key[i] > thr) {
            sel |= 1u << i;
            ++gt;
        }
    int need = k - (int)__reduce_add_sync(FULL_MASK, (unsigned)gt);  // keys equal to thr to take
#pragma unroll
    for (int i = 0; i < NK; ++i) {
        if (need > 0) {  // warp-uniform
            // row i holds positions 32 i + lane: lower lane = lower position
            const uint32_t m = __ballot_sync(FULL_MASK, key[i] == thr);
            const int take = min(need, __popc(m));
            if (((m >> lane) & 1u) && __popc(m & lanemask_lt()) < take) sel |= 1u << i;
            need -= take;
        }
    }
    // compact the k selections into scratch, then rank them
    const int mine = __popc(sel);
    int pos = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(FULL_MASK, pos, off);
        if (lane >= off) pos += o;
    }
    pos -= mine;
#pragma unroll
    for (int i = 0; i < NK; ++i)
        if ((sel >> i) & 1u) scratch[pos++] = make_uint2(key[i], (uint32_t)(lane + 32 * i));
    __syncwarp();
    uint2 me = make_uint2(0u, 0u);
    int r[4] = {0, 0, 0, 0};
    if (lane < k) {
        me = scratch[lane];
#pragma unroll
        for (int q = 0; q < MOE_MAX_TOPK; ++q) {
            if (q < k) {
                const uint2 o = scratch[q];
                r[q & 3] += (o.x > me.x || (o.x == me.x && o.y < me.y)) ? 1 : 0;
            }
        }
    }
    __syncwarp();
    if (lane < k) scratch[(r[0] + r[1]) + (r[2] + r[3])] = me;
    __syncwarp();
    pos_out = -1;
    key_out = 0u;
    if (lane < k) {
        const uint2 w = scratch[lane];
        pos_out = (int)w.y;
        key_out = w.x;
    }
    __syncwarp();
}

// Key of expert e of a logit row (NaN counts as -inf and sets nan_seen);
// positions past E get key 0, below every real key.
__device__ __forceinline__ uint32_t row_key(const float *row, int e, int E, bool &nan_seen) {
    if (e >= E) return 0u;
    float t = row[e];
    if (t != t) {
        nan_seen = true;
        t = -INFINITY;
    }
    return logit_key(t);
}

// Sort value of expert e's logit key: larger is earlier in the selection
// order (descending logit, then ascending index); all values distinct.
__device__ __forceinline__ uint64_t sort_value(uint32_t key, int e) {
    return ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)e);
}

__device__ __forceinline__ uint64_t shfl_xor64(uint64_t v, int m) {
    const uint32_t lo = __shfl_xor_sync(FULL_MASK, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(FULL_MASK, (uint32_t)(v >> 32), m);
    return ((uint64_t)hi << 32) | lo;
}

// Sorts P independent sets of 64 values in descending order, interleaved so
// that their dependent chains overlap: element n = 2 lane + h of set p in
// v[p][h]. Bitonic network: for block size K = 2 .. 64 and distance
// J = K / 2 .. 1, element n is paired with n ^ J and the pair ordered
// descending where (n & K) == 0, ascending elsewhere (the last block, K = 64,
// orders everything descending).
template <int P>
__device__ __forceinline__ void warp_sort64(uint64_t (&v)[P][2], int lane) {
#pragma unroll
    for (int K = 2; K <= 64; K <<= 1) {
#pragma unroll
        for (int J = K >> 1; J > 0; J >>= 1) {
            if (J == 1) {  // partners in the same lane
                const bool desc = ((2 * lane) & K) == 0;
#pragma unroll
                for (int q = 0; q < P; ++q) {
                    const uint64_t a = v[q][0], b = v[q][1];
                    const uint64_t mx = a > b ? a : b, mn = a > b ? b : a;
                    v[q][0] = desc ? mx : mn;
                    v[q][1] = desc ? mn : mx;
                }
            } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int n = 2 * lane + h;
                    const bool take_max = (((n & K) == 0) == ((n & J) == 0));
#pragma unroll
                    for (int q = 0; q < P; ++q) {
                        const uint64_t o = shfl_xor64(v[q][h], J >> 1);
                        v[q][h] = take_max ? (v[q][h] > o ? v[q][h] : o) : (v[q][h] > o ? o : v[q][h]);
                    }
                }
            }
        }
    }
}

// Top-k of a warp's keys, as warp_select, by a threshold instead of a
// bitwise search when it can: the k-th largest of the 32 lanes' maxima is at
// most the k-th largest key (the k lanes with the largest maxima hold k keys
// at least that large), so every selected key is >= it. When at most 64 keys
// are, they are gathered (with their positions) and sorted by one bitonic
// network, and the first k are the selection. Otherwise (many keys equal or
// close to it) warp_select decides. About 500 instructions per warp against
// the bitwise search's 32 compares per lane and bit, which left a batch of
// one warp per token issue-bound. scratch: 64 x 8 bytes of warp-private
// shared memory (as uint2: 64 entries).
template <int NK>
__device__ __forceinline__ void warp_select_thr(const uint32_t (&key)[NK], int k, int lane,
                                                uint2 *scratch, int &pos_out, uint32_t &key_out) {
    if (k > 16) {  // the k-th largest of 32 maxima bounds too little: nearly always > 64 keys
        warp_select<NK>(key, k, lane, scratch, pos_out, key_out);
        return;
    }
    uint32_t m = 0u;
#pragma unroll
    for (int i = 0; i < NK; ++i) m = key[i] > m ? key[i] : m;
    // the lane maxima in descending order over the lanes (bitonic, as
    // warp_sort64 with one value per lane)
#pragma unroll
    for (int K = 2; K <= 32; K <<= 1) {
#pragma unroll
        for (int J = K >> 1; J > 0; J >>= 1) {
            const uint32_t o = __shfl_xor_sync(FULL_MASK, m, J);
            const bool take_max = ((lane & K) == 0) == ((lane & J) == 0);
            m = take_max ? (m > o ? m : o) : (m > o ? o : m);
        }
    }
    const uint32_t t0 = __shfl_sync(FULL_MASK, m, k - 1);
    int c[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < NK; ++i) c[i & 1] += key[i] >= t0 ? 1 : 0;
    const int mine = c[0] + c[1];
    const int total = (int)__reduce_add_sync(FULL_MASK, (unsigned)mine);
    if (total > 64) {
        warp_select<NK>(key, k, lane, scratch, pos_out, key_out);
        return;
    }
    int off = mine;  // exclusive prefix of the lanes' counts
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(FULL_MASK, off, d);
        if (lane >= d) off += o;
    }
    off -= mine;
    uint64_t *cand = reinterpret_cast<uint64_t *>(scratch);
#pragma unroll
    for (int i = 0; i < NK; ++i)
        if (key[i] >= t0) cand[off++] = sort_value(key[i], lane + 32 * i);
    __syncwarp();
    uint64_t v[1][2];
    v[0][0] = 2 * lane < total ? cand[2 * lane] : 0ull;
    v[0][1] = 2 * lane + 1 < total ? cand[2 * lane + 1] : 0ull;
    __syncwarp();
    warp_sort64<1>(v, lane);
    // selection j is element j of the sorted 64: lane j / 2, half j % 2
    const int src = (lane >> 1) & 15;
    const uint32_t lo0 = __shfl_sync(FULL_MASK, (uint32_t)v[0][0], src);
    const uint32_t hi0 = __shfl_sync(FULL_MASK, (uint32_t)(v[0][0] >> 32), src);
    const uint32_t lo1 = __shfl_sync(FULL_MASK, (uint32_t)v[0][1], src);
    const uint32_t hi1 = __shfl_sync(FULL_MASK, (uint32_t)(v[0][1] >> 32), src);
    pos_out = -1;
    key_out = 0u;
    if (lane < k) {
        pos_out = (int)(0xFFFFFFFFu - ((lane & 1) ? lo1 : lo0));
        key_out = (lane & 1) ? hi1 : hi0;
    }
}

// Warp-cooperative top-k of one token's logits (k <= 32, k <= E <= 1024).
// On return lane j < k holds the j-th selection (expert index, logit):
// descending logit, ties to the lower expert index. NaN logits count as -inf
// and set nan_seen. Lane l owns experts l, l + 32, ... (coalesced loads).
// THR: the threshold select (fewer dependent steps: the small-batch plan,
// where one warp's latency is the time); else the bitwise search (fewer
// instructions: the large-batch kernel, where many warps share each SM and
// the threshold select measured 1.8x slower). scratch: 64 entries of
// warp-private shared memory (k entries without THR).
template <bool THR>
__device__ __forceinline__ void warp_topk(const float *row, int E, int k, int lane, int &my_e,
                                          float &my_v, bool &nan_seen, uint2 *scratch) {
    uint32_t key[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) key[i] = row_key(row, lane + 32 * i, E, nan_seen);
    uint32_t kv;
    if constexpr (THR)
        warp_select_thr<32>(key, k, lane, scratch, my_e, kv);
    else
        warp_select<32>(key, k, lane, scratch, my_e, kv);
    my_v = lane < k ? key_logit(kv) : -INFINITY;
}

// Softmax over the k selected logits held by lanes 0..k-1.
__device__ __forceinline__ float warp_select_weight(float my_v, int k, int lane) {
    float vmax = __shfl_sync(FULL_MASK, my_v, 0);
    float ex = (lane < k) ? expf(my_v - vmax) : 0.f;
    float s = ex;
#pragma unroll
    for (int off = 16; off; off >>= 1) s += __shfl_xor_sync(FULL_MASK, s, off);
    return ex / s;
}

// Exclusive block scan of one int per thread over a block of NW warps.
template <int NW>
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int &total) {
    int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(FULL_MASK, inc, off);
        if (lane >= off) inc += o;
    }
    if (lane == 31) warp_tot[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        int t = lane < NW ? warp_tot[lane] : 0;
        int ti = t;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(FULL_MASK, ti, off);
            if (lane >= off) ti += o;
        }
        warp_tot[lane] = ti - t;  // exclusive prefix of warp totals
        if (lane == 31) warp_tot[32] = ti;
    }
    __syncthreads();
    int r = warp_tot[wid] + inc - v;
    total = warp_tot[32];
    __syncthreads();
    return r;
}

// Stable scatter of the flat entries [f0, f1) in flat order by one warp.
// cnt[e] holds the next free position of expert e and is advanced.
__device__ __forceinline__ void warp_stable_scatter(const int32_t *idx, int64_t f0, int64_t f1,
                                                    int E, int *cnt, int32_t *perm, int32_t *inv,
                                                    int *status) {
    int lane = threadIdx.x & 31;
    for (int64_t base = f0; base < f1; base += 32) {
        int64_t f = base + lane;
        bool valid = f < f1;
        int e = valid ? idx[f] : -1;
        if (valid && (e < 0 || e >= E)) { moe_flag(status, MOE_ERR_BAD_INDEX); e = -1; }
        uint32_t m = __match_any_sync(FULL_MASK, e);
        if (e >= 0) {
            int rank = __popc(m & lanemask_lt());
            int pos = cnt[e] + rank;
            perm[pos] = (int32_t)f;
            inv[f] = pos;
        }
        __syncwarp();
        if (e >= 0 && lane == 31 - __clz(m)) cnt[e] += __popc(m);
        __syncwarp();
    }
}

}  // namespace

// ---------------------------------------------------------------------------
// Small batches: one CTA does top-k, histogram, scan and the stable scatter.
// 512 threads (16 warps), one warp per token (warp_topk). (A 1024-thread
// block would cap a thread at 64 registers and push the keys to local
// memory.) The scans take two experts per thread.
// ---------------------------------------------------------------------------
constexpr int kPlanSmallThreads = 512;
constexpr int kPlanSmallWarps = kPlanSmallThreads / 32;

__global__ void __launch_bounds__(kPlanSmallThreads) moe_plan_small_kernel(
    int T, int E, int k, const float *__restrict__ logits, int32_t *topk_idx, float *topk_w,
    int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *active, int *status) {
    // T <= 64 tokens, k <= 32: the selections stay in shared memory, and each
    // expert keeps a bit mask of the tokens that chose it. A token chooses an
    // expert at most once, so the stable position of flat entry t*k+j (expert
    // e) is offsets[e] + the number of tokens before t that chose e.
    __shared__ int s_cnt[MOE_MAX_EXPERTS];
    __shared__ unsigned long long s_mask[MOE_MAX_EXPERTS];
    __shared__ int s_idx[64 * MOE_MAX_TOPK];
    __shared__ uint2 s_scr[kPlanSmallWarps][64];  // each warp's top-k scratch
    __shared__ int s_tot[33];
    __shared__ int s_nan;
    static_assert(2 * kPlanSmallThreads == MOE_MAX_EXPERTS, "two experts per thread in the scans");
    int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    grid_dep_wait();    // the logits may come from the previous kernel
    grid_dep_launch();
    for (int e = tid; e < MOE_MAX_EXPERTS; e += kPlanSmallThreads) {
        s_cnt[e] = 0;
        s_mask[e] = 0ull;
    }
    if (tid == 0) s_nan = 0;
    __syncthreads();
    bool nan_seen = false;
    for (int t = wid; t < T; t += kPlanSmallWarps) {
        int my_e;
        float my_v;
        warp_topk<true>(logits + (int64_t)t * E, E, k, lane, my_e, my_v, nan_seen, s_scr[wid]);
        const float w = warp_select_weight(my_v, k, lane);
        if (lane < k) {
            topk_idx[(int64_t)t * k + lane] = my_e;
            topk_w[(int64_t)t * k + lane] = w;
            s_idx[t * k + lane] = my_e;
            atomicAdd(&s_cnt[my_e], 1);
            atomicOr(&s_mask[my_e], 1ull << t);
        }
    }
    if (__any_sync(FULL_MASK, nan_seen) && lane == 0) s_nan = 1;
    __syncthreads();
    if (tid == 0 && s_nan) moe_flag(status, MOE_ERR_NAN_LOGIT);
    // experts e0 = 2 tid and e0 + 1 (counts are zero past E)
    const int e0 = 2 * tid;
    const int c0 = e0 < E ? s_cnt[e0] : 0, c1 = e0 + 1 < E ? s_cnt[e0 + 1] : 0;
    int total;
    const int off = block_exclusive_scan<kPlanSmallWarps>(c0 + c1, s_tot, total);
    const int a0 = c0 > 0 ? 1 : 0, a1 = c1 > 0 ? 1 : 0;
    const int a = block_exclusive_scan<kPlanSmallWarps>(a0 + a1, s_tot, total);
    if (e0 < E) {
        counts[e0] = c0;
        offsets[e0] = off;
        if (a0) active[1 + a] = e0;
    }
    if (e0 + 1 < E) {
        counts[e0 + 1] = c1;
        offsets[e0 + 1] = off + c0;
        if (a1) active[1 + a + a0] = e0 + 1;
    }
    if (tid == 0) {
        offsets[E] = T * k;
        active[0] = total;
    }
    __syncthreads();
    if (e0 < E) s_cnt[e0] = off;
    if (e0 + 1 < E) s_cnt[e0 + 1] = off + c0;
    __syncthreads();
    for (int f = tid; f < T * k; f += kPlanSmallThreads) {
        const int t = f / k, e = s_idx[f];
        const int pos = s_cnt[e] + __popcll(s_mask[e] & ((1ull << t) - 1ull));
        perm[pos] = f;
        inv[f] = pos;
    }
}

// ---------------------------------------------------------------------------
// Large batches: four kernels.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_topk_kernel(int T, int E, int k,
                                                       const float *__restrict__ logits,
                                                       int32_t *topk_idx, float *topk_w,
                                                       int *status) {
    __shared__ uint2 s_scratch[8][MOE_MAX_TOPK];
    int lane = threadIdx.x & 31;
    int t = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (t >= T) return;
    int my_e;
    float my_v;
    bool nan_seen = false;
    warp_topk<false>(logits + (int64_t)t * E, E, k, lane, my_e, my_v, nan_seen,
                     s_scratch[threadIdx.x >> 5]);
    float w = warp_select_weight(my_v, k, lane);
    if (lane < k) {
        topk_idx[(int64_t)t * k + lane] = my_e;
        topk_w[(int64_t)t * k + lane] = w;
    }
    if (__any_sync(FULL_MASK, nan_seen) && lane == 0) moe_flag(status, MOE_ERR_NAN_LOGIT);
}

// chunk_counts[c][e]: rows of expert e among tokens [c*CH, (c+1)*CH).
__global__ void __launch_bounds__(256) moe_plan_count_kernel(int T, int E, int k, int CH,
                                                             const int32_t *__restrict__ idx,
                                                             int32_t *chunk_counts, int *status) {
    extern __shared__ int s_hist[];  // 8 warps x E
    int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int c = blockIdx.x * 8 + wid;
    int nchunks = (T + CH - 1) / CH;
    int *h = s_hist + wid * E;
    for (int e = lane; e < E; e += 32) h[e] = 0;
    __syncwarp();
    if (c < nchunks) {
        int64_t f0 = (int64_t)c * CH * k;
        int64_t f1 = min((int64_t)(c + 1) * CH, (int64_t)T) * k;
        for (int64_t f = f0 + lane; f < f1; f += 32) {
            int e = idx[f];
            if (e >= 0 && e < E) atomicAdd(&h[e], 1);
            else moe_flag(status, MOE_ERR_BAD_INDEX);
        }
        __syncwarp();
        for (int e = lane; e < E; e += 32) chunk_counts[(int64_t)c * E + e] = h[e];
    }
}

// Column scan of chunk_counts (in place -> chunk bases), counts, offsets, active.
__global__ void __launch_bounds__(1024) moe_plan_scan_kernel(int T, int E, int k, int nchunks,
                                                             int32_t *chunk_counts,
                                                             int32_t *counts, int32_t *offsets,
                                                             int32_t *active) {
    __shared__ int s_tot[33];
    int e = threadIdx.x;
    int run = 0;
    if (e < E) {
        for (int c = 0; c < nchunks; ++c) {
            int v = chunk_counts[(int64_t)c * E + e];
            chunk_counts[(int64_t)c * E + e] = run;
            run += v;
        }
    }
    int total;
    int off = block_exclusive_scan<32>(run, s_tot, total);
    int a = block_exclusive_scan<32>(run > 0 ? 1 : 0, s_tot, total);
    if (e < E) {
        counts[e] = run;
        offsets[e] = off;
        if (run > 0) active[1 + a] = e;
    }
    if (e == 0) {
        offsets[E] = T * k;
        active[0] = total;
    }
}

__global__ void __launch_bounds__(256) moe_plan_scatter_kernel(int T, int E, int k, int CH,
                                                               const int32_t *__restrict__ idx,
                                                               const int32_t *chunk_base,
                                                               const int32_t *offsets,
                                                               int32_t *perm, int32_t *inv,
                                                               int *status) {
    extern __shared__ int s_next[];  // 8 warps x E
    int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int c = blockIdx.x * 8 + wid;
    int nchunks = (T + CH - 1) / CH;
    if (c >= nchunks) return;
    int *nx = s_next + wid * E;
    for (int e = lane; e < E; e += 32) nx[e] = offsets[e] + chunk_base[(int64_t)c * E + e];
    __syncwarp();
    int64_t f0 = (int64_t)c * CH * k;
    int64_t f1 = min((int64_t)(c + 1) * CH, (int64_t)T) * k;
    warp_stable_scatter(idx, f0, f1, E, nx, perm, inv, status);
}

// ---------------------------------------------------------------------------
// Host launchers.
// ---------------------------------------------------------------------------
size_t moe_plan_ws_bytes(int T, int E) {
    if (T <= 0 || moe_plan_is_small(T)) return 0;
    int nchunks = (T + MOE_PLAN_CHUNK - 1) / MOE_PLAN_CHUNK;
    return (size_t)nchunks * E * sizeof(int32_t);
}

cudaError_t moe_launch_plan(int T, int E, int k, const float *logits, const moe_plan_buf *p,
                            void *ws, int *status, cudaStream_t st) {
    if (moe_plan_is_small(T)) {
        return launch_pdl(moe_plan_small_kernel, dim3(1), dim3(kPlanSmallThreads), 0, st,
                          T, E, k, logits, p->topk_idx, p->topk_w, p->counts, p->offsets, p->perm,
                          p->inv, p->active, status);
    }
    int CH = MOE_PLAN_CHUNK;
    int nchunks = (T + CH - 1) / CH;
    int32_t *chunk = (int32_t *)ws;
    moe_topk_kernel<<<(T + 7) / 8, 256, 0, st>>>(T, E, k, logits, p->topk_idx, p->topk_w, status);
    size_t sm = (size_t)8 * E * sizeof(int);
    moe_plan_count_kernel<<<(nchunks + 7) / 8, 256, sm, st>>>(T, E, k, CH, p->topk_idx, chunk,
                                                              status);
    moe_plan_scan_kernel<<<1, 1024, 0, st>>>(T, E, k, nchunks, chunk, p->counts, p->offsets,
                                             p->active);
    moe_plan_scatter_kernel<<<(nchunks + 7) / 8, 256, sm, st>>>(T, E, k, CH, p->topk_idx, chunk,
                                                                p->offsets, p->perm, p->inv,
                                                                status);
    return cudaGetLastError();
}
