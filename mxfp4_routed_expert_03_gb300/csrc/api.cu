// C ABI of the routed-expert FFN library: argument validation, workspace
// carving and kernel launches. See include/moe.h for the contract.
#include <stdlib.h>
#include <string.h>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "kernels.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

// NVTX range over one entry point (host side; shows each call in profiler
// timelines, does nothing when no profiling tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

struct moe_handle {
    moe_desc desc;
    moe_weights w;
    int device;
    int num_sms;
    int *status;  // device word: first error code recorded by a kernel
    CUtensorMap map_gate, map_up, map_down;  // TMA views of the packed E2M1 weights
    CUtensorMap map4_gate, map4_up, map4_down;  // the same bytes unexpanded (FP4 x FP4 mode)
    CUtensorMap map16_gate, map16_up, map16_down;  // FP8 layers: the bf16 copy (after prepare)
    bool fp8;              // weight_format MOE_W_FP8
    CUtensorMap map_sh_gate, map_sh_up, map_sh_down;  // bf16 shared expert (has_shared)
    CUtensorMap map_wr[3];  // the three bf16 terms of W_r (router_mode XWR, after prepare)
    const uint8_t *atoms;  // caller buffer filled by moe_prepare (NULL until then)
    bool wr_ready;         // W_r terms written by moe_prepare
    MoeProf prof;          // optional timing events (moe_profile_kernel)
    int wE;                // experts held by the weight arrays w.* (n_slots when streaming)
    bool streaming;        // expert streaming: w.* are the slot cache, host_w the store
    moe_weights host_w;    // streaming: all experts, host memory the device can read
    void *sstate;          // streaming: device cache state (moe_stream_state_bytes)
    bool from_store;       // streaming from a compressed store (store) instead of host_w
    moe_store store;
    long long timeout;     // limit of every device-side wait (SM clock cycles)
    int inject;            // enum moe_inject (test hook; MOE_INJECT_NONE by default)
};

// Device-side waits give up after this many SM clocks (about one second).
static const long long kTimeoutCycles = 2000000000LL;

// cuTensorMapEncodeTiled, looked up through the runtime so the library does
// not link the driver library directly (it must load on hosts without a GPU).
typedef CUresult (*encode_tiled_fn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                    const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                    const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static encode_tiled_fn encode_tiled() {
    static encode_tiled_fn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (encode_tiled_fn)p;
    }
    return fn;
}

// 2D tensor map over a row-major byte matrix [rows][cols(elements)].
static bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t cols,
                        uint64_t rows, uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows) {
    encode_tiled_fn enc = encode_tiled();
    if (!enc) return false;
    cuuint64_t gd[2] = {cols, rows};
    cuuint64_t gs[1] = {row_bytes};
    cuuint32_t bd[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void *>(base), gd, gs, bd, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Workspace of moe_forward, carved in this order (each region 1 KB aligned):
// per-token two-term E4M3 activations and scales, the same rows laid out as
// the gate/up GEMM's B tiles (one block of 2 * NTMAX rows x 128 bytes per
// token tile and 128-wide K chunk; only the rows a tile uses are written),
// their scale blocks, h as the down GEMM's B tiles and its scale blocks, the
// fp32 output accumulator and the token-tile schedule.
struct FwdLayout {
    size_t xq_hi, xq_lo, xs_hi, xs_lo, xb, xa, hb, ha, acc, prefix, hsh, sk_part, sk_count, y, total;
    int max_tt;
};

// Whether moe_forward's larger batches keep every routed row's output and
// combine them (the FP4 x FP4 mode) instead of adding into an accumulator.
static bool row_out_mode(const moe_handle *h) {
    return h->desc.act_mode == MOE_ACT_MXFP4 && !h->fp8;
}

// Rows kept in bf16 (half the bytes for the down GEMM to write and the
// combine to read) while the experts average at most one wide token tile;
// beyond that each weight tile meets several token tiles, the down GEMM is
// bound by its epilogue, and fp32 rows stored straight from the lanes cost
// it less than the bf16 rows' shared-memory staging (measured: prefill4k,
// 73 rows per expert, 3.32 -> 3.07 ms per step with bf16; router16k, 292
// rows, 10.36 ms with fp32 against 10.61).
static bool row_out_bf16(int T, int k, int E) {
    return (int64_t)T * k <= (int64_t)E * MOE_GEMM_NTMAX;
}

// kdiv: K elements per activation-tile block (128; 64 for the bf16 tiles of
// FP8 layers); n_ctas: the grouped GEMMs' grid; row_out: larger batches keep
// every routed row's output (the FP4 x FP4 mode).
static FwdLayout fwd_layout(int T, int D, int F, int E, int k, bool shared, int n_ctas,
                            bool row_out, int kdiv = 128) {
    FwdLayout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += (bytes + 1023) / 1024 * 1024;
        return o;
    };
    const size_t rows = (size_t)T * k;
    // each active expert contributes ceil(count / NTMAX) <= count / NTMAX + 1 tiles
    L.max_tt = (int)(E + (rows + MOE_GEMM_NTMAX - 1) / MOE_GEMM_NTMAX);
    L.xq_hi = take((size_t)T * D);
    L.xq_lo = take((size_t)T * D);
    L.xs_hi = take((size_t)T * D / 32);
    L.xs_lo = take((size_t)T * D / 32);
    L.xb = take((size_t)L.max_tt * (D / kdiv) * MOE_GEMM_BTILE);
    L.xa = take((size_t)L.max_tt * (D / 128) * 1024);
    L.hb = take((size_t)L.max_tt * (F / kdiv) * MOE_GEMM_BTILE);
    L.ha = take((size_t)L.max_tt * (F / 128) * 1024);
    L.acc = take((size_t)T * D * sizeof(float));
    L.prefix = take((size_t)(E + 1) * sizeof(int32_t));
    L.hsh = take(shared ? (size_t)T * F * 2 : 0);  // shared expert's bf16 h [T][F]
    // small batches (narrow GEMMs): split gate/up tiles meet in 2 slots of
    // 16 x 128 fp32 per CTA; one arrival counter per gate/up weight tile
    const bool small = T <= MOE_GEMM_NT_NARROW;
    L.sk_part = take(small ? (size_t)n_ctas * 2 * 16 * 128 * sizeof(float) : 0);
    L.sk_count = take(small ? std::min(rows, (size_t)E) * (F / 64) * sizeof(int) : 0);
    // larger batches in the FP4 x FP4 mode: every routed row's down-projection
    // output [T k][D] in perm order (bf16 or fp32), for the deterministic combine
    L.y = take(!small && row_out ? rows * D * (row_out_bf16(T, k, E) ? 2 : 4) : 0);
    L.total = off;
    return L;
}

// TMA view of a row-major bf16 matrix [rows][cols]: boxes of 64 columns
// (one 128-byte swizzled row) x box_rows rows.
static bool make_map_bf16(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                          uint32_t box_rows) {
    return make_map_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, cols, rows, cols * 2, 64,
                       box_rows);
}

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// prepared weight scales of the wE experts in the weight arrays: gate/up
// tiles (64 + 64 rows), then down tiles (128 rows)
static size_t gu_atoms_bytes(const moe_desc &d, int wE) {
    return moe_prepared_atoms_bytes(wE, d.d_ff, d.d_model, 64);
}

// Bytes of one bf16 copy of an FP8 layer's matrix array (E x d_model x d_ff).
static size_t bf16_array_bytes(const moe_desc &d) {
    return align_up((size_t)d.n_experts * d.d_model * d.d_ff * 2, 256);
}

// The front of the prepared buffer: MXFP4 layers' re-laid weight scales, or
// FP8 layers' bf16 copies of gate, up and down.
static size_t atoms_bytes(const moe_desc &d, int wE) {
    if (d.weight_format == MOE_W_FP8) return 3 * bf16_array_bytes(d);
    return align_up(gu_atoms_bytes(d, wE) + moe_prepared_atoms_bytes(wE, d.d_model, d.d_ff, 128), 256);
}

MOE_API int64_t moe_expert_bytes(int32_t d_model, int32_t d_ff) {
    if (d_model <= 0 || d_ff <= 0 || d_model % 32 || d_ff % 32) return -1;
    int64_t n = (int64_t)d_model * d_ff;
    return 3 * (n / 2 + n / 32);
}

MOE_API const char *moe_strerror(int code) {
    switch (code) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape or device";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
        case MOE_ERR_NAN_LOGIT: return "NaN router logit";
        case MOE_ERR_BAD_INDEX: return "out-of-range index in plan";
        case MOE_ERR_NOT_PREPARED: return "moe_prepare has not been called on this handle";
        case MOE_ERR_CORRUPT_TILE: return "a compressed-store tile failed its checks";
        default: return "unknown status code";
    }
}

// moe_create for weight arrays holding wE experts (wE = n_experts, or the
// slot count of a streaming layer).
static int create_impl(const moe_desc *d, const moe_weights *w, int wE, moe_handle **out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = NULL;
    if (!d || !w) return MOE_ERR_INVALID_ARG;
    if (d->d_model <= 0 || d->d_ff <= 0 || d->n_experts <= 0 || d->top_k <= 0)
        return MOE_ERR_INVALID_ARG;
    if (d->router_mode != MOE_ROUTER_LOGITS && d->router_mode != MOE_ROUTER_XWR)
        return MOE_ERR_INVALID_ARG;
    if (d->has_shared != 0 && d->has_shared != 1) return MOE_ERR_INVALID_ARG;
    if (d->act_mode != MOE_ACT_EXACT && d->act_mode != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
    if (d->weight_format != MOE_W_MXFP4 && d->weight_format != MOE_W_FP8) return MOE_ERR_INVALID_ARG;
    const bool fp8 = d->weight_format == MOE_W_FP8;
    if (fp8 && d->act_mode != MOE_ACT_EXACT) return MOE_ERR_UNSUPPORTED;
    if (d->top_k > d->n_experts) return MOE_ERR_INVALID_ARG;
    if (d->d_model % 256 || d->d_ff % 128 || d->d_model > MOE_MAX_DMODEL ||
        d->d_ff > MOE_MAX_DFF || d->top_k > MOE_MAX_TOPK || d->n_experts > MOE_MAX_EXPERTS)
        return MOE_ERR_UNSUPPORTED;
    if (moe_decode_per_lane(d->d_model) == 0 || moe_decode_per_lane(d->d_ff) == 0)
        return MOE_ERR_UNSUPPORTED;
    const void *req[] = {w->gate_q, w->gate_s, w->up_q, w->up_s, w->down_q, w->down_s};
    for (const void *p : req)
        if (!p) return MOE_ERR_INVALID_ARG;
    if (((uintptr_t)w->gate_q | (uintptr_t)w->up_q | (uintptr_t)w->down_q) & (fp8 ? 15u : 31u))
        return MOE_ERR_INVALID_ARG;  // TMA of packed E2M1: 32-byte aligned; FP8 16-byte loads
    if (((uintptr_t)w->gate_s | (uintptr_t)w->up_s | (uintptr_t)w->down_s) & (fp8 ? 3u : 15u))
        return MOE_ERR_INVALID_ARG;  // bulk copies of scale rows: 16-byte aligned; FP8 fp32
    if (d->router_mode == MOE_ROUTER_XWR && !w->w_router) return MOE_ERR_INVALID_ARG;
    if (d->has_shared && (!w->sh_gate || !w->sh_up || !w->sh_down)) return MOE_ERR_INVALID_ARG;
    if (d->has_shared && ((uintptr_t)w->sh_gate | (uintptr_t)w->sh_up | (uintptr_t)w->sh_down) & 15u)
        return MOE_ERR_INVALID_ARG;  // TMA bases must be 16-byte aligned
    if (d->router_mode == MOE_ROUTER_XWR && ((uintptr_t)w->w_router & 3u)) return MOE_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (major != 10 || minor != 3) return MOE_ERR_UNSUPPORTED;

    moe_handle *h = (moe_handle *)calloc(1, sizeof(moe_handle));
    if (!h) return MOE_ERR_INVALID_ARG;
    h->desc = *d;
    h->w = *w;
    h->wE = wE;
    h->device = dev;
    h->timeout = kTimeoutCycles;
    h->inject = MOE_INJECT_NONE;
    h->fp8 = fp8;
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        free(h);
        return MOE_ERR_CUDA;
    }
    if (!fp8) {  // (FP8 layers get the maps of their bf16 copy in moe_prepare)
        const uint64_t D = d->d_model, F = d->d_ff, E = wE;  // experts in the weight arrays
        const CUtensorMapDataType fp4 = CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B;
        if (!make_map_2d(&h->map_gate, fp4, w->gate_q, D, E * F, D / 2, 128, 64) ||
            !make_map_2d(&h->map_up, fp4, w->up_q, D, E * F, D / 2, 128, 64) ||
            !make_map_2d(&h->map_down, fp4, w->down_q, F, E * D, F / 2, 128, 128)) {
            free(h);
            return MOE_ERR_CUDA;
        }
        // FP4 x FP4 mode: 128-byte boxes (two 128-wide K blocks) of packed codes
        const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        if (d->act_mode == MOE_ACT_MXFP4 &&
            (!make_map_2d(&h->map4_gate, u8, w->gate_q, D / 2, E * F, D / 2, 128, 64) ||
             !make_map_2d(&h->map4_up, u8, w->up_q, D / 2, E * F, D / 2, 128, 64) ||
             !make_map_2d(&h->map4_down, u8, w->down_q, F / 2, E * D, F / 2, 128, 128))) {
            free(h);
            return MOE_ERR_CUDA;
        }
    }
    {
        const uint64_t D = d->d_model, F = d->d_ff;
        if (d->has_shared &&
            (!make_map_bf16(&h->map_sh_gate, w->sh_gate, D, F, 64) ||
             !make_map_bf16(&h->map_sh_up, w->sh_up, D, F, 64) ||
             !make_map_bf16(&h->map_sh_down, w->sh_down, F, D, 128))) {
            free(h);
            return MOE_ERR_CUDA;
        }
    }
    if (cudaMalloc(&h->status, sizeof(int)) != cudaSuccess) {
        free(h);
        return MOE_ERR_CUDA;
    }
    if (cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(h->status);
        free(h);
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

MOE_API int moe_create(const moe_desc *d, const moe_weights *w, moe_handle **out) {
    return create_impl(d, w, d ? d->n_experts : 0, out);
}

// Host memory the device reads through the same address (pinned and mapped).
static bool device_readable_host(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

MOE_API size_t moe_stream_state_bytes(int32_t n_experts, int32_t n_slots) {
    if (n_experts <= 0 || n_slots <= 0 || n_experts > MOE_MAX_EXPERTS || n_slots > 1024) return 0;
    return moe_stream_state_size(n_experts, n_slots);
}

MOE_API int moe_create_streaming(const moe_desc *d, const moe_weights *host_w,
                                 const moe_weights *slot_w, int32_t n_slots, void *state,
                                 moe_handle **out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = NULL;
    if (!d || !host_w || !slot_w || !state) return MOE_ERR_INVALID_ARG;
    if (d->n_experts <= 0 || n_slots < 1 || n_slots > d->n_experts || n_slots > 1024)
        return MOE_ERR_INVALID_ARG;
    if (d->weight_format != MOE_W_MXFP4) return MOE_ERR_UNSUPPORTED;
    const void *hp[] = {host_w->gate_q, host_w->gate_s, host_w->up_q,
                        host_w->up_s, host_w->down_q, host_w->down_s};
    for (const void *p : hp) {
        // the copy kernel reads these through the same addresses: require
        // registered (pinned) host memory mapped at the host address
        if (!p || !aligned16(p) || !device_readable_host(p)) return MOE_ERR_INVALID_ARG;
    }
    if ((uintptr_t)state & 15u) return MOE_ERR_INVALID_ARG;
    moe_handle *h = nullptr;
    int rc = create_impl(d, slot_w, n_slots, &h);
    if (rc != MOE_OK) return rc;
    h->streaming = true;
    h->host_w = *host_w;
    h->sstate = state;
    if (moe_launch_stream_init(d->n_experts, n_slots, state, 0) != cudaSuccess ||
        cudaStreamSynchronize(0) != cudaSuccess) {
        cudaFree(h->status);
        free(h);
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

MOE_API int moe_create_streaming_store(const moe_desc *d, const moe_store *store,
                                       const moe_weights *slot_w, int32_t n_slots, void *state,
                                       moe_handle **out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = NULL;
    if (!d || !store || !slot_w || !state) return MOE_ERR_INVALID_ARG;
    if (d->n_experts <= 0 || n_slots < 1 || n_slots > d->n_experts || n_slots > 1024)
        return MOE_ERR_INVALID_ARG;
    if (d->weight_format != MOE_W_MXFP4) return MOE_ERR_UNSUPPORTED;
    MoeStoreJob probe;
    if (!moe_store_job_shape(d->d_model, d->d_ff, probe)) return MOE_ERR_INVALID_ARG;
    if (!store->blob || !aligned16(store->blob) || store->blob_bytes <= 0 || !store->tiles ||
        !aligned16(store->tiles) || !store->tables || !aligned16(store->tables) ||
        !device_readable_host(store->blob))
        return MOE_ERR_INVALID_ARG;
    if ((uintptr_t)state & 15u) return MOE_ERR_INVALID_ARG;
    moe_handle *h = nullptr;
    int rc = create_impl(d, slot_w, n_slots, &h);
    if (rc != MOE_OK) return rc;
    h->streaming = true;
    h->from_store = true;
    h->store = *store;
    h->sstate = state;
    if (moe_launch_stream_init(d->n_experts, n_slots, state, 0) != cudaSuccess ||
        cudaStreamSynchronize(0) != cudaSuccess) {
        cudaFree(h->status);
        free(h);
        return MOE_ERR_CUDA;
    }
    *out = h;
    return MOE_OK;
}

// Fills a decode job's store and slot fields.
static void store_job(MoeStoreJob &j, const moe_store &s, int E, const moe_weights &dst,
                      int n_slots, int *status) {
    j.blob = s.blob;
    j.blob_bytes = s.blob_bytes;
    j.tiles = s.tiles;
    j.tables = s.tables;
    j.E = E;
    j.n_slots = n_slots;
    const uint8_t *d6[6] = {dst.gate_q, dst.gate_s, dst.up_q, dst.up_s, dst.down_q, dst.down_s};
    for (int a = 0; a < 6; ++a) j.dst[a] = const_cast<uint8_t *>(d6[a]);
    j.status = status;
}

MOE_API int moe_store_decode(int32_t n_experts, int32_t d_model, int32_t d_ff,
                             const moe_store *store, const int32_t *experts, const int32_t *slots,
                             int32_t n, const moe_weights *slot_w, int32_t n_slots, int32_t *status,
                             void *stream) {
    NvtxRange nvtx_range("moe_store_decode");
    MoeStoreJob j;
    if (n_experts <= 0 || n_experts > MOE_MAX_EXPERTS || n < 0 || n_slots < 1 || !store ||
        !slot_w || !status || !moe_store_job_shape(d_model, d_ff, j))
        return MOE_ERR_INVALID_ARG;
    if (n == 0) return MOE_OK;
    if (!experts || !slots || !store->blob || !aligned16(store->blob) || store->blob_bytes <= 0 ||
        !store->tiles || !aligned16(store->tiles) || !store->tables || !aligned16(store->tables))
        return MOE_ERR_INVALID_ARG;
    const uint8_t *d6[6] = {slot_w->gate_q, slot_w->gate_s, slot_w->up_q,
                            slot_w->up_s, slot_w->down_q, slot_w->down_s};
    for (const uint8_t *p : d6)
        if (!p) return MOE_ERR_INVALID_ARG;
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    store_job(j, *store, n_experts, *slot_w, n_slots, status);
    j.experts = experts;
    j.slots = slots;
    j.n_dev = nullptr;
    j.n_host = n;
    j.max_items = n;
    return moe_launch_store_decode(j, nsm, (cudaStream_t)stream) == cudaSuccess ? MOE_OK
                                                                                : MOE_ERR_CUDA;
}

MOE_API int moe_stream_stats(moe_handle *h, int64_t *hits, int64_t *misses, int32_t *last_misses,
                             void *stream) {
    if (!h || !h->streaming) return MOE_ERR_INVALID_ARG;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MOE_ERR_CUDA;
    MoeStreamHdr hdr;
    if (cudaMemcpy(&hdr, h->sstate, sizeof(hdr), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (hits) *hits = (int64_t)hdr.hits;
    if (misses) *misses = (int64_t)hdr.misses;
    if (last_misses) *last_misses = hdr.last_miss;
    return MOE_OK;
}

// Expert streaming: make every active expert of the plan resident (device-side
// replacement, copies of the misses from host memory, their scale blocks).
static cudaError_t stream_fill(moe_handle *h, const moe_plan_buf *plan, cudaStream_t st) {
    const moe_desc &d = h->desc;
    const int E = d.n_experts, S = h->wE, D = d.d_model, F = d.d_ff;
    cudaError_t err = moe_launch_stream_lru(E, S, plan->active, h->sstate, h->status, st);
    MoeStreamCopy c;
    const moe_weights &hw = h->host_w, &sw = h->w;
    const uint8_t *hs[6] = {hw.gate_q, hw.gate_s, hw.up_q, hw.up_s, hw.down_q, hw.down_s};
    const uint8_t *ss[6] = {sw.gate_q, sw.gate_s, sw.up_q, sw.up_s, sw.down_q, sw.down_s};
    const int64_t n = (int64_t)D * F;
    const int64_t by[6] = {n / 2, n / 32, n / 2, n / 32, n / 2, n / 32};
    for (int i = 0; i < 6; ++i) {
        c.host[i] = hs[i];
        c.slot[i] = const_cast<uint8_t *>(ss[i]);
        c.bytes[i] = by[i];
    }
    const MoeStreamView v = moe_stream_view(h->sstate, E, S);
    if (err == cudaSuccess) {
        h->prof.before(MOE_PROF_STREAM_COPY, st);
        if (h->from_store) {  // decode the misses from the compressed store
            MoeStoreJob j;
            moe_store_job_shape(D, F, j);
            store_job(j, h->store, E, sw, S, h->status);
            j.experts = v.miss_e;
            j.slots = v.miss_s;
            j.n_dev = &v.hdr->last_miss;
            j.n_host = 0;
            j.max_items = S;
            err = moe_launch_store_decode(j, h->num_sms, st);
        } else {
            err = moe_launch_stream_copy(E, S, h->sstate, &c, h->num_sms, st);
        }
        h->prof.after(MOE_PROF_STREAM_COPY, st);
    }
    uint8_t *atoms = const_cast<uint8_t *>(h->atoms);
    if (err == cudaSuccess)
        err = moe_launch_prepare_atoms_slots(F, D, 64, sw.gate_s, sw.up_s, atoms, &v.hdr->last_miss,
                                             v.miss_s, h->num_sms, st);
    if (err == cudaSuccess)
        err = moe_launch_prepare_atoms_slots(D, F, 128, sw.down_s, nullptr,
                                             atoms + gu_atoms_bytes(d, S), &v.hdr->last_miss,
                                             v.miss_s, h->num_sms, st);
    return err;
}

MOE_API void moe_destroy(moe_handle *h) {
    if (!h) return;
    cudaFree(h->status);
    free(h);
}

// Router logits region at the front of moe_plan's workspace (router_mode XWR).
static size_t router_ws_bytes(const moe_handle *h, int T) {
    if (h->desc.router_mode != MOE_ROUTER_XWR) return 0;
    return align_up((size_t)T * h->desc.n_experts * sizeof(float), 256);
}

// Shared-expert regions at the end of moe_decode's workspace: bf16 h [T][F]
// and the fp32 shared output [T][D].
static size_t shared_ws_bytes(const moe_handle *h, int T) {
    if (!h->desc.has_shared) return 0;
    return align_up((size_t)T * h->desc.d_ff * 2, 256) +
           align_up((size_t)T * h->desc.d_model * sizeof(float), 256);
}

static int dense_grid(const moe_handle *h, int epi, int M, int N) {
    const int tiles = moe_dense_tiles(epi, M, N);
    return tiles < h->num_sms ? tiles : h->num_sms;
}

static MoeDenseArgs dense_args(const moe_handle *h, int M, int N, int K, int ldo) {
    MoeDenseArgs a;
    memset(&a, 0, sizeof(a));
    a.M = M;
    a.N = N;
    a.K = K;
    a.ldo = ldo;
    a.status = h->status;
    a.timeout_cycles = h->timeout;
    return a;
}

// logits[T][E] = x . W_r^T in fp32 on tensor cores (three bf16 terms of W_r).
static int run_router(moe_handle *h, int T, const uint16_t *x, float *logits, cudaStream_t st) {
    const moe_desc &d = h->desc;
    CUtensorMap mx;
    if (!make_map_bf16(&mx, x, d.d_model, T, MOE_DENSE_NTILE)) return MOE_ERR_CUDA;
    MoeDenseArgs a = dense_args(h, d.n_experts, T, d.d_model, d.n_experts);
    a.out_f32 = logits;
    h->prof.before(MOE_PROF_ROUTER, st);
    cudaError_t err = moe_launch_dense(MOE_DENSE_ROUTER, &h->map_wr[0], &h->map_wr[1],
                                       &h->map_wr[2], &mx, &a,
                                       dense_grid(h, MOE_DENSE_ROUTER, d.n_experts, T), st);
    h->prof.after(MOE_PROF_ROUTER, st);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// Shared expert: hsh = bf16(silu(x . Ws_gate^T) * (x . Ws_up^T)) [T][F], then
// out[T][D] = hsh . Ws_down^T in fp32 (written, not added).
static int run_shared(moe_handle *h, int T, const uint16_t *x, uint16_t *hsh, float *out,
                      cudaStream_t st) {
    const moe_desc &d = h->desc;
    const int D = d.d_model, F = d.d_ff;
    CUtensorMap mx, mh;
    if (!make_map_bf16(&mx, x, D, T, MOE_DENSE_NTILE) ||
        !make_map_bf16(&mh, hsh, F, T, MOE_DENSE_NTILE))
        return MOE_ERR_CUDA;
    MoeDenseArgs g = dense_args(h, F, T, D, F);
    g.out_bf16 = hsh;
    h->prof.before(MOE_PROF_SHARED_GATEUP, st);
    cudaError_t err = moe_launch_dense(MOE_DENSE_SWIGLU, &h->map_sh_gate, &h->map_sh_up,
                                       &h->map_sh_gate, &mx, &g,
                                       dense_grid(h, MOE_DENSE_SWIGLU, F, T), st);
    h->prof.after(MOE_PROF_SHARED_GATEUP, st);
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    MoeDenseArgs o = dense_args(h, D, T, F, D);
    o.out_f32 = out;
    h->prof.before(MOE_PROF_SHARED_DOWN, st);
    err = moe_launch_dense(MOE_DENSE_STORE, &h->map_sh_down, &h->map_sh_down, &h->map_sh_down, &mh,
                           &o, dense_grid(h, MOE_DENSE_STORE, D, T), st);
    h->prof.after(MOE_PROF_SHARED_DOWN, st);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

MOE_API size_t moe_workspace_bytes(const moe_handle *h, int32_t T, int32_t op) {
    if (!h || T <= 0) return 0;
    const moe_desc &d = h->desc;
    switch (op) {
        case MOE_OP_PLAN:
            return router_ws_bytes(h, T) + align_up(moe_plan_ws_bytes(T, d.n_experts), 256);
        case MOE_OP_DECODE:
            return align_up(moe_decode_ws_bytes(T, d.d_model, d.d_ff, d.top_k), 256) +
                   shared_ws_bytes(h, T);
        case MOE_OP_FORWARD:
            return fwd_layout(T, d.d_model, d.d_ff, d.n_experts, d.top_k, d.has_shared,
                              h->num_sms, row_out_mode(h), h->fp8 ? 64 : 128).total;
        default: return 0;
    }
}

static bool plan_ok(const moe_plan_buf *p) {
    return p && p->topk_idx && p->topk_w && p->counts && p->offsets && p->perm && p->inv &&
           p->active;
}

MOE_API int moe_plan(moe_handle *h, int32_t T, const float *logits, const uint16_t *x,
                     const moe_plan_buf *plan, void *ws, size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_plan");
    if (!h || T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!plan_ok(plan)) return MOE_ERR_INVALID_ARG;
    const bool xwr = h->desc.router_mode == MOE_ROUTER_XWR;
    if (!xwr && !logits) return MOE_ERR_INVALID_ARG;
    if (xwr && (logits || !x || !aligned16(x))) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * h->desc.top_k > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)T * h->desc.n_experts > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (xwr && !h->wr_ready) return MOE_ERR_NOT_PREPARED;
    size_t need = moe_workspace_bytes(h, T, MOE_OP_PLAN);
    if (ws_bytes < need || (need && !ws)) return MOE_ERR_WORKSPACE;
    if (need && ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t lg_bytes = router_ws_bytes(h, T);
    if (xwr) {
        float *lg = (float *)ws;
        int rc = run_router(h, T, x, lg, st);
        if (rc != MOE_OK) return rc;
        logits = lg;
    }
    void *pws = lg_bytes ? (void *)((unsigned char *)ws + lg_bytes) : ws;
    cudaError_t err = moe_launch_plan(T, h->desc.n_experts, h->desc.top_k, logits, plan, pws,
                                      h->status, st);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

MOE_API int moe_router_logits(moe_handle *h, int32_t T, const uint16_t *x, float *logits,
                              void *stream) {
    NvtxRange nvtx_range("moe_router_logits");
    if (!h || T < 0) return MOE_ERR_INVALID_ARG;
    if (h->desc.router_mode != MOE_ROUTER_XWR) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !logits || !aligned16(x) || ((uintptr_t)logits & 3u)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * h->desc.n_experts > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (!h->wr_ready) return MOE_ERR_NOT_PREPARED;
    return run_router(h, T, x, logits, (cudaStream_t)stream);
}

MOE_API int moe_decode(moe_handle *h, int32_t T, const uint16_t *x, const moe_plan_buf *plan,
                       uint16_t *out, void *ws, size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_decode");
    if (!h || T < 0) return MOE_ERR_INVALID_ARG;
    if (h->streaming) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !out || !plan_ok(plan)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * h->desc.top_k > INT32_MAX / 2 || T > 65535) return MOE_ERR_UNSUPPORTED;
    size_t need = moe_workspace_bytes(h, T, MOE_OP_DECODE);
    if (ws_bytes < need || !ws || !aligned16(ws)) return MOE_ERR_WORKSPACE;
    const moe_desc &d = h->desc;
    cudaStream_t st = (cudaStream_t)stream;
    float *sh_out = nullptr;
    if (d.has_shared) {
        unsigned char *p = (unsigned char *)ws +
                           align_up(moe_decode_ws_bytes(T, d.d_model, d.d_ff, d.top_k), 256);
        uint16_t *hsh = (uint16_t *)p;
        sh_out = (float *)(p + align_up((size_t)T * d.d_ff * 2, 256));
        int rc = run_shared(h, T, x, hsh, sh_out, st);
        if (rc != MOE_OK) return rc;
    }
    cudaError_t err = moe_launch_decode(T, d.d_model, d.d_ff, d.n_experts, d.top_k, x, plan, &h->w,
                                        h->fp8, sh_out, out, ws, h->status, h->prof, st);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

MOE_API int moe_decode_noalloc(moe_handle *h, int32_t T, const uint16_t *x,
                               const moe_plan_buf *plan, uint16_t *out, void *stream) {
    NvtxRange nvtx_range("moe_decode_noalloc");
    if (!h || T < 0) return MOE_ERR_INVALID_ARG;
    if (h->streaming) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!x || !out || !plan_ok(plan)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    const moe_desc &d = h->desc;
    if (d.has_shared) return MOE_ERR_UNSUPPORTED;  // the fixed scratch has no shared-expert room
    if ((int64_t)T * d.top_k > MOE_NOALLOC_MAX_ROWS || d.d_ff > MOE_NOALLOC_MAX_DFF ||
        d.d_model > MOE_NOALLOC_MAX_DMODEL ||
        moe_decode_ws_bytes(T, d.d_model, d.d_ff, d.top_k) > moe_noalloc_scratch_bytes())
        return MOE_ERR_WORKSPACE;  // beyond the fixed scratch
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev != h->device) return MOE_ERR_INVALID_ARG;
    void *scratch = nullptr;
    if (moe_noalloc_scratch(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t err = moe_launch_decode(T, d.d_model, d.d_ff, d.n_experts, d.top_k, x, plan, &h->w,
                                        h->fp8, nullptr, out, scratch, h->status, h->prof,
                                        (cudaStream_t)stream);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

MOE_API int moe_forward(moe_handle *h, int32_t T, const uint16_t *x, const moe_plan_buf *plan,
                        uint16_t *out, void *ws, size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("moe_forward");
    if (!h || T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !out || !plan_ok(plan)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * h->desc.top_k > INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!h->atoms) return MOE_ERR_NOT_PREPARED;
    const moe_desc &d = h->desc;
    // a streaming layer must be able to hold every expert a plan can select
    if (h->streaming && (int64_t)T * d.top_k > h->wE && d.n_experts > h->wE)
        return MOE_ERR_UNSUPPORTED;
    const FwdLayout L = fwd_layout(T, d.d_model, d.d_ff, d.n_experts, d.top_k, d.has_shared,
                                   h->num_sms, row_out_mode(h), h->fp8 ? 64 : 128);
    if (ws_bytes < L.total || !ws || ((uintptr_t)ws & 255u)) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    unsigned char *base = (unsigned char *)ws;
    const int D = d.d_model, F = d.d_ff, E = d.n_experts, k = d.top_k, rows = T * k;
    uint8_t *xq_hi = base + L.xq_hi, *xq_lo = base + L.xq_lo;
    uint8_t *xs_hi = base + L.xs_hi, *xs_lo = base + L.xs_lo;
    uint8_t *xb = base + L.xb, *xa = base + L.xa, *hb = base + L.hb, *ha = base + L.ha;
    float *acc = (float *)(base + L.acc);
    int32_t *prefix = (int32_t *)(base + L.prefix);
    float *sk_part = (float *)(base + L.sk_part);
    int *sk_count = (int *)(base + L.sk_count);
    void *y = base + L.y;
    const int n_sk = (int)(std::min((size_t)T * d.top_k, (size_t)d.n_experts) * (d.d_ff / 64));

    // Small batches (every expert one token tile): quantise, gather, schedule
    // and zero the accumulator in one launch; larger ones quantise each token
    // once, schedule the token tiles and gather them (and zero the
    // accumulator where it is used).
    const bool small = T <= MOE_GEMM_NT_NARROW;
    // The FP4 x FP4 mode's down GEMM is bound by its epilogue when it adds
    // into the fp32 accumulator (it issues half the MMAs of the two-term
    // path): there the rows go to y and a combine sums them. The two-term
    // path's down GEMM is bound by its MMA issue, so the reductions cost it
    // nothing and it keeps the accumulator (no extra traffic).
    const bool row_out = !small && row_out_mode(h);
    const bool fp4 = d.act_mode == MOE_ACT_MXFP4;
    cudaError_t err;
    if (h->fp8 && small) {
        err = moe_launch_prep_small_bf16(T, E, k, D, plan->offsets, plan->perm, plan->active, x,
                                         prefix, xb, d.has_shared ? nullptr : acc, sk_count, n_sk,
                                         h->status, st);
    } else if (h->fp8) {
        err = moe_launch_schedule(E, MOE_GEMM_NTMAX, plan->offsets, plan->active, prefix,
                                  h->status, st);
        if (err == cudaSuccess)
            err = moe_launch_gather_x_bf16(L.max_tt, E, k, rows, D, plan->offsets, plan->perm,
                                           plan->active, prefix, x, xb, h->status, st);
    } else if (small && fp4) {
        err = moe_launch_prep_small_fp4(T, E, k, D, plan->offsets, plan->perm, plan->active, x,
                                        prefix, xb, xa, d.has_shared ? nullptr : acc, sk_count,
                                        n_sk, h->status, st);
    } else if (small) {
        err = moe_launch_prep_small(T, E, k, D, plan->offsets, plan->perm, plan->active, x, prefix,
                                    xb, xa, d.has_shared ? nullptr : acc, sk_count, n_sk,
                                    h->status, st);
    } else if (fp4) {  // each token quantised once (into the two-term path's buffers)
        err = moe_launch_quant_x_fp4(T, D, x, xq_hi, xs_hi, st);
        if (err == cudaSuccess)
            err = moe_launch_schedule(E, MOE_GEMM_NTMAX, plan->offsets, plan->active, prefix,
                                      h->status, st);
        if (err == cudaSuccess)
            err = moe_launch_gather_x_fp4(L.max_tt, E, k, rows, D, plan->offsets, plan->perm,
                                          plan->active, prefix, xq_hi, xs_hi, xb, xa, h->status,
                                          st);
    } else {
        err = moe_launch_quant_x(T, D, x, xq_hi, xq_lo, xs_hi, xs_lo, st);
        if (err == cudaSuccess)
            err = moe_launch_schedule(E, MOE_GEMM_NTMAX, plan->offsets, plan->active, prefix,
                                      h->status, st);
        if (err == cudaSuccess)
            err = moe_launch_gather_x(L.max_tt, E, k, rows, D, MOE_GEMM_NTMAX, plan->offsets,
                                      plan->perm, plan->active, prefix, xq_hi, xq_lo, xs_hi,
                                      xs_lo, xb, xa, h->status, st);
    }
    MoeGemmArgs a;
    memset(&a, 0, sizeof(a));
    a.E = E;
    a.k = k;
    a.n_rows = rows;
    a.Dout = D;
    a.offsets = plan->offsets;
    a.perm = plan->perm;
    a.active = plan->active;
    a.tt_prefix = prefix;
    a.topk_w = plan->topk_w;
    a.status = h->status;
    a.timeout_cycles = h->timeout;
    a.inject = MOE_INJECT_NONE;
    if (small) {
        a.sk_part = sk_part;
        a.sk_count = sk_count;
    }
    if (h->streaming) {  // experts resident first; the GEMMs then address their slots
        if (err == cudaSuccess) err = stream_fill(h, plan, st);
        a.w_index = moe_stream_view(h->sstate, E, h->wE).slot_of;
        a.n_wexp = h->wE;
    }
    if (err == cudaSuccess) {
        MoeGemmArgs g1 = a;
        g1.M = F;
        g1.K = D;
        g1.KC = h->fp8 ? D / 64 : D / 128;
        g1.MT = F / 64;  // 64 gate rows + the same 64 up rows per weight tile
        g1.a_atoms = h->atoms;
        g1.b_tiles = xb;
        g1.b_atoms = xa;
        g1.h_tiles = hb;
        g1.h_atoms = ha;
        g1.inject = h->inject;
        h->prof.before(MOE_PROF_FORWARD_GEMM1, st);
        err = h->fp8 ? moe_launch_gemm(MOE_GEMM_GATEUP, &h->map16_gate, &h->map16_up, &g1, T,
                                       h->num_sms, MOE_AF_BF16, st)
              : fp4 ? moe_launch_gemm(MOE_GEMM_GATEUP, &h->map4_gate, &h->map4_up, &g1, T,
                                    h->num_sms, MOE_AF_MXF4, st)
                  : moe_launch_gemm(MOE_GEMM_GATEUP, &h->map_gate, &h->map_up, &g1, T,
                                    h->num_sms, MOE_AF_E4M3X2, st);
        h->prof.after(MOE_PROF_FORWARD_GEMM1, st);
    }
    if (err == cudaSuccess) {
        // the shared expert writes acc: the routed rows add onto it, or the
        // combine adds it last (row_out); without one, small batches zeroed
        // acc in their first launch and larger ones zero it here
        if (d.has_shared) {
            if (run_shared(h, T, x, (uint16_t *)(base + L.hsh), acc, st) != MOE_OK)
                err = cudaErrorLaunchFailure;
        } else if (!small && !row_out) {
            err = cudaMemsetAsync(acc, 0, (size_t)T * D * sizeof(float), st);
        }
    }
    if (err == cudaSuccess) {
        MoeGemmArgs g2 = a;
        g2.M = D;
        g2.MT = D / 128;
        g2.K = F;
        g2.KC = h->fp8 ? F / 64 : F / 128;
        g2.a_atoms = h->atoms + gu_atoms_bytes(d, h->wE);
        g2.b_tiles = hb;
        g2.b_atoms = ha;
        g2.acc = acc;
        if (row_out) {  // plain stores of each row; no accumulator reductions
            g2.y = y;
            g2.y_bf16 = row_out_bf16(T, k, E) ? 1 : 0;
        }
        h->prof.before(MOE_PROF_FORWARD_GEMM2, st);
        err = h->fp8 ? moe_launch_gemm(MOE_GEMM_DOWN, &h->map16_down, &h->map16_down, &g2, T,
                                       h->num_sms, MOE_AF_BF16, st)
              : fp4 ? moe_launch_gemm(MOE_GEMM_DOWN, &h->map4_down, &h->map4_down, &g2, T,
                                    h->num_sms, MOE_AF_MXF4, st)
                  : moe_launch_gemm(MOE_GEMM_DOWN, &h->map_down, &h->map_down, &g2, T,
                                    h->num_sms, MOE_AF_E4M3X2, st);
        h->prof.after(MOE_PROF_FORWARD_GEMM2, st);
    }
    if (err == cudaSuccess)
        err = !row_out ? moe_launch_finalize(T, D, acc, out, st)
                       : row_out_bf16(T, k, E)
                           ? moe_launch_combine_slots_bf16(T, D, k, rows, plan->topk_w, plan->inv,
                                                           (const uint16_t *)y,
                                                           d.has_shared ? acc : nullptr, out,
                                                           h->status, st)
                           : moe_launch_combine_slots(T, D, k, rows, plan->topk_w, plan->inv,
                                                      (const float *)y,
                                                      d.has_shared ? acc : nullptr, out,
                                                      h->status, st);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static size_t wr_terms_bytes(const moe_desc &d) {
    return d.router_mode == MOE_ROUTER_XWR
               ? align_up((size_t)d.n_experts * d.d_model * 2, 256) * 3
               : 0;
}

MOE_API size_t moe_prepared_bytes(const moe_handle *h) {
    if (!h) return 0;
    return atoms_bytes(h->desc, h->wE) + wr_terms_bytes(h->desc);
}

MOE_API int moe_prepare(moe_handle *h, void *buf, size_t bytes, void *stream) {
    NvtxRange nvtx_range("moe_prepare");
    if (!h || !buf) return MOE_ERR_INVALID_ARG;
    if (bytes < moe_prepared_bytes(h)) return MOE_ERR_WORKSPACE;
    if ((uintptr_t)buf & 255u) return MOE_ERR_INVALID_ARG;
    const moe_desc &d = h->desc;
    const int E = d.n_experts, D = d.d_model, F = d.d_ff;
    uint8_t *out = (uint8_t *)buf;
    cudaStream_t st = (cudaStream_t)stream;
    // gate/up tiles: 64 gate rows over the same 64 up rows; down tiles: 128 rows
    // (a streaming layer's slots are prepared as experts arrive)
    cudaError_t err = cudaSuccess;
    if (h->fp8) {
        // the bf16 copy the prefill GEMMs stream: gate, up [E][F][D], down [E][D][F]
        const size_t ab = bf16_array_bytes(d);
        uint16_t *g16 = (uint16_t *)out, *u16 = (uint16_t *)(out + ab),
                 *d16 = (uint16_t *)(out + 2 * ab);
        err = moe_launch_fp8_dequant(E, F, D, h->w.gate_q, (const float *)h->w.gate_s, g16, st);
        if (err == cudaSuccess)
            err = moe_launch_fp8_dequant(E, F, D, h->w.up_q, (const float *)h->w.up_s, u16, st);
        if (err == cudaSuccess)
            err = moe_launch_fp8_dequant(E, D, F, h->w.down_q, (const float *)h->w.down_s, d16, st);
        if (err == cudaSuccess &&
            (!make_map_2d(&h->map16_gate, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, g16, D,
                          (uint64_t)E * F, (uint64_t)D * 2, 64, 64) ||
             !make_map_2d(&h->map16_up, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u16, D,
                          (uint64_t)E * F, (uint64_t)D * 2, 64, 64) ||
             !make_map_2d(&h->map16_down, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d16, F,
                          (uint64_t)E * D, (uint64_t)F * 2, 64, 128)))
            return MOE_ERR_CUDA;
    } else if (!h->streaming) {
        err = moe_launch_prepare_atoms(E, F, D, 64, h->w.gate_s, h->w.up_s, out, st);
        if (err == cudaSuccess)
            err = moe_launch_prepare_atoms(E, D, F, 128, h->w.down_s, nullptr,
                                           out + gu_atoms_bytes(d, h->wE), st);
    }
    if (err != cudaSuccess) return MOE_ERR_CUDA;
    if (d.router_mode == MOE_ROUTER_XWR) {
        // W_r = t0 + t1 + t2 exactly, three bf16 [E][D] arrays after the scale atoms
        const size_t tb = wr_terms_bytes(d) / 3;
        uint16_t *t[3];
        for (int i = 0; i < 3; ++i) t[i] = (uint16_t *)(out + atoms_bytes(d, h->wE) + i * tb);
        if (moe_launch_split3((int64_t)E * D, h->w.w_router, t[0], t[1], t[2], st) != cudaSuccess)
            return MOE_ERR_CUDA;
        for (int i = 0; i < 3; ++i)
            if (!make_map_bf16(&h->map_wr[i], t[i], D, E, 128)) return MOE_ERR_CUDA;
        h->wr_ready = true;
    }
    h->atoms = out;
    return MOE_OK;
}

MOE_API int moe_profile_kernel(moe_handle *h, int32_t which, void *ev_start, void *ev_stop) {
    if (!h || which < MOE_PROF_NONE || which > MOE_PROF_STREAM_COPY) return MOE_ERR_INVALID_ARG;
    if (which != MOE_PROF_NONE && (!ev_start || !ev_stop)) return MOE_ERR_INVALID_ARG;
    h->prof.which = which;
    h->prof.start = (cudaEvent_t)ev_start;
    h->prof.stop = (cudaEvent_t)ev_stop;
    return MOE_OK;
}

MOE_API int moe_set_fault_injection(moe_handle *h, int32_t mode, int64_t timeout_cycles) {
    if (!h || (mode != MOE_INJECT_NONE && mode != MOE_INJECT_GEMM_STALL)) return MOE_ERR_INVALID_ARG;
    if (timeout_cycles > 0 && timeout_cycles < 100000) return MOE_ERR_INVALID_ARG;
    h->inject = mode;
    h->timeout = timeout_cycles > 0 ? (long long)timeout_cycles : kTimeoutCycles;
    return MOE_OK;
}

MOE_API int moe_status(moe_handle *h, void *stream) {
    if (!h) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, h->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (v != 0 && cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
    return v;
}
