/*
 * moe.h — C ABI of the routed-expert FFN library (libmoe.so), GB300 / sm_103a.
 *
 * The operation is one routed-MoE layer of a Kimi-K3-style model: every token
 * selects top_k of n_experts experts (16 of 896 in K3: MoonTail, intro;
 * Moonshine README, "How the engine works"), all rows selecting each expert
 * are grouped and only the unique selected experts are read (Moonshine README,
 * "How the engine works", prefill paragraph; Moonshine GitHub README,
 * "Prefill"), each selected expert runs its SwiGLU FFN on MXFP4 weights
 * (MoonTail, requester/volunteer table: "Routed expert FFN"; Moonshine GitHub
 * README, MiMo section: "MXFP4 kernels"), and the weighted expert outputs are
 * reduced back to token order (Moonshine README, "Run layer-major prefill":
 * the MoE tail's weighted reduction). Decode is token-major and prefill
 * layer-major (Moonshine README, "How the engine works"); here that split is
 * moe_decode (CUDA-core streaming of the selected experts) versus
 * moe_forward (grouped block-scaled tensor-core GEMMs).
 *
 * Conventions for every call below:
 *  - Pointers are DEVICE pointers unless marked "host". All calls are
 *    asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *    default stream) except moe_create, moe_destroy, moe_status and the
 *    size queries, which are host-only.
 *  - No call allocates or frees device memory, except moe_create (one 4-byte
 *    device status word) and moe_destroy (frees it). Scratch memory is the
 *    caller's `ws` buffer, sized by moe_workspace_bytes; the prepared weight
 *    scales of moe_prepare live in a caller buffer too.
 *  - The caller owns every buffer; the handle keeps the weight pointers it was
 *    given (it does not copy weights), so they must outlive the handle.
 *  - Return value: MOE_OK (0) or a negative MOE_ERR_* code. Argument errors are
 *    detected on the host before anything is launched. Data errors found on
 *    the device (NaN logits, out-of-range indices in a caller-supplied plan,
 *    an expired device-side wait) are recorded in the handle's status word and
 *    reported by moe_status; the kernels skip the offending element instead of
 *    faulting.
 *
 * Data layouts (row-major, C order):
 *   x        bf16 [T][d_model]               (uint16 bit patterns)
 *   logits   fp32 [T][n_experts]
 *   out      bf16 [T][d_model]
 *   MXFP4 matrix with N rows and reduction length K (K % 32 == 0):
 *     codes  uint8 [N][K/2]   element kk in byte kk/2, even element in the low
 *                             nibble; each nibble an OCP E2M1 code
 *     scales uint8 [N][K/32]  OCP E8M0 (2^(b-127)), one per 32 elements along K
 *   gate, up  per expert N = d_ff,    K = d_model   -> [E][d_ff][d_model/2] ...
 *   down      per expert N = d_model, K = d_ff      -> [E][d_model][d_ff/2] ...
 *   w_router  fp32 [n_experts][d_model]   (router_mode MOE_ROUTER_XWR only)
 *   sh_gate, sh_up bf16 [d_ff][d_model]; sh_down bf16 [d_model][d_ff]
 *                                         (has_shared only)
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status_code {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = -1,     /* null pointer, negative size, bad desc field */
    MOE_ERR_UNSUPPORTED = -2,     /* shape outside the supported envelope, or no sm_103 GPU */
    MOE_ERR_WORKSPACE = -3,       /* ws_bytes smaller than moe_workspace_bytes() */
    MOE_ERR_CUDA = -4,            /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = -5,  /* a device-side wait hit its iteration limit */
    MOE_ERR_NAN_LOGIT = -6,       /* a router logit was NaN (treated as -inf) */
    MOE_ERR_BAD_INDEX = -7,       /* out-of-range expert / row index in a plan */
    MOE_ERR_NOT_PREPARED = -8,    /* moe_forward before moe_prepare */
    MOE_ERR_CORRUPT_TILE = -9     /* a compressed-store tile failed its checks (record, table,
                                     final coder states, word count or Adler-32); the bytes
                                     of its slot are then undefined */
};

enum moe_router_mode {
    MOE_ROUTER_LOGITS = 0,  /* moe_plan takes fp32 logits [T][E] */
    MOE_ROUTER_XWR = 1      /* moe_plan computes logits = x . W_r^T in fp32 */
};

enum moe_op {
    MOE_OP_PLAN = 0,
    MOE_OP_FORWARD = 1,
    MOE_OP_DECODE = 2
};

/* Kernels moe_profile_kernel can bracket with events. */
enum moe_prof_kernel {
    MOE_PROF_NONE = 0,
    MOE_PROF_DECODE_GATEUP = 1,   /* moe_decode: gate/up + SwiGLU streaming kernel */
    MOE_PROF_DECODE_DOWN = 2,     /* moe_decode: down-projection streaming kernel */
    MOE_PROF_FORWARD_GEMM1 = 3,   /* moe_forward: grouped gate/up GEMM */
    MOE_PROF_FORWARD_GEMM2 = 4,   /* moe_forward: grouped down GEMM + weighted scatter */
    MOE_PROF_ROUTER = 5,          /* moe_plan / moe_router_logits: x . W_r GEMM */
    MOE_PROF_SHARED_GATEUP = 6,   /* shared expert: gate/up GEMM + SwiGLU */
    MOE_PROF_SHARED_DOWN = 7,     /* shared expert: down GEMM */
    MOE_PROF_STREAM_COPY = 8      /* expert streaming: copy (or, from a compressed store, decode)
                                     of the missing experts from host memory */
};

/* Precision of the activations the tensor cores see in moe_forward.
 * MOE_ACT_EXACT: x and h as two E4M3 terms with an E8M0 scale per 32 values
 * each, about bf16's 8 significant bits, within the layer's parity tolerance.
 * MOE_ACT_MXFP4: the FP4 x FP4 mode, x and h as one MXFP4 term (E2M1 with an
 * E8M0 scale per 32, converted as OCP MX v1.0 section 6.3 specifies: scale
 * 2^(floor(log2 max|v|) - 2), elements rounded to nearest even, clamped to
 * 6), MMAs of kind::mxf4 at the FP4 tensor rate. Its output differs from the
 * exact layer by far more than bf16 rounding (normwise max error about 0.2 on
 * N(0,1) inputs at the K3 shape): a separately reported fast mode for the
 * pages' MXFP4 expert kernels shared by the K3 and MiMo lanes (Moonshine
 * GitHub README, "Running MiMo V2.6 Flash"), not the parity path. moe_decode
 * always computes with exact products (it ignores act_mode). */
enum moe_act_mode {
    MOE_ACT_EXACT = 0,
    MOE_ACT_MXFP4 = 1
};

/* Storage format of the routed experts' weights.
 * MOE_W_MXFP4: the MXFP4 layout above (E2M1 codes + E8M0 scale per 32).
 * MOE_W_FP8: the FP8 lane (Moonshine GitHub README, "GLM 5.3 Flash status":
 *   FP8 E4M3FN experts with a fused decode GEMV and a BF16-dequant prefill).
 *   The pages give no scale layout; here each matrix with N rows and
 *   reduction length K is
 *     codes  uint8 [N][K]                        one OCP E4M3FN code per weight
 *     scales fp32  [ceil(N/128)][ceil(K/128)]    one scale per 128 x 128 block
 *   weight = value(code) * scale, passed through the same moe_weights fields
 *   (gate_q / gate_s ...; the scale pointers point at fp32 data, 4-byte
 *   aligned; codes 16-byte aligned). moe_decode (and moe_decode_noalloc)
 *   streams the codes on CUDA cores with exact products; moe_forward runs bf16
 *   tensor-core GEMMs on a bf16 copy of the experts (each weight rounded to
 *   nearest even) that moe_prepare writes into its caller buffer. act_mode
 *   must be MOE_ACT_EXACT; expert streaming is not offered for this format. */
enum moe_weight_format {
    MOE_W_MXFP4 = 0,
    MOE_W_FP8 = 1
};

/* Layer shape. Supported envelope: d_model a multiple of 256, d_ff of 128,
 * d_model <= 16384, d_ff <= 8192, 1 <= top_k <= 32, top_k <= n_experts <= 1024. */
typedef struct moe_desc {
    int32_t d_model;
    int32_t d_ff;
    int32_t n_experts;
    int32_t top_k;
    int32_t router_mode;    /* enum moe_router_mode */
    int32_t has_shared;     /* 1: one always-on bf16 SwiGLU shared expert, weight 1.0 */
    int32_t act_mode;       /* enum moe_act_mode (moe_forward only) */
    int32_t weight_format;  /* enum moe_weight_format */
} moe_desc;

/* Device pointers to the layer's weights (see layouts above). Unused fields NULL. */
typedef struct moe_weights {
    const uint8_t *gate_q, *gate_s;
    const uint8_t *up_q, *up_s;
    const uint8_t *down_q, *down_s;
    const float *w_router;
    const uint16_t *sh_gate, *sh_up, *sh_down;
} moe_weights;

/* Route plan, caller-allocated device buffers, written by moe_plan:
 *   topk_idx int32 [T][top_k]  selected experts, descending logit, ties to the
 *                              lower expert index (+0 == -0)
 *   topk_w   fp32  [T][top_k]  exp(l_j - l_max) / sum over the selected
 *   counts   int32 [E]         rows routed to each expert
 *   offsets  int32 [E+1]       exclusive scan of counts; offsets[E] = T*top_k
 *   perm     int32 [T*top_k]   flat indices t*top_k+j sorted by (expert, flat)
 *   inv      int32 [T*top_k]   inv[perm[p]] = p
 *   active   int32 [E+1]       active[0] = number of experts with rows,
 *                              active[1..] = those experts, ascending
 * moe_forward and moe_decode read topk_w, offsets, perm, inv and active. */
typedef struct moe_plan_buf {
    int32_t *topk_idx;
    float *topk_w;
    int32_t *counts;
    int32_t *offsets;
    int32_t *perm;
    int32_t *inv;
    int32_t *active;
} moe_plan_buf;

typedef struct moe_handle moe_handle;

/* Host. Validates the shape against the supported envelope and the current
 * device (must be compute capability 10.3), records the weight pointers and
 * allocates the 4-byte device status word. *out is NULL on failure. */
int moe_create(const moe_desc *desc, const moe_weights *weights, moe_handle **out);

/* Host. Frees the status word and the handle. NULL is a no-op. */
void moe_destroy(moe_handle *h);

/* Host. Bytes of one expert's three MXFP4 matrices (codes + scales):
 * 3 * (d_model*d_ff/2 + d_model*d_ff/32). 17,547,264 for d_model=7168,
 * d_ff=1536. Returns -1 if either size is not a positive multiple of 32. */
int64_t moe_expert_bytes(int32_t d_model, int32_t d_ff);

/* Host. Bytes of the buffer moe_prepare fills. FP8 layers: the bf16 copy of
 * every expert's three matrices (3 * n_experts * d_model * d_ff * 2 bytes,
 * each matrix array rounded up to 256; 59.2 GB for an 896-expert K3-shaped
 * layer), plus the W_r terms below for router_mode MOE_ROUTER_XWR. MXFP4
 * layers: the three weight-scale arrays
 * (3 * n_experts * d_model * d_ff / 32 bytes when d_model and d_ff are
 * multiples of 256, 924 MB for the 896-expert K3 layer; a K chunk pair is
 * padded when the chunk count is odd; rounded up to 256) plus, for router_mode MOE_ROUTER_XWR, three bf16
 * copies of W_r's shape (3 * n_experts * d_model * 2 bytes, each rounded up to
 * 256; 38.5 MB for K3). */
size_t moe_prepared_bytes(const moe_handle *h);

/* One-time weight-layout preparation for moe_forward (asynchronous on
 * `stream`). Re-lays the E8M0 weight scales into the order the tensor cores
 * consume them: for each (expert, 128-row weight tile, pair of 128-wide K
 * chunks) one contiguous 1 KB block, the layout of one TMEM lane quadrant of
 * a 128x256b tensor-memory copy (lane l < 32, column j < 8 at byte
 * (l / 8) * 256 + (j / 4) * 128 + (l % 8) * 16 + (j % 4) * 4; column j holds
 * the four block scales of tile row 32 * (j % 4) + l in K chunk
 * 2 * pair + j / 4). Gate/up tiles are 64 gate rows over the same 64 up
 * rows, down tiles 128 consecutive rows. `buf` is caller-owned device memory
 * of at least moe_prepared_bytes(h) bytes, 256-byte aligned; the handle keeps
 * the pointer, so it must outlive the handle, and the weight scales must not
 * change afterwards without calling moe_prepare again. moe_decode does not
 * need it; moe_forward returns MOE_ERR_NOT_PREPARED without it.
 * For router_mode MOE_ROUTER_XWR it also splits W_r into three bf16 terms
 * t0 + t1 + t2 == W_r exactly (t0 the round-to-nearest bf16 of W_r, t1 of the
 * remainder, t2 of what is left), which the router GEMM reads; moe_plan and
 * moe_router_logits return MOE_ERR_NOT_PREPARED without it, and w_router must
 * not change afterwards without calling moe_prepare again. */
int moe_prepare(moe_handle *h, void *buf, size_t bytes, void *stream);

/* Host. Scratch bytes `op` (enum moe_op) needs for T tokens; 0 for T == 0.
 * MOE_OP_PLAN includes the fp32 logits [T][E] for router_mode MOE_ROUTER_XWR;
 * MOE_OP_DECODE and MOE_OP_FORWARD include the shared expert's intermediate
 * (bf16 [T][d_ff], and for decode its fp32 output [T][d_model]) when
 * has_shared is set. */
size_t moe_workspace_bytes(const moe_handle *h, int32_t T, int32_t op);

/* Route T tokens: top-k + weights, then the stable per-expert plan.
 * MOE_ROUTER_LOGITS: logits fp32 [T][E] given, x ignored (may be NULL).
 * MOE_ROUTER_XWR: logits must be NULL and x given (16-byte aligned); the
 * logits are first computed as in moe_router_logits into the front of ws
 * (requires moe_prepare). ws: >= moe_workspace_bytes(h, T, MOE_OP_PLAN),
 * 256-byte aligned when that is non-zero. T == 0 is a no-op returning MOE_OK. */
int moe_plan(moe_handle *h, int32_t T, const float *logits, const uint16_t *x,
             const moe_plan_buf *plan, void *ws, size_t ws_bytes, void *stream);

/* The router alone (router_mode MOE_ROUTER_XWR): logits fp32 [T][E] =
 * x . W_r^T with fp32 accumulation, on tensor cores as three bf16 GEMMs
 * against the W_r terms moe_prepare made (so every product is exact and only
 * the fp32 accumulation rounds). The router is part of the resident static
 * tier (Moonshine README, "How the engine works"). x bf16 [T][d_model],
 * 16-byte aligned; logits caller-owned, 4-byte aligned. No workspace.
 * Returns MOE_ERR_INVALID_ARG for router_mode MOE_ROUTER_LOGITS and
 * MOE_ERR_NOT_PREPARED before moe_prepare. */
int moe_router_logits(moe_handle *h, int32_t T, const uint16_t *x, float *logits, void *stream);

/* Layer-major expert FFN for a planned batch (prefill): grouped block-scaled
 * MXFP4 GEMMs on tcgen05 tensor cores (gate/up with SwiGLU, then down with
 * the weighted scatter), finalised to bf16 out [T][d_model]. With has_shared
 * the shared expert (bf16 tensor-core GEMMs, SwiGLU, weight 1.0) is added
 * before the bf16 rounding.
 * Requires moe_prepare. ws: >= moe_workspace_bytes(h, T, MOE_OP_FORWARD),
 * 256-byte aligned. */
int moe_forward(moe_handle *h, int32_t T, const uint16_t *x, const moe_plan_buf *plan,
                uint16_t *out, void *ws, size_t ws_bytes, void *stream);

/* Token-major expert FFN (decode, any T; intended for T <= 16): streams only
 * the active experts' packed codes with 128-bit loads and reduces on CUDA
 * cores in fp32, then combines deterministically in top-k order (the shared
 * expert's output, with has_shared, added last).
 * ws: >= moe_workspace_bytes(h, T, MOE_OP_DECODE). */
int moe_decode(moe_handle *h, int32_t T, const uint16_t *x, const moe_plan_buf *plan,
               uint16_t *out, void *ws, size_t ws_bytes, void *stream);

/* moe_decode without any device allocation, for callers that cannot call
 * cudaMalloc (for example code running where the allocator is owned by
 * someone else, or which must not allocate after start-up). No passage of the
 * pages describes this entry point; it is an interface convenience with no
 * counterpart there.
 * The scratch moe_decode takes from `ws` lives instead in one fixed array
 * inside the library (a static device array of about 9.5 MB that every GPU
 * which loads the library holds until the process exits). It fits T * top_k
 * <= 256 routed rows for d_ff <= 2048 and d_model <= 8192; larger calls
 * return MOE_ERR_WORKSPACE. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress; again after the device's context
 * changed, e.g. after cudaDeviceReset), so make that first call before any
 * stream capture. All calls share the array: calls whose kernels overlap on
 * the GPU (other streams, other threads) race on it and must be serialised by
 * the caller. Same inputs, outputs and results as moe_decode; the plan comes
 * from moe_plan, which needs no workspace for T <= 64 with router_mode
 * MOE_ROUTER_LOGITS. Layers with has_shared return MOE_ERR_UNSUPPORTED (the
 * fixed array has no room for the shared expert's intermediates). */
int moe_decode_noalloc(moe_handle *h, int32_t T, const uint16_t *x, const moe_plan_buf *plan,
                       uint16_t *out, void *stream);

/* ---------------------------------------------------------------------------
 * Expert streaming: the routed experts stay in a large slow tier and the ones
 * a batch selects are copied into a fixed number of per-layer slots with
 * online least-recently-used replacement, reading the route union once per
 * batch (Moonshine README, "How the engine works"; Moonshine GitHub README,
 * "Decode"). On GB300
 * the slow tier is host memory that the GPU reads directly (pinned host
 * allocations are device-addressable; over NVLink-C2C on Grace) and the slots
 * are HBM. The cache is managed on the device: no host round trip per call.
 *
 * Replacement rule (exact, so that callers and tests can predict it): each
 * moe_forward call advances a clock; every active expert of the plan that is
 * resident gets its slot stamped with the clock (a hit); the missing experts,
 * in increasing expert index, take the slots not stamped by this call in
 * increasing (stamp, slot) order (empty slots carry stamp 0, so they go
 * first), evicting the experts held there.
 * ------------------------------------------------------------------------- */

/* Host. Bytes of the device cache-state buffer for a streaming handle:
 * clock, counters, slot_of [n_experts], expert_of / stamp [n_slots], last
 * miss lists. */
size_t moe_stream_state_bytes(int32_t n_experts, int32_t n_slots);

/* Host. Like moe_create for a layer whose routed experts live in host memory.
 *   host_w  gate/up/down codes and scales of all n_experts experts (layouts of
 *           moe_weights), host memory the device can read (e.g. cudaHostAlloc);
 *           each array 16-byte aligned; w_router / sh_* are ignored here.
 *   slot_w  device arrays in the same layouts holding n_slots experts (the
 *           cache; 32-byte aligned codes, 16-byte aligned scales), plus the
 *           resident-tier pointers w_router / sh_gate / sh_up / sh_down as for
 *           moe_create.
 *   n_slots 1..min(n_experts, 1024).
 *   state   device buffer of moe_stream_state_bytes(n_experts, n_slots) bytes,
 *           caller-owned, zero-initialised by this call (stream 0, synchronous).
 * moe_prepared_bytes then sizes the prepared buffer for n_slots experts;
 * moe_prepare re-lays only the resident tier (W_r) and records the buffer:
 * slots are prepared as experts arrive. moe_forward makes every active expert
 * of the plan resident before its GEMMs (misses copied from host memory) and
 * returns MOE_ERR_UNSUPPORTED when T * top_k exceeds n_slots while n_experts
 * does too (the plan could then need more slots than exist). moe_decode and
 * moe_decode_noalloc return MOE_ERR_UNSUPPORTED on a streaming handle. */
int moe_create_streaming(const moe_desc *desc, const moe_weights *host_w,
                         const moe_weights *slot_w, int32_t n_slots, void *state,
                         moe_handle **out);

/* Host. Synchronises `stream` and reads the cache counters of a streaming
 * handle: total hits and misses (experts) over all calls, and the misses of
 * the last call. MOE_ERR_INVALID_ARG for other handles. */
int moe_stream_stats(moe_handle *h, int64_t *hits, int64_t *misses, int32_t *last_misses,
                     void *stream);

/* ---------------------------------------------------------------------------
 * Compressed expert store: the slow tier holds the experts rANS-coded in
 * independent 16 KiB tiles, and the GPU decodes the missing experts of a call
 * straight into ordinary cache slots (Moonshine GitHub README, "Expert-stream
 * compression" / "MZG2 production store": redundant MXFP4 negative zeros
 * canonicalised, independently bounded 16 KiB tiles, a checksum per tile and
 * a check of the coder's final state, decode on the GPU into decoded cache
 * slots). The pages fix no byte format; this library's format:
 *  - An expert's arrays in the order gate_q, gate_s, up_q, up_s, down_q,
 *    down_s (layouts of moe_weights; D*F/2 bytes per code array, D*F/32 per
 *    scale array). Canonical bytes: every E2M1 code 0x8 (negative zero) in
 *    the code arrays becomes 0x0 (same value); scale bytes unchanged.
 *  - One frequency table per (expert, array): f[256] (uint16), summing to
 *    4096; f[b] = 0 for bytes absent from the array, else
 *    max(1, floor(count * 4096 / n)), after which, while the sum exceeds 4096,
 *    the largest entry (lowest byte value among equals) loses one, and while
 *    it falls short, the largest gains one. cum[b] = f[0] + ... + f[b-1].
 *  - Each array is cut into 16384-byte tiles (the last may be shorter); an
 *    expert has moe_store_tiles_per_expert() tiles, arrays in order. A tile
 *    of n bytes is coded by 32 interleaved rANS coders (byte i to coder i % 32,
 *    step i / 32) with 32-bit states in [2^16, 2^32) and 16-bit words.
 *    Decoding, steps in increasing order: each coder with a byte in the step
 *    takes q = x % 4096, the byte b with cum[b] <= q < cum[b] + f[b], sets
 *    x = f[b] * (x / 4096) + q - cum[b] and, if x < 2^16, reads the next word
 *    (x = x * 2^16 + w; within a step, coders in increasing order). Encoding
 *    is the exact reverse, starting every coder at 2^16; a sound tile ends
 *    with every state at 2^16 and every word read.
 *  - Stored tile: the 32 final states (uint32, coder 0 first) then the words
 *    (uint16) in read order, when 128 + 2 * words < n; otherwise the n
 *    canonical bytes (raw). Zero-padded to a multiple of 16 bytes, back to back.
 * ------------------------------------------------------------------------- */

/* One tile's record (32 bytes). */
typedef struct moe_tile_rec {
    uint32_t offset_lo, offset_hi;  /* bytes from the start of the blob; multiple of 16 */
    uint32_t n_bytes;               /* decoded bytes, 1..16384 */
    uint32_t n_words;               /* 16-bit words of a coded tile; 0 when raw */
    uint32_t adler;                 /* Adler-32 (zlib's definition) of the canonical bytes */
    uint32_t flags;                 /* bit 0: stored raw */
    uint32_t reserved[2];           /* 0 */
} moe_tile_rec;

/* A store as the device reads it. */
typedef struct moe_store {
    const uint8_t *blob;         /* host memory the device can read (cudaHostAlloc or
                                    registered, mapped at the host address), 16-byte aligned */
    int64_t blob_bytes;
    const moe_tile_rec *tiles;   /* device, [n_experts][tiles per expert], 16-byte aligned */
    const uint16_t *tables;      /* device, [n_experts][6][256], 16-byte aligned */
} moe_store;

/* Host. Tiles of one expert: sum over the six arrays of ceil(bytes / 16384);
 * -1 unless d_model and d_ff are positive multiples of 32. 1071 for K3. */
int32_t moe_store_tiles_per_expert(int32_t d_model, int32_t d_ff);

/* Host. Blob capacity moe_store_encode needs: every tile at its raw size
 * rounded up to 16 bytes, for n_experts experts (the encoder first lays each
 * expert out at that stride, then packs the blob). -1 on bad sizes. */
int64_t moe_store_blob_bound(int32_t n_experts, int32_t d_model, int32_t d_ff);

/* Host. Builds the store of experts 0..n_experts-1 from HOST weight arrays
 * (host_w: gate/up/down codes and scales in the layouts of moe_weights; any
 * host memory; other fields ignored). Writes blob (host, blob_cap >=
 * moe_store_blob_bound bytes; *blob_bytes receives the packed size), tiles
 * (host, n_experts * tiles-per-expert records) and tables (host,
 * n_experts * 6 * 256). n_threads host threads (<= 0: one per core). Copy
 * tiles and tables to the device and keep the blob in device-readable host
 * memory for moe_create_streaming_store / moe_store_decode. */
int moe_store_encode(int32_t n_experts, int32_t d_model, int32_t d_ff, const moe_weights *host_w,
                     uint8_t *blob, int64_t blob_cap, int64_t *blob_bytes, moe_tile_rec *tiles,
                     uint16_t *tables, int32_t n_threads);

/* Decodes experts[i] of the store into slot slots[i] of the arrays in slot_w
 * (device arrays holding n_slots experts, layouts of moe_weights), i < n.
 * experts and slots are device int32 [n]; status a device int32 that receives
 * the first error (MOE_ERR_BAD_INDEX for an expert or slot out of range,
 * MOE_ERR_CORRUPT_TILE for a tile that fails a check; the kernel skips that
 * tile and never reads or writes out of bounds). Asynchronous on `stream`. */
int moe_store_decode(int32_t n_experts, int32_t d_model, int32_t d_ff, const moe_store *store,
                     const int32_t *experts, const int32_t *slots, int32_t n,
                     const moe_weights *slot_w, int32_t n_slots, int32_t *status, void *stream);

/* Host. moe_create_streaming with the routed experts in a compressed store:
 * moe_forward decodes each call's missing experts from the store into their
 * slots (instead of copying them). Same slot_w, n_slots and state rules;
 * the store's arrays must outlive the handle. */
int moe_create_streaming_store(const moe_desc *desc, const moe_store *store,
                               const moe_weights *slot_w, int32_t n_slots, void *state,
                               moe_handle **out);

/* Host. Instrumentation for timing one kernel on the library's own stream:
 * while `which` names a kernel (enum moe_prof_kernel), every later call that
 * launches it records ev_start (a cudaEvent_t) immediately before that launch
 * and ev_stop immediately after it, on the call's stream. The caller owns the
 * events and may swap them between calls; MOE_PROF_NONE turns it off. */
int moe_profile_kernel(moe_handle *h, int32_t which, void *ev_start, void *ev_stop);

/* Test hooks for the device-side timeout path. Every wait inside the
 * library's kernels is bounded; when one runs out the kernel records
 * MOE_ERR_DEVICE_TIMEOUT, stops its work, waits (bounded) for its own copies
 * and MMAs in flight, releases its tensor memory and returns, so the context
 * stays usable and the next call runs normally. The pages' counterpart is a
 * system that refuses or reports rather than half-running or hanging
 * (Moonshine GitHub README, MiMo section: memory guards and request
 * deadlines; MeshMoE Cell page: failure detection); they describe no such
 * hook. Off by default; meant for tests only. */
enum moe_inject {
    MOE_INJECT_NONE = 0,
    MOE_INJECT_GEMM_STALL = 1  /* moe_forward's gate/up GEMM: in every CTA the first MMA issuer
                                  waits on a barrier that nothing signals, so that wait runs
                                  out with operand copies in flight */
};

/* Host. Sets the handle's injection mode (enum moe_inject) and the limit of
 * every device-side wait of its later calls, in SM clock cycles
 * (timeout_cycles <= 0: the default, 2e9 cycles, about one second; otherwise
 * at least 1e5). Returns MOE_ERR_INVALID_ARG for an unknown mode or a limit
 * below 1e5. */
int moe_set_fault_injection(moe_handle *h, int32_t mode, int64_t timeout_cycles);

/* Host. Synchronises `stream`, returns the first device-side error recorded
 * since the last call (MOE_OK if none) and clears it. */
int moe_status(moe_handle *h, void *stream);

/* Host. Static description of a status code. */
const char *moe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
