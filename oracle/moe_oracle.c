/*
 * CPU oracle for the routed-expert FFN of a Kimi-K3-style MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it. It shares no code with the CUDA library (no headers, tables or
 * helpers); its inputs come from the seeded generator in synth/ or from the
 * caller, never from the GPU.
 *
 * What it computes, in the order the pages state the problem:
 *   route   - each token selects 16 of 896 experts per routed layer
 *             (MoonTail, intro; Moonshine README, "How the engine works");
 *             weights are the softmax over the selected logits, ties go to the
 *             lower expert index;
 *   plan    - all rows selecting each expert are grouped, and only the unique
 *             selected experts are touched (Moonshine README, "How the engine
 *             works", prefill paragraph; Moonshine GitHub README, "Prefill");
 *   ffn     - per (token, selected expert) the SwiGLU expert FFN on MXFP4
 *             weights (MoonTail, requester/volunteer table: "Routed expert
 *             FFN"; Moonshine GitHub README, MiMo section: the shared "MXFP4
 *             kernels"), then the weighted reduction back to token order
 *             (Moonshine README, "Run layer-major prefill": weighted reduction).
 *
 * MXFP4 follows the OCP Microscaling (MX) format: E2M1 elements (1 sign bit,
 * 2 exponent bits with bias 1, 1 mantissa bit) sharing one E8M0 scale
 * (2^(b-127), b = 255 is NaN) per 32 consecutive elements along K. The pages
 * only name the format; the byte layout used here is one reading:
 * element kk of a row lives in byte kk/2, the even element in the low nibble.
 *
 * All floating point is fp64. Every product of a decoded weight and a bf16
 * activation is exact in fp64; sums run in plain sequential order.
 *
 * Parity pins (tests/test_oracle_*.py): OCP E2M1 value table, torch's E8M0 and
 * E4M3 decoders, brute-force dense evaluation in numpy, the E=1/k=1 textbook
 * SwiGLU FFN, the k=E full softmax mixture, a closed-form all-ones expert,
 * exact power-of-two scaling, and numpy's stable argsort for route and plan.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---- MXFP4 element and scale decode (OCP MX: E2M1, E8M0) ---------------- */

/* E2M1: sign s, exponent field e (bias 1), mantissa bit m.
 * e == 0 is subnormal: (-1)^s * 2^(1-1) * (0 + m/2); otherwise
 * (-1)^s * 2^(e-1) * (1 + m/2). Code 8 is the redundant negative zero. */
ORACLE_API double oracle_e2m1(int code) {
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -mag : mag;
}

/* E8M0: 2^(b - 127); b = 255 encodes NaN. */
ORACLE_API double oracle_e8m0(int b) {
    if (b == 255) return NAN;
    return ldexp(1.0, b - 127);
}

static int oracle_code_at(const uint8_t *q_row, int64_t kk) {
    uint8_t byte = q_row[kk / 2];
    return (kk % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
}

/* W[n][kk] = e2m1(code(n, kk)) * e8m0(S[n][kk / 32]); rows x K, row-major. */
ORACLE_API int oracle_dequant(const uint8_t *q, const uint8_t *s, int64_t rows, int64_t K,
                              double *out) {
    if (K % 32 != 0) return -1;
    for (int64_t n = 0; n < rows; ++n)
        for (int64_t kk = 0; kk < K; ++kk)
            out[n * K + kk] = oracle_e2m1(oracle_code_at(q + n * (K / 2), kk)) *
                              oracle_e8m0(s[n * (K / 32) + kk / 32]);
    return 0;
}

static double oracle_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ---- Route: top-k of E per token, softmax over the selected logits ------- */

typedef struct { double v; int e; } oracle_cand;

static int oracle_cand_cmp(const void *a, const void *b) {
    const oracle_cand *x = (const oracle_cand *)a, *y = (const oracle_cand *)b;
    if (x->v > y->v) return -1;   /* descending logit */
    if (x->v < y->v) return 1;
    return (x->e < y->e) ? -1 : (x->e > y->e);  /* tie: lower expert first */
}

/* idx[t][j], w[t][j] for j < k: the k largest logits of token t in descending
 * order (ties to the lower index; +0 and -0 compare equal) and
 * w_j = exp(l_j - l_max) / sum_i exp(l_i - l_max) over the selected i.
 * Returns -2 if a logit is NaN (the pages define no order for NaN). */
ORACLE_API int oracle_route(int T, int E, int k, const double *logits, int32_t *idx, double *w) {
    if (k < 1 || k > E) return -1;
    oracle_cand *c = (oracle_cand *)malloc(sizeof(oracle_cand) * (size_t)E);
    int rc = 0;
    for (int t = 0; t < T && rc == 0; ++t) {
        for (int e = 0; e < E; ++e) {
            c[e].v = logits[(int64_t)t * E + e];
            c[e].e = e;
            if (isnan(c[e].v)) rc = -2;
        }
        if (rc) break;
        qsort(c, (size_t)E, sizeof(oracle_cand), oracle_cand_cmp);
        double lmax = c[0].v, z = 0.0;
        for (int j = 0; j < k; ++j) z += exp(c[j].v - lmax);
        for (int j = 0; j < k; ++j) {
            idx[(int64_t)t * k + j] = c[j].e;
            w[(int64_t)t * k + j] = exp(c[j].v - lmax) / z;
        }
    }
    free(c);
    return rc;
}

/* ---- Plan: group the T*k (token, slot) rows by expert -------------------- */

/* counts[e] = #{flat f = t*k + j : idx[f] == e};  offsets = exclusive scan,
 * offsets[E] = T*k;  perm = flat indices in (expert, flat) order (a stable
 * counting sort);  inv[perm[p]] = p;  active[0] = number of experts with a
 * non-empty segment, active[1..] = those experts, ascending (the route union). */
ORACLE_API int oracle_plan(int T, int E, int k, const int32_t *idx, int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *active) {
    int64_t n = (int64_t)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t f = 0; f < n; ++f) {
        if (idx[f] < 0 || idx[f] >= E) return -1;
        counts[idx[f]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
    for (int64_t f = 0; f < n; ++f) {
        int32_t p = fill[idx[f]]++;
        perm[p] = (int32_t)f;
        inv[f] = p;
    }
    free(fill);
    int na = 0;
    for (int e = 0; e < E; ++e)
        if (counts[e] > 0) active[1 + na++] = e;
    active[0] = na;
    return 0;
}

/* ---- Router logits (in-library router workload) -------------------------- */

/* logits[t][e] = sum_d x[t][d] * W_r[e][d]; x bf16 [T][D], W_r fp32 [E][D]. */
ORACLE_API void oracle_router_logits(int T, int D, int E, const uint16_t *x, const float *wr,
                                     double *logits) {
#pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d)
                acc += oracle_bf16(x[(int64_t)t * D + d]) * (double)wr[(int64_t)e * D + d];
            logits[(int64_t)t * E + e] = acc;
        }
}

/* ---- Expert FFN and weighted combine ------------------------------------- */

static double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* MXFP4 matrix-vector product: y[n] = sum_kk W[n][kk] * v[kk] for one row n. */
static double oracle_mx_row_dot(const uint8_t *q, const uint8_t *s, int64_t n, int64_t K,
                                const double *v) {
    const uint8_t *qr = q + n * (K / 2);
    const uint8_t *sr = s + n * (K / 32);
    double acc = 0.0;
    for (int64_t kk = 0; kk < K; ++kk)
        acc += oracle_e2m1(oracle_code_at(qr, kk)) * oracle_e8m0(sr[kk / 32]) * v[kk];
    return acc;
}

/*
 * out[i][:] = sum_j w[i][j] * FFN_{idx[i][j]}(x[i]) for n_tok tokens, where
 *   FFN_e(x) = W_down[e] . ( silu(W_gate[e] . x) * (W_up[e] . x) ).
 * The experts' weights are given compacted: store slot s holds expert
 * store_expert[s]; gate/up are [F][D/2] codes + [F][D/32] scales, down is
 * [D][F/2] + [D][F/32], per slot. out is overwritten.
 * Returns -3 if a selected expert is missing from the store.
 */
ORACLE_API int oracle_ffn(int n_tok, int D, int F, int k, const uint16_t *x, const int32_t *idx,
                          const double *w, int n_store, const int32_t *store_expert,
                          const uint8_t *gate_q, const uint8_t *gate_s, const uint8_t *up_q,
                          const uint8_t *up_s, const uint8_t *down_q, const uint8_t *down_s,
                          double *out) {
    if (D % 32 || F % 32) return -1;
    double *xv = (double *)malloc(sizeof(double) * (size_t)D);
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    int rc = 0;
    const int64_t gq = (int64_t)F * D / 2, gs = (int64_t)F * D / 32;
    for (int i = 0; i < n_tok && rc == 0; ++i) {
        for (int d = 0; d < D; ++d) {
            xv[d] = oracle_bf16(x[(int64_t)i * D + d]);
            out[(int64_t)i * D + d] = 0.0;
        }
        for (int j = 0; j < k; ++j) {
            int e = idx[(int64_t)i * k + j];
            int slot = -1;
            for (int s = 0; s < n_store; ++s)
                if (store_expert[s] == e) { slot = s; break; }
            if (slot < 0) { rc = -3; break; }
            const uint8_t *Gq = gate_q + slot * gq, *Gs = gate_s + slot * gs;
            const uint8_t *Uq = up_q + slot * gq, *Us = up_s + slot * gs;
            const uint8_t *Dq = down_q + slot * gq, *Ds = down_s + slot * gs;
#pragma omp parallel for schedule(static)
            for (int f = 0; f < F; ++f) {
                double g = oracle_mx_row_dot(Gq, Gs, f, D, xv);
                double u = oracle_mx_row_dot(Uq, Us, f, D, xv);
                h[f] = oracle_silu(g) * u;
            }
            double wj = w[(int64_t)i * k + j];
#pragma omp parallel for schedule(static)
            for (int d = 0; d < D; ++d)
                out[(int64_t)i * D + d] += wj * oracle_mx_row_dot(Dq, Ds, d, F, h);
        }
    }
    free(xv);
    free(h);
    return rc;
}

/*
 * Shared expert (always-on, weight 1.0), bf16 weights:
 *   out[i][:] += Ws_down . ( silu(Ws_gate . x) * (Ws_up . x) )
 * Ws_gate, Ws_up [F][D]; Ws_down [D][F].
 */
ORACLE_API void oracle_shared_ffn(int n_tok, int D, int F, const uint16_t *x, const uint16_t *sg,
                                  const uint16_t *su, const uint16_t *sd, double *out) {
    double *h = (double *)malloc(sizeof(double) * (size_t)F);
    for (int i = 0; i < n_tok; ++i) {
        const uint16_t *xi = x + (int64_t)i * D;
#pragma omp parallel for schedule(static)
        for (int f = 0; f < F; ++f) {
            double g = 0.0, u = 0.0;
            for (int d = 0; d < D; ++d) {
                double xd = oracle_bf16(xi[d]);
                g += oracle_bf16(sg[(int64_t)f * D + d]) * xd;
                u += oracle_bf16(su[(int64_t)f * D + d]) * xd;
            }
            h[f] = oracle_silu(g) * u;
        }
#pragma omp parallel for schedule(static)
        for (int d = 0; d < D; ++d) {
            double y = 0.0;
            for (int f = 0; f < F; ++f) y += oracle_bf16(sd[(int64_t)d * F + f]) * h[f];
            out[(int64_t)i * D + d] += y;
        }
    }
    free(h);
}
