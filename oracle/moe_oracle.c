/*
 * moe_oracle.c -- plain single-threaded CPU oracle (TEST INFRASTRUCTURE ONLY).
 *
 * See moe_oracle.h for the readings of the pages this follows.  Every
 * function is written as the plain definition: loops in (t, k) or (t, r)
 * order, no blocking, no fusion.  Build with -ffp-contract=off so that the
 * only fused multiply-add is the explicit fmaf() in the combine.
 *
 * Sources:
 *   "Inside the Nebius + PyTorch DeepSeek V3 recipe", section "Mixture-of-
 *   experts and wide expert parallelism" (experts partitioned across EP
 *   ranks; dispatch sends tokens to their assigned experts, combine returns
 *   expert outputs to their original positions; each GPU holds 8 of 256
 *   experts at EP32);
 *   Hybrid-EP news article (cryptojournalpost, Feb 2 2026), "Why This
 *   Issues for AI Infrastructure" (8 of 256
 *   experts active per token), "Technical Structure"
 *   (dispatch and combine operators) and "Availability and Integration"
 *   (worst-case buffer preallocation);
 *   "MoE / Hybrid-EP Validation", "FP8 dispatch restriction" and the
 *   measured-reference table (FP8 dispatch).
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs */

static uint32_t f32_bits(float v) { uint32_t u; memcpy(&u, &v, 4); return u; }
static float bits_f32(uint32_t u) { float v; memcpy(&v, &u, 4); return v; }

/* bfloat16 keeps the upper 16 bits of the binary32 pattern (sign, 8-bit
 * exponent, 7 mantissa bits).  Round to nearest: look at the 16 dropped bits;
 * above half -> round the magnitude up, below half -> truncate, exactly half
 * -> make the kept lowest bit even.  A carry out of the mantissa moves to the
 * next binade (and from the largest finite value to infinity), which is the
 * IEEE result. */
uint16_t moe_ref_bf16_encode(float v)
{
    uint32_t u = f32_bits(v);
    if (isnan(v)) return (uint16_t)((u >> 16) | 0x0040u);   /* quiet NaN, sign kept */
    uint32_t upper = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

float moe_ref_bf16_decode(uint16_t b) { return bits_f32((uint32_t)b << 16); }

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 encodes subnormals M * 2^-9;
 * fields 1..15 encode (1 + M/8) * 2^(E-7), except S.1111.111 which is NaN,
 * so the largest finite magnitude is 1.75 * 2^8 = 448 and there is no
 * infinity.  Conversion: round to nearest with ties to even, magnitudes at or
 * above 448 saturate to 448 (the "satfinite" conversion). */
uint8_t moe_ref_e4m3_encode(float v)
{
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < 0.015625) {                         /* below 2^-6: subnormal step 2^-9 */
        double m = nearbyint(a * 512.0);        /* exact scaling, ties to even   */
        return (uint8_t)(sign | (uint8_t)m);    /* m == 8 is the code of 2^-6    */
    }
    int e2;
    double f = frexp(a, &e2);                   /* a = f * 2^e2, f in [0.5, 1)   */
    int ex = e2 - 1;                            /* a = (2f) * 2^ex, 2f in [1, 2) */
    double mant = nearbyint((2.0 * f - 1.0) * 8.0);   /* exact, ties to even      */
    if (mant == 8.0) { mant = 0.0; ex += 1; }
    return (uint8_t)(sign | (uint8_t)(((ex + 7) << 3) | (int)mant));
}

float moe_ref_e4m3_decode(uint8_t q)
{
    int s = q >> 7, e = (q >> 3) & 0xF, m = q & 7;
    double v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);    /* (1 + m/8) * 2^(e-7) */
    return (float)(s ? -v : v);
}

/* ---------------------------------------------------------------- layout */

int moe_ref_layout(const int32_t* topk_idx, const float* topk_w,
                   int32_t T, int32_t K, int32_t E, int32_t R, int64_t capacity,
                   int32_t* tokens_per_expert, int32_t* expert_offset,
                   int32_t* tokens_per_rank, int32_t* rank_offset,
                   int32_t* recv_expert_offset, int32_t* recv_slot,
                   int32_t* expert_slot, int32_t* recv_src_token,
                   int32_t* expert_src_row, float* expert_weight)
{
    if (T < 0 || K <= 0 || E <= 0 || R <= 0 || E % R != 0 || capacity < 0) return MOE_REF_ERR_ARG;
    if (!topk_idx || !tokens_per_expert || !expert_offset || !tokens_per_rank || !rank_offset ||
        !recv_expert_offset || !recv_slot || !expert_slot || !recv_src_token || !expert_src_row)
        return MOE_REF_ERR_ARG;
    const int32_t m = E / R;                    /* experts per (virtual) rank */
    int err = 0;
    int32_t* primary_count = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!primary_count || !seen) { free(primary_count); free(seen); return MOE_REF_ERR_ARG; }

    /* tokens_per_expert[e] = #{(t,k) : idx[t,k] == e}; out-of-range ids are
     * flagged and then ignored like masked entries. */
    for (int32_t e = 0; e < E; ++e) tokens_per_expert[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) { err |= MOE_REF_ERR_EXPERT_ID; continue; }
            tokens_per_expert[e] += 1;
        }
    expert_offset[0] = 0;
    for (int32_t e = 0; e < E; ++e) expert_offset[e + 1] = expert_offset[e] + tokens_per_expert[e];

    /* primary expert of (t, r): the smallest valid id of token t on rank r;
     * P[e] counts the (t, r) pairs whose primary is e. */
    for (int64_t t = 0; t < T; ++t)
        for (int32_t r = 0; r < R; ++r) {
            int32_t p = -1;
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = topk_idx[t * K + k];
                if (e < 0 || e >= E || e / m != r) continue;
                if (p < 0 || e < p) p = e;
            }
            if (p >= 0) primary_count[p] += 1;
        }
    recv_expert_offset[0] = 0;
    for (int32_t e = 0; e < E; ++e) recv_expert_offset[e + 1] = recv_expert_offset[e] + primary_count[e];
    for (int32_t r = 0; r < R; ++r) {
        rank_offset[r] = recv_expert_offset[r * m];
        tokens_per_rank[r] = recv_expert_offset[(r + 1) * m] - recv_expert_offset[r * m];
    }
    rank_offset[R] = recv_expert_offset[E];
    int64_t n_pairs = recv_expert_offset[E];
    if (n_pairs > capacity) err |= MOE_REF_ERR_CAPACITY;

    /* recv_slot[t, r] = recv_expert_offset[p] + #{t' < t : p(t', r) == p}:
     * rows ordered by (primary expert, token). */
    for (int64_t i = 0; i < capacity; ++i) recv_src_token[i] = -1;
    for (int32_t e = 0; e < E; ++e) seen[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t r = 0; r < R; ++r) {
            int32_t p = -1;
            for (int32_t k = 0; k < K; ++k) {
                int32_t e = topk_idx[t * K + k];
                if (e < 0 || e >= E || e / m != r) continue;
                if (p < 0 || e < p) p = e;
            }
            int32_t slot = -1;
            if (p >= 0) {
                slot = recv_expert_offset[p] + seen[p];
                seen[p] += 1;
                if (slot < capacity) recv_src_token[slot] = (int32_t)t;
                else slot = -1;
            }
            recv_slot[t * R + r] = slot;
        }

    /* expert_slot[t, k] = expert_offset[e] + #{(t',k') < (t,k) : idx == e}:
     * expert-major rows ordered by (expert, token, k). */
    int64_t n_entries = (int64_t)T * K;
    for (int64_t i = 0; i < n_entries; ++i) {
        expert_src_row[i] = -1;
        if (topk_w && expert_weight) expert_weight[i] = 0.0f;
    }
    for (int32_t e = 0; e < E; ++e) seen[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            if (e < 0 || e >= E) { expert_slot[t * K + k] = -1; continue; }
            int32_t row = expert_offset[e] + seen[e];
            seen[e] += 1;
            expert_slot[t * K + k] = row;
            expert_src_row[row] = recv_slot[t * R + e / m];
            if (topk_w && expert_weight) expert_weight[row] = topk_w[t * K + k];
        }

    free(primary_count);
    free(seen);
    return err;
}

/* ------------------------------------------------- multi-source layout */

/* Does token g have a valid expert on rank r? */
static int reaches_rank(const int32_t* topk_idx, int64_t g, int32_t K, int32_t E, int32_t m, int32_t r)
{
    for (int32_t k = 0; k < K; ++k) {
        int32_t e = topk_idx[g * K + k];
        if (e >= 0 && e < E && e / m == r) return 1;
    }
    return 0;
}

int moe_ref_layout_sources(const int32_t* topk_idx, const float* topk_w,
                           int32_t S, int32_t Ts, int32_t K, int32_t E, int32_t R,
                           int32_t* tokens_per_expert, int32_t* expert_offset,
                           int32_t* tokens_per_rank, int32_t* rank_offset,
                           int32_t* recv_source_offset, int32_t* recv_slot,
                           int32_t* expert_slot, int32_t* recv_src_token,
                           int32_t* expert_src_row, float* expert_weight)
{
    if (S <= 0 || Ts < 0 || K <= 0 || E <= 0 || R <= 0 || E % R != 0) return MOE_REF_ERR_ARG;
    if (!topk_idx || !tokens_per_expert || !expert_offset || !tokens_per_rank || !rank_offset ||
        !recv_source_offset || !recv_slot || !expert_slot || !recv_src_token || !expert_src_row)
        return MOE_REF_ERR_ARG;
    const int32_t m = E / R;
    const int64_t T = (int64_t)S * Ts;
    int err = 0;
    int32_t* seen = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!seen) return MOE_REF_ERR_ARG;

    /* per-expert counts and offsets, as in the single-source layout */
    for (int32_t e = 0; e < E; ++e) tokens_per_expert[e] = 0;
    for (int64_t g = 0; g < T; ++g)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[g * K + k];
            if (e == -1) continue;
            if (e < -1 || e >= E) { err |= MOE_REF_ERR_EXPERT_ID; continue; }
            tokens_per_expert[e] += 1;
        }
    expert_offset[0] = 0;
    for (int32_t e = 0; e < E; ++e) expert_offset[e + 1] = expert_offset[e] + tokens_per_expert[e];

    /* destination regions: each rank walks the tokens in (source, token)
     * order and takes the ones that reach it, one row each */
    for (int64_t i = 0; i < (int64_t)R * T; ++i) recv_src_token[i] = -1;
    for (int32_t r = 0; r < R; ++r) {
        int32_t used = 0;
        for (int32_t s = 0; s < S; ++s) {
            recv_source_offset[(int64_t)r * (S + 1) + s] = used;
            for (int32_t t = 0; t < Ts; ++t) {
                int64_t g = (int64_t)s * Ts + t;
                int32_t slot = -1;
                if (reaches_rank(topk_idx, g, K, E, m, r)) {
                    slot = (int32_t)((int64_t)r * T + used);
                    recv_src_token[slot] = (int32_t)g;
                    used += 1;
                }
                recv_slot[g * R + r] = slot;
            }
        }
        recv_source_offset[(int64_t)r * (S + 1) + S] = used;
        tokens_per_rank[r] = used;
        rank_offset[r] = (int32_t)((int64_t)r * T);
    }
    rank_offset[R] = (int32_t)((int64_t)R * T);

    /* expert-major rows ordered by (expert, token, k), as in the
     * single-source layout */
    for (int64_t i = 0; i < T * K; ++i) {
        expert_src_row[i] = -1;
        if (topk_w && expert_weight) expert_weight[i] = 0.0f;
    }
    for (int64_t g = 0; g < T; ++g)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[g * K + k];
            if (e < 0 || e >= E) { expert_slot[g * K + k] = -1; continue; }
            int32_t row = expert_offset[e] + seen[e];
            seen[e] += 1;
            expert_slot[g * K + k] = row;
            expert_src_row[row] = recv_slot[g * R + e / m];
            if (topk_w && expert_weight) expert_weight[row] = topk_w[g * K + k];
        }
    free(seen);
    return err;
}

/* -------------------------------------------------------------- dispatch */

int moe_ref_dispatch_bf16(const uint16_t* x, int32_t T, int32_t H, int32_t R,
                          const int32_t* recv_slot, int64_t capacity,
                          uint16_t* recv_x)
{
    if (!x || !recv_slot || !recv_x || T < 0 || H <= 0 || R <= 0) return MOE_REF_ERR_ARG;
    int err = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t r = 0; r < R; ++r) {
            int64_t slot = recv_slot[t * R + r];
            if (slot < 0) continue;
            if (slot >= capacity) { err |= MOE_REF_ERR_CAPACITY; continue; }
            for (int64_t h = 0; h < H; ++h) recv_x[slot * H + h] = x[t * H + h];
        }
    return err;
}

int moe_ref_dispatch_fp8(const uint16_t* x, int32_t T, int32_t H, int32_t R,
                         const int32_t* recv_slot, int64_t capacity,
                         uint8_t* recv_q, float* recv_scales)
{
    if (!x || !recv_slot || !recv_q || !recv_scales || T < 0 || H <= 0 || R <= 0 || H % 128 != 0)
        return MOE_REF_ERR_ARG;
    const int32_t nb = H / 128;
    int err = 0;
    uint8_t q_row[128];
    for (int64_t t = 0; t < T; ++t)
        for (int32_t b = 0; b < nb; ++b) {
            /* amax of the block, exact (a max of magnitudes) */
            float amax = 0.0f;
            for (int32_t j = 0; j < 128; ++j) {
                float v = fabsf(moe_ref_bf16_decode(x[t * H + b * 128 + j]));
                if (v > amax) amax = v;
            }
            float s = amax / 448.0f;                          /* fp32, RN */
            for (int32_t j = 0; j < 128; ++j) {
                float v = moe_ref_bf16_decode(x[t * H + b * 128 + j]);
                q_row[j] = (amax == 0.0f) ? (uint8_t)0x00 : moe_ref_e4m3_encode(v / s);
            }
            for (int32_t r = 0; r < R; ++r) {
                int64_t slot = recv_slot[t * R + r];
                if (slot < 0) continue;
                if (slot >= capacity) { err |= MOE_REF_ERR_CAPACITY; continue; }
                memcpy(recv_q + slot * H + (int64_t)b * 128, q_row, 128);
                recv_scales[slot * nb + b] = s;
            }
        }
    return err;
}

/* OCP Microscaling (MX) formats: a block of 32 values shares one power-of-two
 * scale X = 2^shared_exp stored as an E8M0 byte (biased exponent, bias 127);
 * shared_exp is floor(log2 of the block's largest magnitude) minus the
 * exponent of the element format's largest normal (8 for E4M3), so the
 * largest element lands in [256, 512) before the element conversion, which
 * rounds to nearest even and saturates at 448.  Multiplying by a power of two
 * is exact except for results below the fp32 normal range, which ldexpf
 * rounds once. */
int moe_ref_dispatch_mxfp8(const uint16_t* x, int32_t T, int32_t H, int32_t R,
                           const int32_t* recv_slot, int64_t capacity,
                           uint8_t* recv_q, uint8_t* recv_scales)
{
    if (!x || !recv_slot || !recv_q || !recv_scales || T < 0 || H <= 0 || R <= 0 || H % 32 != 0)
        return MOE_REF_ERR_ARG;
    const int32_t nb = H / 32;
    int err = 0;
    uint8_t q_row[32];
    for (int64_t t = 0; t < T; ++t)
        for (int32_t b = 0; b < nb; ++b) {
            float amax = 0.0f;
            for (int32_t j = 0; j < 32; ++j) {
                float v = fabsf(moe_ref_bf16_decode(x[t * H + b * 32 + j]));
                if (v > amax) amax = v;
            }
            int shared_exp = -127;
            if (amax > 0.0f) {
                int e2;
                frexpf(amax, &e2);                 /* amax = f * 2^e2, f in [0.5, 1) */
                shared_exp = (e2 - 1) - 8;         /* floor(log2(amax)) - 8 */
                if (shared_exp < -127) shared_exp = -127;
                if (shared_exp > 127) shared_exp = 127;
            }
            for (int32_t j = 0; j < 32; ++j) {
                float v = moe_ref_bf16_decode(x[t * H + b * 32 + j]);
                q_row[j] = moe_ref_e4m3_encode(ldexpf(v, -shared_exp));
            }
            for (int32_t r = 0; r < R; ++r) {
                int64_t slot = recv_slot[t * R + r];
                if (slot < 0) continue;
                if (slot >= capacity) { err |= MOE_REF_ERR_CAPACITY; continue; }
                memcpy(recv_q + slot * H + (int64_t)b * 32, q_row, 32);
                recv_scales[slot * nb + b] = (uint8_t)(shared_exp + 127);
            }
        }
    return err;
}

/* --------------------------------------------------------------- combine */

int moe_ref_combine(const uint16_t* y, int64_t n_rows, int32_t T, int32_t K,
                    int32_t H, const int32_t* expert_slot, const float* topk_w,
                    uint16_t* out)
{
    if (!y || !expert_slot || !topk_w || !out || T < 0 || K <= 0 || H <= 0) return MOE_REF_ERR_ARG;
    int err = 0;
    float* acc = (float*)malloc((size_t)H * sizeof(float));
    if (!acc) return MOE_REF_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) acc[h] = 0.0f;
        /* each element's sum is the chain over k = 0, 1, ..., K-1 */
        for (int32_t k = 0; k < K; ++k) {
            int64_t row = expert_slot[t * K + k];
            if (row < 0) continue;
            if (row >= n_rows) { err |= MOE_REF_ERR_CAPACITY; continue; }
            float w = topk_w[t * K + k];
            for (int32_t h = 0; h < H; ++h)
                acc[h] = fmaf(w, moe_ref_bf16_decode(y[row * H + h]), acc[h]);
        }
        for (int32_t h = 0; h < H; ++h) out[t * H + h] = moe_ref_bf16_encode(acc[h]);
    }
    free(acc);
    return err;
}

/* -------------------------------------------------------------- backward */

/* Dispatch copies x[t] to one receive row per destination rank, so its
 * adjoint sums the gradients of those rows back into token t. */
int moe_ref_dispatch_backward(const uint16_t* grad_recv, int64_t n_rows, int32_t T, int32_t R,
                              int32_t H, const int32_t* recv_slot, uint16_t* grad_x)
{
    if (!grad_recv || !recv_slot || !grad_x || T < 0 || R <= 0 || H <= 0) return MOE_REF_ERR_ARG;
    int err = 0;
    float* acc = (float*)malloc((size_t)H * sizeof(float));
    if (!acc) return MOE_REF_ERR_ARG;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < H; ++h) acc[h] = 0.0f;
        for (int32_t r = 0; r < R; ++r) {
            int64_t row = recv_slot[t * R + r];
            if (row < 0) continue;
            if (row >= n_rows) { err |= MOE_REF_ERR_CAPACITY; continue; }
            for (int32_t h = 0; h < H; ++h) acc[h] = acc[h] + moe_ref_bf16_decode(grad_recv[row * H + h]);
        }
        for (int32_t h = 0; h < H; ++h) grad_x[t * H + h] = moe_ref_bf16_encode(acc[h]);
    }
    free(acc);
    return err;
}

/* Combine computes out[t] = sum_k w[t,k] * y[slot(t,k)]; its gradients are
 * w[t,k] * grad_out[t] for the expert rows and <grad_out[t], y[slot(t,k)]>
 * for the router weights. */
int moe_ref_combine_backward(const uint16_t* grad_out, const uint16_t* y, int64_t n_rows, int32_t T,
                             int32_t K, int32_t H, const int32_t* expert_slot, const float* topk_w,
                             uint16_t* grad_y, double* grad_w)
{
    if (!grad_out || !y || !expert_slot || !topk_w || !grad_y || !grad_w || T < 0 || K <= 0 || H <= 0)
        return MOE_REF_ERR_ARG;
    int err = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int64_t row = expert_slot[t * K + k];
            grad_w[t * K + k] = 0.0;
            if (row < 0) continue;
            if (row >= n_rows) { err |= MOE_REF_ERR_CAPACITY; continue; }
            float w = topk_w[t * K + k];
            double dot = 0.0;
            for (int32_t h = 0; h < H; ++h) {
                float g = moe_ref_bf16_decode(grad_out[t * H + h]);
                float prod = w * g;                                  /* fp32, round to nearest */
                grad_y[row * H + h] = moe_ref_bf16_encode(prod);
                dot += (double)g * (double)moe_ref_bf16_decode(y[row * H + h]);
            }
            grad_w[t * K + k] = dot;
        }
    return err;
}

/* ------------------------------------------------------------ low latency */

int moe_ref_ll_dispatch(const uint16_t* x, const int32_t* topk_idx, int32_t T, int32_t K, int32_t E,
                        int32_t H, int32_t cap, uint16_t* recv, int32_t* tokens_per_expert,
                        int32_t* ll_slot)
{
    if (!x || !topk_idx || !recv || !tokens_per_expert || !ll_slot || T < 0 || K <= 0 || E <= 0 || H <= 0 || cap < 0)
        return MOE_REF_ERR_ARG;
    int err = 0;
    for (int32_t e = 0; e < E; ++e) tokens_per_expert[e] = 0;
    for (int64_t t = 0; t < T; ++t)
        for (int32_t k = 0; k < K; ++k) {
            int32_t e = topk_idx[t * K + k];
            int32_t slot = -1;
            if (e < -1 || e >= E) {
                err |= MOE_REF_ERR_EXPERT_ID;
            } else if (e >= 0) {
                /* tokens_per_expert[e] counts the earlier entries of e so far */
                int32_t j = tokens_per_expert[e];
                if (j < cap) {
                    slot = e * cap + j;
                    tokens_per_expert[e] = j + 1;
                    memcpy(recv + (int64_t)slot * H, x + t * H, (size_t)H * sizeof(uint16_t));
                } else {
                    err |= MOE_REF_ERR_CAPACITY;
                }
            }
            ll_slot[t * K + k] = slot;
        }
    return err;
}
