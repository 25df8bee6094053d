/*
 * abi_roundtrip.c -- the C ABI of libmoe_ep.so used from plain C99 (no C++,
 * no Python, no torch): device memory from the CUDA runtime, one routing
 * layout carved from a single allocation, bf16 dispatch, an identity
 * "expert" on the host (y row j = the receive row expert_src_row[j]), and
 * combine with weights 1/K.  For every fully routed token the fp32 chain
 * 0.25x + 0.25x + 0.25x + 0.25x is exact for bf16 x, so the output must equal
 * x bit for bit; the counts must add up to the valid entries and pairs.
 * Prints "abi roundtrip ok" and exits 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "moe_ep.h"

#define T 300
#define K 4
#define E 16
#define R 4
#define H 64

#define CHECK_CUDA(call)                                                      \
    do {                                                                      \
        cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess) {                                              \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_)); \
            return 1;                                                         \
        }                                                                     \
    } while (0)

#define CHECK_MOE(call)                                                       \
    do {                                                                      \
        moe_status s_ = (call);                                               \
        if (s_ != MOE_OK) {                                                   \
            fprintf(stderr, "%s failed: %s\n", #call, moe_status_string(s_)); \
            return 1;                                                         \
        }                                                                     \
    } while (0)

static uint32_t lcg(uint32_t* state) {
    *state = *state * 1664525u + 1013904223u;
    return *state >> 8;
}

int main(void) {
    static int32_t idx[T * K];
    static float w[T * K];
    static uint16_t x[T * H], out[T * H], recv[T * R * H], y[T * K * H];
    static int32_t expert_src_row[T * K], tokens_per_expert[E], tokens_per_rank[R];
    uint32_t state = 12345u;
    int t, k, j, h;

    /* K distinct experts per token, a few entries masked */
    for (t = 0; t < T; ++t) {
        for (k = 0; k < K; ++k) {
            int e, dup;
            do {
                e = (int)(lcg(&state) % E);
                dup = 0;
                for (j = 0; j < k; ++j) dup |= idx[t * K + j] == e;
            } while (dup);
            idx[t * K + k] = e;
            w[t * K + k] = 0.25f;
        }
        if (t % 17 == 5) idx[t * K + 3] = -1;     /* masked: its weight never counts */
    }
    /* bf16 activations: small integers / 8, plus a sign (exact in bf16) */
    for (j = 0; j < T * H; ++j) {
        const uint32_t v = lcg(&state);
        const float f = (float)((int)(v % 255) - 127) / 8.0f;
        uint32_t bits;
        memcpy(&bits, &f, 4);
        x[j] = (uint16_t)(bits >> 16);            /* exact: at most 8 significant bits */
    }

    const int64_t capacity = (int64_t)T * (K < R ? K : R);
    const size_t lbytes = moe_layout_bytes(T, K, E, R, capacity);
    if (lbytes == 0) {
        fprintf(stderr, "moe_layout_bytes returned 0\n");
        return 1;
    }
    void *d_layout, *d_idx, *d_w, *d_x, *d_recv, *d_y, *d_out;
    CHECK_CUDA(cudaMalloc(&d_layout, lbytes));
    CHECK_CUDA(cudaMalloc(&d_idx, sizeof(idx)));
    CHECK_CUDA(cudaMalloc(&d_w, sizeof(w)));
    CHECK_CUDA(cudaMalloc(&d_x, sizeof(x)));
    CHECK_CUDA(cudaMalloc(&d_recv, (size_t)capacity * H * 2));
    CHECK_CUDA(cudaMalloc(&d_y, sizeof(y)));
    CHECK_CUDA(cudaMalloc(&d_out, sizeof(out)));
    CHECK_CUDA(cudaMemcpy(d_idx, idx, sizeof(idx), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_w, w, sizeof(w), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_x, x, sizeof(x), cudaMemcpyHostToDevice));

    moe_layout L;
    CHECK_MOE(moe_layout_init(&L, T, K, E, R, capacity, d_layout, lbytes));
    /* a bad argument is refused synchronously, before anything is enqueued */
    if (moe_dispatch((const uint16_t*)d_x, 12, &L, MOE_FORMAT_BF16, d_recv, NULL, NULL, NULL) != MOE_ERR_INVALID_ARG) {
        fprintf(stderr, "hidden 12 was not refused\n");
        return 1;
    }
    CHECK_MOE(moe_dispatch_layout((const int32_t*)d_idx, (const float*)d_w, E, R, &L, NULL, NULL));
    CHECK_MOE(moe_dispatch((const uint16_t*)d_x, H, &L, MOE_FORMAT_BF16, d_recv, NULL, NULL, NULL));

    /* identity expert: y row j is the receive row of its (token, rank) */
    CHECK_CUDA(cudaMemcpy(recv, d_recv, (size_t)capacity * H * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(expert_src_row, L.expert_src_row, sizeof(expert_src_row), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(tokens_per_expert, L.tokens_per_expert, sizeof(tokens_per_expert), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(tokens_per_rank, L.tokens_per_rank, sizeof(tokens_per_rank), cudaMemcpyDeviceToHost));
    int n_valid = 0, n_expert = 0, n_pairs = 0, n_reach = 0;
    for (j = 0; j < T * K; ++j) n_valid += idx[j] >= 0;
    for (j = 0; j < E; ++j) n_expert += tokens_per_expert[j];
    for (j = 0; j < R; ++j) n_pairs += tokens_per_rank[j];
    for (t = 0; t < T; ++t) {
        int seen[R] = {0};
        for (k = 0; k < K; ++k)
            if (idx[t * K + k] >= 0) seen[idx[t * K + k] / (E / R)] = 1;
        for (j = 0; j < R; ++j) n_reach += seen[j];
    }
    if (n_expert != n_valid || n_pairs != n_reach) {
        fprintf(stderr, "counts: experts %d vs %d entries, ranks %d vs %d pairs\n", n_expert, n_valid, n_pairs,
                n_reach);
        return 1;
    }
    memset(y, 0, sizeof(y));
    for (j = 0; j < n_valid; ++j) {
        const int row = expert_src_row[j];
        if (row < 0 || row >= n_pairs) {
            fprintf(stderr, "expert_src_row[%d] = %d out of range\n", j, row);
            return 1;
        }
        memcpy(y + (size_t)j * H, recv + (size_t)row * H, H * 2);
    }
    CHECK_CUDA(cudaMemcpy(d_y, y, sizeof(y), cudaMemcpyHostToDevice));
    /* masked entries never enter the sum, so a token with one gets 3/4 of x,
       which need not be a bf16 value; only fully routed tokens are compared */
    CHECK_MOE(moe_combine((const uint16_t*)d_y, H, &L, (const float*)d_w, (uint16_t*)d_out, NULL, NULL));
    uint32_t flags = 0;
    CHECK_MOE(moe_layout_read_status(&L, NULL, &flags));
    if (flags != 0) {
        fprintf(stderr, "device status flags %#x\n", flags);
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(out, d_out, sizeof(out), cudaMemcpyDeviceToHost));
    int checked = 0;
    for (t = 0; t < T; ++t) {
        if (t % 17 == 5) continue;                /* 3 of 4 entries valid: out = 0.75 x */
        for (h = 0; h < H; ++h)
            if (out[t * H + h] != x[t * H + h]) {
                fprintf(stderr, "token %d column %d: %#06x, expected %#06x\n", t, h, out[t * H + h], x[t * H + h]);
                return 1;
            }
        ++checked;
    }
    printf("abi roundtrip ok: %d tokens, %d pairs, %d entries, %d tokens compared bit for bit\n", T, n_pairs,
           n_valid, checked);
    cudaFree(d_layout); cudaFree(d_idx); cudaFree(d_w); cudaFree(d_x);
    cudaFree(d_recv); cudaFree(d_y); cudaFree(d_out);
    return 0;
}
