// backward.cu -- backward of the combine: the gradients of the expert outputs
// and of the router weights.
//
// The combine computes out[t] = sum_k w[t,k] * y[slot(t,k)] (moe_ep.h); MoE
// training needs its adjoint (the pages' workload is training: Hybrid-EP
// news article, "Efficiency Numbers"; "MoE / Hybrid-EP Validation",
// "Expected results"):
//   grad_y[slot(t,k), :] = bf16_rne(fp32(w[t,k] * grad_out[t, :]))
//   grad_w[t, k]         = sum_h grad_out[t, h] * y[slot(t,k), h]   (fp32)
//
// One CTA per token.  Each thread owns 16-byte column groups of the row: it
// loads grad_out once, then for every group the K expert rows back to back
// (K x 16 bytes in flight), writes the K scaled gradient groups and keeps K
// partial dot products (fused multiply-adds in column order).  The K dot
// products are then reduced across the CTA in a fixed order (warp butterfly,
// then the warps in index order), so the result is deterministic.  Bytes:
// grad_out read once, each expert row read once, each gradient row written
// once.
#include <climits>

#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kBwdThreads = 128;
constexpr int kBwdMaxK = 8;          // larger K: groups of 8 entries

struct CombineBwdArgs {
    const uint4* grad_out;           // [T, H/8]
    const uint4* y;                  // [n_rows, H/8]
    const int32_t* expert_slot;      // [T, K]
    const float* w;                  // [T, K]
    uint4* grad_y;                   // [n_rows, H/8]
    float* grad_w;                   // [T, K]
    int32_t T, K, H8;
    int64_t n_rows;
    uint32_t* status;
};

__device__ __forceinline__ uint4 scale8(uint4 g, float w) {
    const uint32_t u[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(__fmul_rn(w, __uint_as_float(u[j] << 16)),
                                                       __fmul_rn(w, __uint_as_float(u[j] & 0xffff0000u)));
        o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float dot8(uint4 g, uint4 y, float acc) {
    const uint32_t ug[4] = {g.x, g.y, g.z, g.w};
    const uint32_t uy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc = __fmaf_rn(__uint_as_float(ug[j] << 16), __uint_as_float(uy[j] << 16), acc);
        acc = __fmaf_rn(__uint_as_float(ug[j] & 0xffff0000u), __uint_as_float(uy[j] & 0xffff0000u), acc);
    }
    return acc;
}

__global__ void __launch_bounds__(kBwdThreads)
combine_backward_kernel(CombineBwdArgs a) {
    pdl_wait();
    __shared__ float s_part[kBwdThreads / 32][kBwdMaxK];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    bool bad = false;
    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        for (int k0 = 0; k0 < a.K; k0 += kBwdMaxK) {
            const int nk = min(kBwdMaxK, a.K - k0);
            int32_t slot[kBwdMaxK];
            float wk[kBwdMaxK], part[kBwdMaxK];
#pragma unroll
            for (int q = 0; q < kBwdMaxK; ++q) {
                slot[q] = -1;
                wk[q] = 0.0f;
                part[q] = 0.0f;
                if (q < nk) {
                    const int32_t s = __ldg(a.expert_slot + t * a.K + k0 + q);
                    bad |= s >= a.n_rows;
                    slot[q] = (s >= 0 && s < a.n_rows) ? s : -1;
                    wk[q] = __ldg(a.w + t * a.K + k0 + q);
                }
            }
            for (int v = tid; v < a.H8; v += kBwdThreads) {
                const uint4 g = ld_stream_v4(a.grad_out + t * a.H8 + v);
                uint4 yv[kBwdMaxK];
#pragma unroll
                for (int q = 0; q < kBwdMaxK; ++q)
                    yv[q] = slot[q] >= 0 ? ld_stream_v4(a.y + static_cast<int64_t>(slot[q]) * a.H8 + v)
                                         : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int q = 0; q < kBwdMaxK; ++q) {
                    if (slot[q] < 0) continue;
                    part[q] = dot8(g, yv[q], part[q]);
                    st_stream_v4(a.grad_y + static_cast<int64_t>(slot[q]) * a.H8 + v, scale8(g, wk[q]));
                }
            }
            // deterministic reduction of the nk dot products
#pragma unroll
            for (int q = 0; q < kBwdMaxK; ++q) {
                float p = part[q];
#pragma unroll
                for (int d = 16; d >= 1; d >>= 1) p += __shfl_xor_sync(0xffffffffu, p, d);
                if (lane == 0) s_part[warp][q] = p;
            }
            __syncthreads();
            if (tid < nk) {
                float sum = 0.0f;
                for (int w8 = 0; w8 < kBwdThreads / 32; ++w8) sum += s_part[w8][tid];
                const int32_t s = __ldg(a.expert_slot + t * a.K + k0 + tid);
                a.grad_w[t * a.K + k0 + tid] = (s >= 0 && s < a.n_rows) ? sum : 0.0f;
            }
            __syncthreads();
        }
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

}  // namespace

cudaError_t launch_combine_backward(const uint16_t* grad_out, const uint16_t* y, int32_t hidden, const moe_layout* L,
                                    const float* topk_w, uint16_t* grad_y, float* grad_w, cudaStream_t stream,
                                    int32_t num_channels) {
    if (L->T == 0) return cudaSuccess;
    CombineBwdArgs a;
    a.grad_out = reinterpret_cast<const uint4*>(grad_out);
    a.y = reinterpret_cast<const uint4*>(y);
    a.expert_slot = L->expert_slot;
    a.w = topk_w;
    a.grad_y = reinterpret_cast<uint4*>(grad_y);
    a.grad_w = grad_w;
    a.T = L->T; a.K = L->K; a.H8 = hidden / 8;
    a.n_rows = static_cast<int64_t>(L->T) * L->K;
    a.status = L->status;
    int64_t grid = num_channels > 0 ? num_channels : L->T;
    if (grid > L->T) grid = L->T;
    if (grid < 1) grid = 1;
    if (grid > INT32_MAX) grid = INT32_MAX;
    combine_backward_kernel<<<static_cast<unsigned>(grid), kBwdThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
