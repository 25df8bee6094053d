// combine.cu -- MoE combine: gather the expert outputs of every token back to
// its position and sum them with the router weights.
//
// out[t, :] = bf16_rne( fma chain over k = 0..K-1 of topk_w[t,k] * y[expert_slot[t,k], :] )
// in fp32, starting from 0, skipping masked entries ("Inside the Nebius +
// PyTorch DeepSeek V3 recipe", section "Mixture-of-experts and wide expert
// parallelism": combine returns expert outputs to their original positions;
// the weighted fp32 sum emitted as bf16 is the reading documented in moe_ep.h).
//
// HBM-bound gather: each thread owns one 16-byte column group (8 bf16) of one
// token, issues the K row loads of that group back to back (K x 16 bytes in
// flight per thread), then runs the fma chain in ascending k and writes 16
// bytes.  Consecutive threads cover consecutive column groups of the same
// token, so every load and store instruction of a warp touches 512
// contiguous bytes.  y is read exactly once (streaming, evict-first) and out
// written once.
#include <cuda_bf16.h>

#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kCombineThreads = 256;

struct CombineArgs {
    const uint4* y;              // [n_rows, H/8] of 8 x bf16
    const int32_t* expert_slot;  // [T, K]
    const float* w;              // [T, K]
    uint4* out;                  // [T, H/8]
    int32_t T, K, H8;
    int64_t n_rows;
    uint32_t* status;
};

__device__ __forceinline__ void fma8(float (&acc)[8], float w, uint4 v) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc[2 * j] = __fmaf_rn(w, __uint_as_float(u[j] << 16), acc[2 * j]);
        acc[2 * j + 1] = __fmaf_rn(w, __uint_as_float(u[j] & 0xffff0000u), acc[2 * j + 1]);
    }
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
    uint32_t u[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        u[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}

// KT > 0: compile-time top-k; KT == 0: runtime K (up to MOE_MAX_TOPK), loaded
// in groups of 8.
template <int KT>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(CombineArgs a) {
    const int64_t n_items = static_cast<int64_t>(a.T) * a.H8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kCombineThreads;
    bool bad = false;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * kCombineThreads + threadIdx.x; it < n_items; it += stride) {
        const int64_t t = it / a.H8;
        const int64_t v = it - t * a.H8;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        if constexpr (KT > 0) {
            uint4 vals[KT];
            float ws[KT];
            bool ok[KT];
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                const int32_t slot = __ldg(a.expert_slot + t * KT + k);
                ws[k] = __ldg(a.w + t * KT + k);
                ok[k] = slot >= 0 && slot < a.n_rows;
                bad |= slot >= a.n_rows;
                vals[k] = ok[k] ? ld_stream_v4(a.y + static_cast<int64_t>(slot) * a.H8 + v) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < KT; ++k)
                if (ok[k]) fma8(acc, ws[k], vals[k]);
        } else {
            for (int k0 = 0; k0 < a.K; k0 += 8) {
                uint4 vals[8];
                float ws[8];
                bool ok[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int k = k0 + q;
                    ok[q] = false;
                    ws[q] = 0.0f;
                    vals[q] = make_uint4(0, 0, 0, 0);
                    if (k < a.K) {
                        const int32_t slot = __ldg(a.expert_slot + t * a.K + k);
                        ws[q] = __ldg(a.w + t * a.K + k);
                        ok[q] = slot >= 0 && slot < a.n_rows;
                        bad |= slot >= a.n_rows;
                        if (ok[q]) vals[q] = ld_stream_v4(a.y + static_cast<int64_t>(slot) * a.H8 + v);
                    }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    if (ok[q]) fma8(acc, ws[q], vals[q]);
            }
        }
        st_stream_v4(a.out + it, pack8(acc));
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

template <int KT>
cudaError_t launch_k(const CombineArgs& a, cudaStream_t stream, int32_t num_channels) {
    const int64_t n_items = static_cast<int64_t>(a.T) * a.H8;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<KT>, kCombineThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = num_channels > 0 ? num_channels : static_cast<int64_t>(sm_count()) * per_sm;
    const int64_t need = (n_items + kCombineThreads - 1) / kCombineThreads;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    combine_kernel<KT><<<static_cast<unsigned>(grid), kCombineThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_combine(const uint16_t* y, int32_t hidden, const moe_layout* L, const float* topk_w,
                           uint16_t* out, cudaStream_t stream, int32_t num_channels) {
    if (L->T == 0) return cudaSuccess;
    CombineArgs a;
    a.y = reinterpret_cast<const uint4*>(y);
    a.expert_slot = L->expert_slot;
    a.w = topk_w;
    a.out = reinterpret_cast<uint4*>(out);
    a.T = L->T; a.K = L->K; a.H8 = hidden / 8;
    a.n_rows = static_cast<int64_t>(L->T) * L->K;
    a.status = L->status;
    switch (L->K) {
        case 1: return launch_k<1>(a, stream, num_channels);
        case 2: return launch_k<2>(a, stream, num_channels);
        case 4: return launch_k<4>(a, stream, num_channels);
        case 6: return launch_k<6>(a, stream, num_channels);
        case 8: return launch_k<8>(a, stream, num_channels);
        default: return launch_k<0>(a, stream, num_channels);
    }
}

}  // namespace moe
