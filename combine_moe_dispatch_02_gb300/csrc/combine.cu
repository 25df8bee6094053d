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
    const int32_t* expert_slot;  // [T, K]: row of each (t, k), -1 = none
    const float* w;              // [T, K], or NULL for unit weights
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
    pdl_wait();
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
                ws[k] = a.w ? __ldg(a.w + t * KT + k) : 1.0f;
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
                        ws[q] = a.w ? __ldg(a.w + t * a.K + k) : 1.0f;
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
    pdl_trigger();
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

constexpr int kCombineWaves = 4;

template <int KT>
cudaError_t launch_k(const CombineArgs& a, cudaStream_t stream, int32_t num_channels) {
    const int64_t n_items = static_cast<int64_t>(a.T) * a.H8;
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_kernel<KT>, kCombineThreads, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    // four waves of resident CTAs by default: on GB300 (the whole step, three
    // full-size shapes) faster than one persistent wave and than one item per
    // thread, or within noise of the better of the two
    int64_t grid = num_channels > 0 ? num_channels : static_cast<int64_t>(sm_count()) * per_sm * kCombineWaves;
    const int64_t need = (n_items + kCombineThreads - 1) / kCombineThreads;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    // A programmatic launch: the grid may be set up while its predecessor's
    // last CTAs drain, and waits (griddepcontrol.wait) for that grid's
    // completion before it reads anything.  Against an ordinary launch after
    // the one-item-per-warp dispatch (GB300, alternating processes): the
    // dispatch + combine pair 0.3-1.1 us shorter at the DeepSeek-V3 and
    // Qwen-like shapes.  Against the earlier many-wave TMA dispatch it had
    // measured ~15% slower, which is why this was an ordinary launch before.
    return launch_pdl(combine_kernel<KT>, dim3(static_cast<unsigned>(grid)), dim3(kCombineThreads), 0, stream, a);
}

// TMA-staged variant --------------------------------------------------------
//
// Items are (token, 1024-column chunk).  A producer warp reads the token's K
// slots and weights once, then for each item waits for a free stage, posts
// the expected byte count on the stage's "full" mbarrier and issues one TMA
// bulk copy per valid entry (lane k copies row expert_slot[t,k]'s chunk).
// Four consumer warps (one 16-byte column group per thread) wait on "full",
// run the fp32 fma chain over k = 0..K-1 reading the rows from shared memory,
// store 16 bytes of output and release the stage through its "empty"
// mbarrier.  Every wait is bounded.
constexpr int kTmaCE = 1024;                        // columns per item
constexpr int kTmaConsumers = kTmaCE / 8;           // one 16-byte group per consumer thread
constexpr int kTmaThreads = 32 + kTmaConsumers;     // producer warp + 4 consumer warps
constexpr int kTmaMaxK = 8;
constexpr int kTmaStages = 4;

struct TmaStageMeta {
    float w[kTmaMaxK];
    uint32_t ok;                                    // bit k: entry k has a valid row
};

__global__ void __launch_bounds__(kTmaThreads)
combine_tma_kernel(CombineArgs a, uint64_t timeout_ns) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kTmaStages;
    TmaStageMeta* meta = reinterpret_cast<TmaStageMeta*>(smem + 16 * kTmaStages);
    uint8_t* stage0 = smem + align_up(16 * kTmaStages + sizeof(TmaStageMeta) * kTmaStages, 128);
    const size_t stage_bytes = static_cast<size_t>(a.K) * kTmaCE * 2;
    const int H = a.H8 * 8;
    const int nchunk = (H + kTmaCE - 1) / kTmaCE;
    const int64_t n_items = static_cast<int64_t>(a.T) * nchunk;
    const int64_t i0 = n_items * blockIdx.x / gridDim.x;
    const int n = static_cast<int>(n_items * (blockIdx.x + 1) / gridDim.x - i0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (n <= 0) return;
    if (tid == 0) {
        for (int s = 0; s < kTmaStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kTmaConsumers / 32);
        }
        fence_mbar_init();
    }
    __syncthreads();
    bool bad = false, timed_out = false;
    int issued = 0;                                 // producer: items whose loads were posted

    if (warp == 0) {
        // ---------------- producer
        int64_t cur_t = -1;
        int32_t slot = -1;
        float wk = 0.0f;
        uint32_t ok = 0;
        for (int i = 0; i < n; ++i) {
            const int s = i % kTmaStages;
            const int64_t item = i0 + i;
            const int64_t t = item / nchunk;
            const int c = static_cast<int>(item - t * nchunk);
            if (t != cur_t) {
                cur_t = t;
                slot = lane < a.K ? __ldg(a.expert_slot + t * a.K + lane) : -1;
                wk = lane < a.K ? __ldg(a.w + t * a.K + lane) : 0.0f;
                bad |= slot >= a.n_rows;
                ok = __ballot_sync(0xffffffffu, slot >= 0 && slot < a.n_rows);
            }
            if (i >= kTmaStages) {
                const bool got = mbar_wait_bounded(&empty[s], static_cast<uint32_t>(i / kTmaStages - 1) & 1u, timeout_ns);
                if (__any_sync(0xffffffffu, !got)) { timed_out = true; break; }
            }
            const int elems = min(kTmaCE, H - c * kTmaCE);
            const uint32_t bytes = static_cast<uint32_t>(elems) * 2u;
            if (lane < a.K) meta[s].w[lane] = wk;
            if (lane == 0) meta[s].ok = ok;
            __syncwarp();
            if (lane == 0) mbar_arrive_expect_tx(&full[s], bytes * __popc(ok));
            __syncwarp();
            if ((ok >> lane) & 1u)
                bulk_g2s(stage0 + s * stage_bytes + static_cast<size_t>(lane) * kTmaCE * 2,
                         reinterpret_cast<const uint8_t*>(a.y) + (static_cast<int64_t>(slot) * H + c * kTmaCE) * 2,
                         bytes, &full[s]);
            ++issued;
        }
    } else {
        // ---------------- consumers
        const int j = tid - 32;                     // 16-byte column group within the chunk
        for (int i = 0; i < n; ++i) {
            const int s = i % kTmaStages;
            const int64_t item = i0 + i;
            const int64_t t = item / nchunk;
            const int c = static_cast<int>(item - t * nchunk);
            const bool got = mbar_wait_bounded(&full[s], static_cast<uint32_t>(i / kTmaStages) & 1u, timeout_ns);
            if (__any_sync(0xffffffffu, !got)) { timed_out = true; break; }
            const int elems = min(kTmaCE, H - c * kTmaCE);
            const uint32_t ok = meta[s].ok;
            if (j * 8 < elems) {
                float acc[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
                const uint8_t* st = stage0 + s * stage_bytes + j * 16;
                for (int k = 0; k < a.K; ++k) {
                    if (!((ok >> k) & 1u)) continue;
                    const uint4 v = *reinterpret_cast<const uint4*>(st + static_cast<size_t>(k) * kTmaCE * 2);
                    fma8(acc, meta[s].w[k], v);
                }
                st_stream_v4(a.out + t * a.H8 + c * (kTmaCE / 8) + j, pack8(acc));
            }
            __syncwarp();
            if (lane == 0) {
                asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(&empty[s])) : "memory");
            }
        }
    }
    // after a timeout on either side, the producer waits (bounded) for the
    // loads it posted before the CTA's shared memory goes away
    const bool any_timeout = __syncthreads_or(timed_out);
    if (any_timeout && warp == 0) drain_ring_loads(full, kTmaStages, issued, timeout_ns);
    pdl_trigger();
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
    if (any_timeout && tid == 0) atomicOr(a.status, MOE_DEVERR_TIMEOUT);
}

}  // namespace

// Backward of the bf16 dispatch: the same gather with unit weights over the
// token's receive rows (recv_slot[t, 0..R)), ascending rank order.  With
// weight 1 the fused multiply-add chain is an fp32 add chain.
cudaError_t launch_dispatch_backward(const uint16_t* grad_recv, int32_t hidden, const moe_layout* L,
                                     uint16_t* grad_x, cudaStream_t stream, int32_t num_channels) {
    if (L->T == 0) return cudaSuccess;
    if (gather_wide_supported(grad_recv, grad_x, hidden))
        return launch_gather_wide(grad_recv, L->recv_slot, nullptr, L->T, L->R, L->capacity, hidden, grad_x,
                                  L->status, stream, num_channels);
    CombineArgs a;
    a.y = reinterpret_cast<const uint4*>(grad_recv);
    a.expert_slot = L->recv_slot;
    a.w = nullptr;
    a.out = reinterpret_cast<uint4*>(grad_x);
    a.T = L->T; a.K = L->R; a.H8 = hidden / 8;
    a.n_rows = L->capacity;
    a.status = L->status;
    switch (L->R) {
        case 1: return launch_k<1>(a, stream, num_channels);
        case 2: return launch_k<2>(a, stream, num_channels);
        case 4: return launch_k<4>(a, stream, num_channels);
        case 8: return launch_k<8>(a, stream, num_channels);
        default: return launch_k<0>(a, stream, num_channels);
    }
}

// Combine over the low-latency layout: the same weighted gather, with the
// slot map ll_slot into y [E * cap, H].
cudaError_t launch_ll_combine(const uint16_t* y, const int32_t* ll_slot, const float* topk_w, int32_t T, int32_t K,
                              int64_t n_rows, int32_t hidden, uint16_t* out, uint32_t* status, cudaStream_t stream,
                              int32_t num_channels) {
    if (T == 0) return cudaSuccess;
    CombineArgs a;
    a.y = reinterpret_cast<const uint4*>(y);
    a.expert_slot = ll_slot;
    a.w = topk_w;
    a.out = reinterpret_cast<uint4*>(out);
    a.T = T; a.K = K; a.H8 = hidden / 8;
    a.n_rows = n_rows;
    a.status = status;
    switch (K) {
        case 1: return launch_k<1>(a, stream, num_channels);
        case 2: return launch_k<2>(a, stream, num_channels);
        case 4: return launch_k<4>(a, stream, num_channels);
        case 6: return launch_k<6>(a, stream, num_channels);
        case 8: return launch_k<8>(a, stream, num_channels);
        default: return launch_k<0>(a, stream, num_channels);
    }
}

cudaError_t launch_combine(const uint16_t* y, int32_t hidden, const moe_layout* L, const float* topk_w,
                           uint16_t* out, cudaStream_t stream, int32_t num_channels, int32_t variant,
                           uint64_t timeout_ns) {
    if (L->T == 0) return cudaSuccess;
    CombineArgs a;
    a.y = reinterpret_cast<const uint4*>(y);
    a.expert_slot = L->expert_slot;
    a.w = topk_w;
    a.out = reinterpret_cast<uint4*>(out);
    a.T = L->T; a.K = L->K; a.H8 = hidden / 8;
    a.n_rows = static_cast<int64_t>(L->T) * L->K;
    a.status = L->status;
    if (variant == 4 && gather_wide_supported(y, out, hidden))
        return launch_gather_wide(y, L->expert_slot, topk_w, L->T, L->K, a.n_rows, hidden, out, L->status, stream,
                                  num_channels);
    if (variant == 1 && L->K <= kTmaMaxK) {
        const size_t smem = align_up(16 * kTmaStages + sizeof(TmaStageMeta) * kTmaStages, 128) +
                            static_cast<size_t>(kTmaStages) * L->K * kTmaCE * 2;
        cudaError_t err = cudaFuncSetAttribute(combine_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
        if (err != cudaSuccess) return err;
        int per_sm = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, combine_tma_kernel, kTmaThreads, smem);
        if (err != cudaSuccess) return err;
        if (per_sm < 1) per_sm = 1;
        const int64_t n_items = static_cast<int64_t>(L->T) * ((hidden + kTmaCE - 1) / kTmaCE);
        int64_t grid = num_channels > 0 ? num_channels : static_cast<int64_t>(sm_count()) * per_sm;
        if (grid > n_items) grid = n_items;
        if (grid < 1) grid = 1;
        combine_tma_kernel<<<static_cast<unsigned>(grid), kTmaThreads, smem, stream>>>(a, timeout_ns);
        return cudaGetLastError();
    }
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
