// dispatch.cu -- MoE token dispatch into the packed receive buffer.
//
// Every token row is written once per destination (virtual) rank, to the
// receive row recv_slot[t, r] computed by the layout ("Inside the Nebius +
// PyTorch DeepSeek V3 recipe", section "Mixture-of-experts and wide expert
// parallelism": dispatch sends tokens to their assigned experts' ranks).
// Optionally the row is quantised to FP8 E4M3 with one fp32 scale per 1x128
// block in the same pass ("MoE / Hybrid-EP Validation", section "FP8 dispatch
// restriction"; recipe documented in moe_ep.h).
//
// Structure (Hybrid-EP news article, "Technical Structure": each CUDA block is
// an independent channel that pushes chunks through pipeline stages without
// cross-block synchronisation):
//   * the grid is a set of channels; channel b owns a contiguous range of
//     (token, column-chunk) items;
//   * a TMA bulk copy brings each item's source row chunk into a shared-memory
//     stage (mbarrier transaction counting), `stages` items ahead;
//   * bf16: one TMA bulk store per destination row streams the stage back out
//     (lanes of the warp issue the stores of different ranks in parallel);
//   * FP8: the CTA's warps compute block amax, scale and E4M3 codes into an
//     output stage, which TMA bulk stores send to every destination row; the
//     scales go out with plain stores.
// x is read from HBM once; the receive rows are written once each.
#include <cuda_fp8.h>

#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kMaxStages = 8;
constexpr int kSlotBatchInts = 2048;     // recv_slot entries staged per batch
constexpr int kFp8Threads = 128;

struct DispatchArgs {
    const uint8_t* x;            // bf16 [T, H]
    uint8_t* recv;               // bf16 or E4M3 [capacity, H]
    float* recv_scales;          // [capacity, H/128] (FP8 only)
    const int32_t* recv_slot;    // [T, R]
    int32_t T, H, R;
    int64_t capacity;
    int32_t nchunk, chunk_elems; // each row split into nchunk chunks of chunk_elems (last one shorter)
    int32_t stages;
    int32_t slot_batch;          // tokens whose recv_slot rows are staged at once
    uint32_t* status;
    uint64_t timeout_ns;
};

struct ItemRange {
    int64_t i0;
    int n;
};

__device__ __forceinline__ ItemRange channel_items(const DispatchArgs& a) {
    const int64_t n_items = static_cast<int64_t>(a.T) * a.nchunk;
    const int64_t i0 = n_items * blockIdx.x / gridDim.x;
    const int64_t i1 = n_items * (blockIdx.x + 1) / gridDim.x;
    return {i0, static_cast<int>(i1 - i0)};
}

__device__ __forceinline__ void smem_carve(uint8_t* smem, const DispatchArgs& a, uint64_t** bars,
                                           int32_t** slots, uint8_t** after) {
    *bars = reinterpret_cast<uint64_t*>(smem);
    *slots = reinterpret_cast<int32_t*>(smem + 8 * kMaxStages);
    const size_t used = 8 * kMaxStages + sizeof(int32_t) * static_cast<size_t>(a.slot_batch) * a.R;
    *after = smem + align_up(used, 128);
}

// bf16 -------------------------------------------------------------------

__global__ void __launch_bounds__(32)
dispatch_bf16_kernel(DispatchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const ItemRange rg = channel_items(a);
    if (rg.n <= 0) return;
    uint64_t* bars;
    int32_t* s_slots;
    uint8_t* stage0;
    smem_carve(smem, a, &bars, &s_slots, &stage0);
    const int lane = threadIdx.x;
    const int S = a.stages;
    const uint32_t stage_bytes = static_cast<uint32_t>(a.chunk_elems) * 2u;
    const int64_t row_bytes = static_cast<int64_t>(a.H) * 2;

    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    auto issue_load = [&](int k) {
        const int64_t i = rg.i0 + k;
        const int64_t t = i / a.nchunk;
        const int c = static_cast<int>(i - t * a.nchunk);
        const int s = k % S;
        const uint32_t bytes = static_cast<uint32_t>(min(a.chunk_elems, a.H - c * a.chunk_elems)) * 2u;
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_g2s(stage0 + static_cast<size_t>(s) * stage_bytes,
                 a.x + t * row_bytes + static_cast<int64_t>(c) * a.chunk_elems * 2, bytes, &bars[s]);
    };
    if (lane == 0) {
        for (int k = 0; k < S && k < rg.n; ++k) issue_load(k);
    }

    const int64_t last_token = (rg.i0 + rg.n - 1) / a.nchunk;
    int64_t batch_t0 = 0, batch_t1 = -1;
    bool bad = false, timed_out = false;
    for (int k = 0; k < rg.n; ++k) {
        const int64_t i = rg.i0 + k;
        const int64_t t = i / a.nchunk;
        const int c = static_cast<int>(i - t * a.nchunk);
        const int s = k % S;
        if (t >= batch_t1) {
            batch_t0 = t;
            batch_t1 = min(t + a.slot_batch, last_token + 1);
            __syncwarp();
            const int cnt = static_cast<int>(batch_t1 - batch_t0) * a.R;
            for (int j = lane; j < cnt; j += 32) s_slots[j] = __ldg(a.recv_slot + batch_t0 * a.R + j);
            __syncwarp();
        }
        const bool ok = mbar_wait_bounded(&bars[s], static_cast<uint32_t>(k / S) & 1u, a.timeout_ns);
        if (__any_sync(0xffffffffu, !ok)) {   // warp-uniform exit
            timed_out = true;
            break;
        }
        const uint32_t bytes = static_cast<uint32_t>(min(a.chunk_elems, a.H - c * a.chunk_elems)) * 2u;
        const int32_t* trow = s_slots + (t - batch_t0) * a.R;
        for (int r = lane; r < a.R; r += 32) {
            const int32_t slot = trow[r];
            if (slot < 0) continue;
            if (slot >= a.capacity) { bad = true; continue; }
            bulk_s2g(a.recv + static_cast<int64_t>(slot) * row_bytes + static_cast<int64_t>(c) * a.chunk_elems * 2,
                     stage0 + static_cast<size_t>(s) * stage_bytes, bytes);
        }
        bulk_commit();
        // refill the stage consumed one step earlier once its stores have read it
        if (k >= 1 && k - 1 + S < rg.n) {
            bulk_wait_read<1>();
            __syncwarp();
            if (lane == 0) issue_load(k - 1 + S);
        }
    }
    bulk_wait_all();
    const uint32_t any_bad = __ballot_sync(0xffffffffu, bad);
    const uint32_t any_tmo = __ballot_sync(0xffffffffu, timed_out);
    if (lane == 0) {
        if (any_bad) atomicOr(a.status, MOE_DEVERR_CAPACITY);
        if (any_tmo) atomicOr(a.status, MOE_DEVERR_TIMEOUT);
    }
}

// FP8 E4M3 ------------------------------------------------------------------

__device__ __forceinline__ uint32_t quantize4(uint2 raw, float s, bool zero_block) {
    // four bf16 values -> four E4M3 bytes (element 0 in the lowest byte)
    if (zero_block) return 0u;
    const float v0 = __uint_as_float(raw.x << 16), v1 = __uint_as_float(raw.x & 0xffff0000u);
    const float v2 = __uint_as_float(raw.y << 16), v3 = __uint_as_float(raw.y & 0xffff0000u);
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(v0, s), __fdiv_rn(v1, s)), __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(v2, s), __fdiv_rn(v3, s)), __NV_SATFINITE, __NV_E4M3);
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__global__ void __launch_bounds__(kFp8Threads)
dispatch_fp8_kernel(DispatchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    const ItemRange rg = channel_items(a);
    if (rg.n <= 0) return;
    uint64_t* bars;
    int32_t* s_slots;
    uint8_t* rest;
    smem_carve(smem, a, &bars, &s_slots, &rest);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int S = a.stages;
    const int nbc = a.chunk_elems / 128;                   // blocks per chunk
    const int nb_row = a.H / 128;
    float* s_scale = reinterpret_cast<float*>(rest);       // [S][nbc]
    uint8_t* stage_in = rest + align_up(sizeof(float) * S * nbc, 128);
    const uint32_t in_bytes = static_cast<uint32_t>(a.chunk_elems) * 2u;
    uint8_t* stage_out = stage_in + static_cast<size_t>(S) * in_bytes;
    const uint32_t out_bytes = static_cast<uint32_t>(a.chunk_elems);
    const int64_t x_row_bytes = static_cast<int64_t>(a.H) * 2;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto issue_load = [&](int k) {
        const int64_t i = rg.i0 + k;
        const int64_t t = i / a.nchunk;
        const int c = static_cast<int>(i - t * a.nchunk);
        const int s = k % S;
        const uint32_t bytes = static_cast<uint32_t>(min(a.chunk_elems, a.H - c * a.chunk_elems)) * 2u;
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_g2s(stage_in + static_cast<size_t>(s) * in_bytes,
                 a.x + t * x_row_bytes + static_cast<int64_t>(c) * a.chunk_elems * 2, bytes, &bars[s]);
    };
    if (tid == 0) {
        for (int k = 0; k < S && k < rg.n; ++k) issue_load(k);
    }

    const int64_t last_token = (rg.i0 + rg.n - 1) / a.nchunk;
    int64_t batch_t0 = 0, batch_t1 = -1;
    bool bad = false, timed_out = false;
    for (int k = 0; k < rg.n; ++k) {
        const int64_t i = rg.i0 + k;
        const int64_t t = i / a.nchunk;
        const int c = static_cast<int>(i - t * a.nchunk);
        const int s = k % S;
        const int elems = min(a.chunk_elems, a.H - c * a.chunk_elems);
        const int nb = elems / 128;
        if (t >= batch_t1) {
            batch_t0 = t;
            batch_t1 = min(t + a.slot_batch, last_token + 1);
            __syncthreads();
            const int cnt = static_cast<int>(batch_t1 - batch_t0) * a.R;
            for (int j = tid; j < cnt; j += kFp8Threads) s_slots[j] = __ldg(a.recv_slot + batch_t0 * a.R + j);
        }
        // the output stage of item k-S must have been read by its bulk stores
        if (warp == 0 && k >= S) bulk_wait_read_n(S - 1);
        const bool ok = mbar_wait_bounded(&bars[s], static_cast<uint32_t>(k / S) & 1u, a.timeout_ns);
        if (__syncthreads_or(!ok)) { timed_out = true; break; }

        // quantise: warp w takes blocks w, w+4, ...; lane holds 4 consecutive values
        const uint8_t* in = stage_in + static_cast<size_t>(s) * in_bytes;
        uint8_t* out = stage_out + static_cast<size_t>(s) * out_bytes;
        for (int b = warp; b < nb; b += kFp8Threads / 32) {
            const uint2 raw = *reinterpret_cast<const uint2*>(in + (b * 128 + lane * 4) * 2);
            float amax = fmaxf(fmaxf(fabsf(__uint_as_float(raw.x << 16)), fabsf(__uint_as_float(raw.x & 0xffff0000u))),
                               fmaxf(fabsf(__uint_as_float(raw.y << 16)), fabsf(__uint_as_float(raw.y & 0xffff0000u))));
#pragma unroll
            for (int d = 16; d >= 1; d >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, d));
            const float sc = __fdiv_rn(amax, 448.0f);
            *reinterpret_cast<uint32_t*>(out + b * 128 + lane * 4) = quantize4(raw, sc, amax == 0.0f);
            if (lane == 0) s_scale[s * nbc + b] = sc;
        }
        fence_proxy_async_smem();
        __syncthreads();
        // the input stage is free again: fetch item k+S into it
        if (tid == 0 && k + S < rg.n) {
            fence_proxy_async_smem();
            issue_load(k + S);
        }
        const int32_t* trow = s_slots + (t - batch_t0) * a.R;
        if (warp == 0) {
            for (int r = lane; r < a.R; r += 32) {
                const int32_t slot = trow[r];
                if (slot < 0) continue;
                if (slot >= a.capacity) { bad = true; continue; }
                bulk_s2g(a.recv + static_cast<int64_t>(slot) * a.H + static_cast<int64_t>(c) * a.chunk_elems,
                         out, static_cast<uint32_t>(elems));
            }
            bulk_commit();
        }
        for (int j = tid; j < a.R * nb; j += kFp8Threads) {
            const int r = j / nb, b = j - r * nb;
            const int32_t slot = trow[r];
            if (slot < 0 || slot >= a.capacity) continue;
            a.recv_scales[static_cast<int64_t>(slot) * nb_row + c * nbc + b] = s_scale[s * nbc + b];
        }
    }
    if (warp == 0) bulk_wait_all();
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
    if (timed_out && tid == 0) atomicOr(a.status, MOE_DEVERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_dispatch(const uint16_t* x, int32_t hidden, const moe_layout* L, bool fp8,
                            void* recv_x, float* recv_scales, cudaStream_t stream,
                            int32_t num_channels, int32_t stages, uint64_t timeout_ns) {
    if (L->T == 0) return cudaSuccess;
    DispatchArgs a;
    a.x = reinterpret_cast<const uint8_t*>(x);
    a.recv = static_cast<uint8_t*>(recv_x);
    a.recv_scales = recv_scales;
    a.recv_slot = L->recv_slot;
    a.T = L->T; a.H = hidden; a.R = L->R;
    a.capacity = L->capacity;
    a.status = L->status;
    a.timeout_ns = timeout_ns;
    // column chunks: at most 16 KB of bf16 input per stage
    const int32_t max_elems = 8192;
    const int32_t gran = fp8 ? 128 : 8;
    a.nchunk = (hidden + max_elems - 1) / max_elems;
    a.chunk_elems = ((hidden + a.nchunk - 1) / a.nchunk + gran - 1) / gran * gran;
    a.slot_batch = kSlotBatchInts / L->R;
    if (a.slot_batch < 1) a.slot_batch = 1;
    int S = stages > 0 ? stages : (fp8 ? 3 : 4);
    if (S < 2) S = 2;
    if (S > kMaxStages) S = kMaxStages;
    a.stages = S;

    size_t smem = align_up(8 * kMaxStages + sizeof(int32_t) * static_cast<size_t>(a.slot_batch) * a.R, 128);
    if (fp8) {
        const int nbc = a.chunk_elems / 128;
        smem += align_up(sizeof(float) * S * nbc, 128) + static_cast<size_t>(S) * a.chunk_elems * 3;
    } else {
        smem += static_cast<size_t>(S) * a.chunk_elems * 2;
    }
    const void* fn = fp8 ? reinterpret_cast<const void*>(dispatch_fp8_kernel)
                         : reinterpret_cast<const void*>(dispatch_bf16_kernel);
    const int threads = fp8 ? kFp8Threads : 32;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t n_items = static_cast<int64_t>(L->T) * a.nchunk;
    int64_t grid = num_channels > 0 ? num_channels : static_cast<int64_t>(sm_count()) * per_sm;
    if (grid > n_items) grid = n_items;
    if (grid < 1) grid = 1;
    if (fp8) dispatch_fp8_kernel<<<static_cast<unsigned>(grid), threads, smem, stream>>>(a);
    else dispatch_bf16_kernel<<<static_cast<unsigned>(grid), threads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
