// gather_wide.cu -- weighted row gather with 32-byte vector accesses: the
// combine (out[t] = sum_k w[t,k] * y[expert_slot[t,k]]) and the backward of
// the bf16 dispatch (grad_x[t] = sum_r grad_recv[recv_slot[t,r]], unit
// weights) -- the operators of combine.cu ("Inside the Nebius + PyTorch
// DeepSeek V3 recipe", section "Mixture-of-experts and wide expert
// parallelism": combine returns the expert outputs to their tokens' positions),
// with the work split of the 32-byte dispatch (dispatch_wide.cu):
//
//   * an item is one 512-column segment of one token and belongs to one warp;
//     lane l owns the 16 consecutive columns 16l .. 16l+15 of the segment and
//     reads them from each source row with one 32-byte load, so a warp load
//     instruction covers 1 KB of one row (32 whole sectors);
//   * the token's slot row is read once per item: lane k holds slot k, and a
//     ballot leaves the valid ones.  Rows are then taken in ascending k,
//     kGatherBatch at a time with all their loads in flight, so a sparse row
//     (the dispatch backward: 5 of 8, or 6 of 32 ranks per token) costs only
//     its valid entries;
//   * the sum is the fp32 fused multiply-add chain of combine.cu in the same
//     order (ascending k, from +0), two columns per packed fma.rn.f32x2
//     (bit for bit the scalar chain), rounded to bf16 once;
//   * one item per warp by default, in CTAs of four warps (many short CTAs
//     that the block scheduler balances); num_channels CTAs otherwise, each
//     warp striding over items.
//
// Launch shape (GB300, single launch after an L2 flush; dispatch backward at
// the DeepSeek-V3 / Qwen-like / DeepSeek-16B-like shapes): three rows in
// flight and 128-thread CTAs, 59.1 / 36.6 / 69.4 us.  Four rows: 59.2 /
// 38.7 / 71.4 us; five: 59.9 / 42.8 / 73.5 us; eight rows in 256-thread CTAs
// (118 registers): 71.7 / 59.4 / 83.7 us; 16-byte lanes: slower at every
// shape.  The 16-byte gather of combine.cu took 59.2 / 55.4 / 227 us: it
// walks every slot of the row, so a sparse row keeps few loads in flight.
//
// Slots >= n_rows are flagged (MOE_DEVERR_CAPACITY) and skipped; negative
// slots are skipped.  Every access is in bounds: a lane whose columns lie
// past the row (the last segment of a row whose width is not a multiple of
// 512) loads and stores nothing.
#include <climits>

#include <cuda_bf16.h>

#include "fastdiv.h"
#include "moe_common.cuh"
#include "packed_f32x2.cuh"

namespace moe {

namespace {

constexpr int kGatherThreads = 128;
constexpr int kGatherWarps = kGatherThreads / 32;
constexpr int kGatherBatch = 3;          // rows in flight per warp
constexpr int kGatherSeg = 512;          // columns per item
constexpr int kGatherLaneCols = 16;      // columns per lane (32 bytes)

struct GatherArgs {
    const uint8_t* y;            // bf16 [n_rows, H]
    const int32_t* slot;         // [T, K]: source row of (t, k), -1 = none
    const float* w;              // [T, K], or NULL for unit weights
    uint8_t* out;                // bf16 [T, H]
    int32_t T, K, H, nseg;
    int64_t n_rows, n_items;
    FastDiv seg_div;             // division by nseg
    int32_t items_fit_u32;       // every item index of the launch is below 2^32
    uint32_t* status;
};

// acc (eight column pairs) += w * the 16 bf16 values of v, per pair one
// packed fused multiply-add.
__device__ __forceinline__ void fma16(uint64_t (&acc)[8], uint64_t w2, const uint32_t (&v)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fma_f32x2(w2, bf16x2_to_f32x2(v[j]), acc[j]);
}

__global__ void __launch_bounds__(kGatherThreads)
gather_wide_kernel(GatherArgs a) {
    pdl_wait();
    const uint32_t full = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kGatherWarps;
    bool bad = false;
    for (int64_t item = static_cast<int64_t>(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5); item < a.n_items;
         item += n_warps) {
        int32_t t, seg;
        if (a.items_fit_u32) {
            const uint32_t q = fastdiv(static_cast<uint32_t>(item), a.seg_div);
            t = static_cast<int32_t>(q);
            seg = static_cast<int32_t>(static_cast<uint32_t>(item) - q * static_cast<uint32_t>(a.nseg));
        } else {
            t = static_cast<int32_t>(item / a.nseg);
            seg = static_cast<int32_t>(item - static_cast<int64_t>(t) * a.nseg);
        }
        const int col = seg * kGatherSeg + lane * kGatherLaneCols;
        const bool in = col < a.H;               // H % 16 == 0: all 16 columns or none
        uint64_t acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0ull;        // (+0, +0)
        const int32_t* srow = a.slot + static_cast<int64_t>(t) * a.K;
        const float* wrow = a.w ? a.w + static_cast<int64_t>(t) * a.K : nullptr;
        for (int k0 = 0; k0 < a.K; k0 += 32) {
            const int k = k0 + lane;
            const int32_t s = k < a.K ? __ldg(srow + k) : -1;
            const float wk = (k < a.K && wrow) ? __ldg(wrow + k) : 1.0f;
            bad |= s >= a.n_rows;
            uint32_t valid = __ballot_sync(full, s >= 0 && s < a.n_rows);
            while (valid) {                      // warp-uniform
                // the next (up to) kGatherBatch valid rows, all loads in flight
                uint32_t v[kGatherBatch][8];
                float wb[kGatherBatch];
                int nb = 0;
#pragma unroll
                for (int b = 0; b < kGatherBatch; ++b) {
                    wb[b] = 0.0f;
                    if (valid) {
                        const int src = __ffs(valid) - 1;
                        valid &= valid - 1;
                        const int64_t row = __shfl_sync(full, s, src);
                        wb[b] = __shfl_sync(full, wk, src);
                        if (in) ld_stream_v8(v[b], a.y + (row * a.H + col) * 2);
                        nb = b + 1;
                    }
                }
                // their products, ascending k; nothing is added for an empty batch slot
#pragma unroll
                for (int b = 0; b < kGatherBatch; ++b)
                    if (b < nb && in) fma16(acc, pack_f32x2(wb[b], wb[b]), v[b]);
            }
        }
        if (in) {
            uint32_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float lo, hi;
                unpack_f32x2(acc[j], lo, hi);
                const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
                o[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
            st_stream_v8(a.out + (static_cast<int64_t>(t) * a.H + col) * 2, o);
        }
    }
    pdl_trigger();
    // per warp, no CTA-wide barrier: a warp that is done leaves at once
    if (__any_sync(full, bad) && lane == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

}  // namespace

bool gather_wide_supported(const void* y, const void* out, int32_t hidden) {
    const bool aligned = ((reinterpret_cast<uintptr_t>(y) | reinterpret_cast<uintptr_t>(out)) & 31u) == 0;
    return aligned && hidden % kGatherLaneCols == 0;
}

cudaError_t launch_gather_wide(const uint16_t* y, const int32_t* slot, const float* w, int32_t T, int32_t K,
                               int64_t n_rows, int32_t hidden, uint16_t* out, uint32_t* status,
                               cudaStream_t stream, int32_t num_channels) {
    if (T == 0) return cudaSuccess;
    GatherArgs a;
    a.y = reinterpret_cast<const uint8_t*>(y);
    a.slot = slot;
    a.w = w;
    a.out = reinterpret_cast<uint8_t*>(out);
    a.T = T; a.K = K; a.H = hidden;
    a.nseg = (hidden + kGatherSeg - 1) / kGatherSeg;
    a.n_rows = n_rows;
    a.n_items = static_cast<int64_t>(T) * a.nseg;
    a.status = status;
    a.seg_div = make_fastdiv(static_cast<uint32_t>(a.nseg));
    const int64_t need = (a.n_items + kGatherWarps - 1) / kGatherWarps;     // one item per warp
    int64_t grid = num_channels > 0 ? num_channels : need;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    a.items_fit_u32 = a.n_items + grid * kGatherWarps <= (int64_t{1} << 32) ? 1 : 0;
    // An ordinary launch, like combine.cu's: a gather grid made resident early
    // (programmatic launch) competes with the draining producer of its rows.
    gather_wide_kernel<<<static_cast<unsigned>(grid), kGatherThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
