// ll.cu -- low-latency (decode) dispatch into a fixed per-expert buffer.
//
// DeepEP ships low-latency kernels for decode next to its high-throughput
// ones ("Inside the Nebius + PyTorch DeepSeek V3 recipe", section "DeepEP").
// Their point is a static receive shape: every valid entry (t,k) of expert e
// lands at row e * cap + j of recv [E, cap, H], j = the entry's position among
// e's entries in (t,k) order, so the experts can run on fixed-size inputs.
//
// One launch, no workspace: decode batches are small (T * K <= 4096 entries
// here), so every CTA loads the whole routing into shared memory and computes
// all the positions itself (warp-aggregated ranks with per-warp histograms, as
// in the layout scan, then a scan across warps); then it copies its share of
// the token rows with 16-byte vector loads and stores.  CTA 0 also writes the
// slot map and the per-expert counts.  The combine for this layout is the
// regular weighted gather over the slot map (combine.cu).
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kLLThreads = 256;
constexpr int kLLWarps = kLLThreads / 32;

struct LLArgs {
    const uint4* x;              // [T, H/8]
    const int32_t* topk_idx;     // [T, K]
    int32_t T, K, E, H8, cap;
    uint4* recv;                 // [E * cap, H/8]
    int32_t* tokens_per_expert;  // [E]
    int32_t* ll_slot;            // [T, K]
    uint32_t* status;
};

__global__ void __launch_bounds__(kLLThreads)
ll_dispatch_kernel(LLArgs a) {
    extern __shared__ int32_t sm[];
    const int n = a.T * a.K;
    int32_t* s_e = sm;                          // [n]: expert of entry i, or -1
    int32_t* s_pos = s_e + n;                   // [n]: position within the warp's segment, then row
    int32_t* s_hist = s_pos + n;                // [warps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();

    bool bad_id = false;
    for (int i = tid; i < n; i += kLLThreads) {
        int e = a.topk_idx[i];
        if (e < -1 || e >= a.E) { bad_id = true; e = -1; }
        s_e[i] = e;
    }
    for (int i = tid; i < kLLWarps * a.E; i += kLLThreads) s_hist[i] = 0;
    __syncthreads();

    // positions inside each warp's contiguous segment (ballot per id bit)
    const int seg = ((n + kLLWarps - 1) / kLLWarps + 31) / 32 * 32;
    const int nbits = 32 - __clz(max(a.E - 1, 1));
    int32_t* my_hist = s_hist + warp * a.E;
    const uint32_t lt = lanemask_lt();
    for (int c = 0; c * 32 < seg; ++c) {
        const int i = warp * seg + c * 32 + lane;
        const int e = i < n ? s_e[i] : -1;
        uint32_t peers = __ballot_sync(0xffffffffu, e >= 0);
        if (e < 0) peers = ~peers;
        for (int b = 0; b < nbits; ++b) {
            const bool bit = (e >> b) & 1;
            const uint32_t bb = __ballot_sync(0xffffffffu, bit);
            peers &= bit ? bb : ~bb;
        }
        const int base = e >= 0 ? my_hist[e] : 0;
        __syncwarp();
        if (e >= 0 && (peers & lt) == 0) my_hist[e] = base + __popc(peers);
        __syncwarp();
        if (i < n) s_pos[i] = base + __popc(peers & lt);
    }
    __syncthreads();
    // exclusive scan across the warps; totals per expert
    for (int e = tid; e < a.E; e += kLLThreads) {
        int run = 0;
        for (int w = 0; w < kLLWarps; ++w) {
            const int v = s_hist[w * a.E + e];
            s_hist[w * a.E + e] = run;
            run += v;
        }
        if (blockIdx.x == 0) a.tokens_per_expert[e] = min(run, a.cap);
    }
    __syncthreads();
    bool overflow = false;
    for (int i = tid; i < n; i += kLLThreads) {
        const int e = s_e[i];
        int32_t row = -1;
        if (e >= 0) {
            const int j = s_hist[(i / seg) * a.E + e] + s_pos[i];
            if (j < a.cap) row = e * a.cap + j; else overflow = true;
        }
        s_pos[i] = row;
        if (blockIdx.x == 0) a.ll_slot[i] = row;
    }
    const int flags = __syncthreads_or(bad_id) ? MOE_DEVERR_EXPERT_ID : 0;
    const int flags2 = __syncthreads_or(overflow) ? MOE_DEVERR_CAPACITY : 0;
    if (blockIdx.x == 0 && tid == 0) *a.status = static_cast<uint32_t>(flags | flags2);
    pdl_trigger();

    // copy this CTA's entries: flat (entry, 16-byte group) loop, four in flight
    const int64_t i0 = static_cast<int64_t>(n) * blockIdx.x / gridDim.x;
    const int64_t i1 = static_cast<int64_t>(n) * (blockIdx.x + 1) / gridDim.x;
    const int64_t total = (i1 - i0) * a.H8;
    for (int64_t f = tid; f < total; f += 4 * kLLThreads) {
        uint4 v[4];
        int64_t dst[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int64_t g = f + u * kLLThreads;
            dst[u] = -1;
            if (g < total) {
                const int64_t i = i0 + g / a.H8;
                const int64_t c = g - (g / a.H8) * a.H8;
                const int32_t row = s_pos[i];
                if (row >= 0) {
                    v[u] = ld_stream_v4(a.x + (i / a.K) * a.H8 + c);
                    dst[u] = static_cast<int64_t>(row) * a.H8 + c;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (dst[u] >= 0) a.recv[dst[u]] = v[u];
    }
}

}  // namespace

int32_t ll_max_entries() { return 4096; }

cudaError_t launch_ll_dispatch(const uint16_t* x, const int32_t* topk_idx, int32_t T, int32_t K, int32_t E,
                               int32_t hidden, int32_t cap, uint16_t* recv, int32_t* tokens_per_expert,
                               int32_t* ll_slot, uint32_t* status, cudaStream_t stream, int32_t num_channels) {
    LLArgs a;
    a.x = reinterpret_cast<const uint4*>(x);
    a.topk_idx = topk_idx;
    a.T = T; a.K = K; a.E = E; a.H8 = hidden / 8; a.cap = cap;
    a.recv = reinterpret_cast<uint4*>(recv);
    a.tokens_per_expert = tokens_per_expert;
    a.ll_slot = ll_slot;
    a.status = status;
    const int n = T * K;
    const size_t smem = sizeof(int32_t) * (2 * static_cast<size_t>(n) + static_cast<size_t>(kLLWarps) * E);
    cudaError_t err = cudaFuncSetAttribute(ll_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    // about four entries per CTA, at most two CTAs per SM
    int64_t grid = num_channels > 0 ? num_channels : (n + 3) / 4;
    const int64_t max_grid = static_cast<int64_t>(sm_count()) * 2;
    if (num_channels <= 0 && grid > max_grid) grid = max_grid;
    if (grid < 1) grid = 1;
    return launch_pdl(ll_dispatch_kernel, dim3(static_cast<unsigned>(grid)), dim3(kLLThreads), smem, stream, a);
}

}  // namespace moe
