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
// in the layout scan, then a scan across warps).  A CTA owns a range of
// tokens: it reads each token row once (16-byte vectors in registers; the
// first row's loads are issued before the ranking, so their latency hides
// behind it) and writes it to every destination row of the token.  CTA 0 also
// writes the slot map and the per-expert counts.  The combine for this layout
// is the regular weighted gather over the slot map (combine.cu).
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kLLThreads = 256;
constexpr int kLLWarps = kLLThreads / 32;
constexpr int kLLVecs = 4;                    // 16-byte vectors per thread per column group (8192 columns)

struct LLArgs {
    const uint4* x;              // [T, H/8]
    const int32_t* topk_idx;     // [T, K]
    int32_t T, K, E, H8, cap;
    uint4* recv;                 // [E * cap, H/8]
    int32_t* tokens_per_expert;  // [E]
    int32_t* ll_slot;            // [T, K]
    uint32_t* status;
};

// Column group [c0, c0 + kLLVecs * kLLThreads) of token t's row (16-byte
// vectors; t < 0 or columns past the row give zeros).
__device__ __forceinline__ void load_group(const LLArgs& a, int t, int c0, int tid, uint4 (&v)[kLLVecs]) {
#pragma unroll
    for (int j = 0; j < kLLVecs; ++j) {
        const int c = c0 + j * kLLThreads + tid;
        v[j] = (t >= 0 && c < a.H8) ? ld_stream_v4(a.x + static_cast<int64_t>(t) * a.H8 + c) : make_uint4(0u, 0u, 0u, 0u);
    }
}

__global__ void __launch_bounds__(kLLThreads)
ll_dispatch_kernel(LLArgs a) {
    extern __shared__ int32_t sm[];
    const int n = a.T * a.K;
    int32_t* s_e = sm;                          // [n]: expert of entry i, or -1
    int32_t* s_pos = s_e + n;                   // [n]: position within the warp's segment, then row
    int32_t* s_hist = s_pos + n;                // [warps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    // this CTA's tokens; the first row's first column group is loaded now
    const int t_begin = static_cast<int>(static_cast<int64_t>(a.T) * blockIdx.x / gridDim.x);
    const int t_end = static_cast<int>(static_cast<int64_t>(a.T) * (blockIdx.x + 1) / gridDim.x);
    uint4 v[kLLVecs];
    load_group(a, t_begin < t_end ? t_begin : -1, 0, tid, v);

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

    // each token row once into registers, then out to the token's destination rows
    const int group = kLLVecs * kLLThreads;                   // 16-byte vectors per column group
    for (int t = t_begin; t < t_end; ++t) {
        for (int c0 = 0; c0 < a.H8; c0 += group) {
            if (t != t_begin || c0 != 0) load_group(a, t, c0, tid, v);
            for (int k = 0; k < a.K; ++k) {
                const int32_t row = s_pos[t * a.K + k];          // the same for every thread
                if (row < 0) continue;
                uint4* dst = a.recv + static_cast<int64_t>(row) * a.H8;
#pragma unroll
                for (int j = 0; j < kLLVecs; ++j) {
                    const int c = c0 + j * kLLThreads + tid;
                    if (c < a.H8) dst[c] = v[j];
                }
            }
        }
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
    // one token per CTA, at most two CTAs per SM (then several tokens per CTA)
    int64_t grid = num_channels > 0 ? num_channels : T;
    const int64_t max_grid = static_cast<int64_t>(sm_count()) * 2;
    if (num_channels <= 0 && grid > max_grid) grid = max_grid;
    if (grid > T) grid = T;
    if (grid < 1) grid = 1;
    return launch_pdl(ll_dispatch_kernel, dim3(static_cast<unsigned>(grid)), dim3(kLLThreads), smem, stream, a);
}

}  // namespace moe
