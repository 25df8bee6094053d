// ll.cu -- low-latency (decode) dispatch into a fixed per-expert buffer.
//
// DeepEP ships low-latency kernels for decode next to its high-throughput
// ones ("Inside the Nebius + PyTorch DeepSeek V3 recipe", section "DeepEP").
// Their point is a static receive shape: every valid entry (t,k) of expert e
// lands at row e * cap + j of recv [E, cap, H], j = the entry's position among
// e's entries in (t,k) order, so the experts can run on fixed-size inputs.
//
// One launch, no workspace.  A CTA owns a range of tokens and needs only the
// rows of its own entries: row(t,k) = e * cap + j with j = #{earlier entries
// of expert e}.  It counts the entries before its first token per expert
// (shared-memory atomics over a histogram; T * K <= 4096 entries, all of a
// thread's id loads in flight at once), then one warp walks its own entries
// in order, 32 at a time: lanes with the same expert find each other with
// one match instruction, take base + their rank among them, and the group's
// lowest lane advances the count.  No CTA ranks the whole batch.  CTA 0 also
// counts every entry for tokens_per_expert and the status word.  Each token
// row is read once (16-byte vectors in registers; the first row's loads are
// issued before the counting, so their latency hides behind it) and written
// to every destination row of the token.  The combine for this layout is the
// regular weighted gather over the slot map (combine.cu).
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kLLThreads = 256;
constexpr int kLLVecs = 4;                    // 16-byte vectors per thread per column group (8192 columns)
constexpr int kLLMaxEntries = 4096;           // T * K
constexpr int kLLIdsPerThread = kLLMaxEntries / kLLThreads;

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
// vectors; t < 0 or columns past the row give zeros).  32-byte vectors
// measured no faster here: a CTA's writes are bound by its SM's store path to
// L2 (about 112 KB per token at 62 GB/s per SM), not by store instructions.
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
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // this CTA's tokens and entries [i_begin, i_end)
    const int t_begin = static_cast<int>(static_cast<int64_t>(a.T) * blockIdx.x / gridDim.x);
    const int t_end = static_cast<int>(static_cast<int64_t>(a.T) * (blockIdx.x + 1) / gridDim.x);
    const int i_begin = t_begin * a.K, i_end = t_end * a.K, m = i_end - i_begin;
    const bool first = blockIdx.x == 0;        // also counts every entry: tokens_per_expert, status
    int32_t* s_count = sm;                      // [E]: entries of e before the current one
    int32_t* s_total = s_count + a.E;           // [E] (CTA 0): all entries of e
    int32_t* s_own = s_total + a.E;             // [m]: expert of each own entry (-1: masked or bad), then its row
    __shared__ uint32_t s_flags;
    pdl_wait();
    uint4 v[kLLVecs];
    load_group(a, t_begin < t_end ? t_begin : -1, 0, tid, v);

    // the ids this CTA needs (those before its last token; CTA 0: all of them)
    const int limit = first ? n : i_end;
    int32_t e_in[kLLIdsPerThread];
#pragma unroll
    for (int u = 0; u < kLLIdsPerThread; ++u) {
        const int i = tid + u * kLLThreads;
        e_in[u] = i < limit ? __ldg(a.topk_idx + i) : -1;
    }
    for (int e = tid; e < 2 * a.E; e += kLLThreads) s_count[e] = 0;
    if (tid == 0) s_flags = 0u;
    __syncthreads();
    bool bad_id = false;
#pragma unroll
    for (int u = 0; u < kLLIdsPerThread; ++u) {
        const int i = tid + u * kLLThreads;
        if (i >= limit) break;
        int e = e_in[u];
        if (e < -1 || e >= a.E) { bad_id = true; e = -1; }     // counted as masked
        if (e >= 0 && i < i_begin) atomicAdd(&s_count[e], 1);
        if (e >= 0 && first) atomicAdd(&s_total[e], 1);
        if (i >= i_begin && i < i_end) s_own[i - i_begin] = e;
    }
    if (bad_id) atomicOr(&s_flags, MOE_DEVERR_EXPERT_ID);
    __syncthreads();

    // own entries in (t,k) order, 32 at a time: base count + rank among equal experts
    if (warp == 0) {
        const uint32_t lt = lanemask_lt();
        bool overflow = false;
        for (int q0 = 0; q0 < m; q0 += 32) {
            const int q = q0 + lane;
            const int e = q < m ? s_own[q] : -1;
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            const int base = e >= 0 ? s_count[e] : 0;
            __syncwarp();
            int32_t row = -1;
            if (e >= 0) {
                const int j = base + __popc(peers & lt);
                if (j < a.cap) row = e * a.cap + j; else overflow = true;
                if ((peers & lt) == 0) s_count[e] = base + __popc(peers);
            }
            if (q < m) {
                s_own[q] = row;
                a.ll_slot[i_begin + q] = row;
            }
            __syncwarp();
        }
        if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicOr(&s_flags, MOE_DEVERR_CAPACITY);
    } else if (first) {
        // CTA 0: the counts; any expert over capacity overflowed somewhere
        bool over = false;
        for (int e = tid - 32; e < a.E; e += kLLThreads - 32) {
            a.tokens_per_expert[e] = min(s_total[e], a.cap);
            over |= s_total[e] > a.cap;
        }
        if (over) atomicOr(&s_flags, MOE_DEVERR_CAPACITY);
    }
    __syncthreads();
    if (first && tid == 0) *a.status = s_flags;
    pdl_trigger();

    // each token row once into registers, then out to the token's destination rows
    const int group = kLLVecs * kLLThreads;                   // 16-byte vectors per column group
    for (int t = t_begin; t < t_end; ++t) {
        for (int c0 = 0; c0 < a.H8; c0 += group) {
            if (t != t_begin || c0 != 0) load_group(a, t, c0, tid, v);
            for (int k = 0; k < a.K; ++k) {
                const int32_t row = s_own[(t - t_begin) * a.K + k];   // the same for every thread
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

int32_t ll_max_entries() { return kLLMaxEntries; }

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
    if (n > kLLMaxEntries) return cudaErrorInvalidValue;     // the host checks ll_max_entries() first
    // one token per CTA, at most two CTAs per SM (then several tokens per CTA)
    int64_t grid = num_channels > 0 ? num_channels : T;
    const int64_t max_grid = static_cast<int64_t>(sm_count()) * 2;
    if (num_channels <= 0 && grid > max_grid) grid = max_grid;
    if (grid > T) grid = T;
    if (grid < 1) grid = 1;
    // two expert counters per expert and one word per entry of the largest token range
    const int64_t max_tokens = (static_cast<int64_t>(T) + grid - 1) / grid;
    const size_t smem = sizeof(int32_t) * (2 * static_cast<size_t>(E) + static_cast<size_t>(max_tokens) * K);
    cudaError_t err = cudaFuncSetAttribute(ll_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_pdl(ll_dispatch_kernel, dim3(static_cast<unsigned>(grid)), dim3(kLLThreads), smem, stream, a);
}

}  // namespace moe
