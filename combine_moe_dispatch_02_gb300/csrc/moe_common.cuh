// moe_common.cuh -- device helpers shared by the dispatch-layout, dispatch and
// combine kernels: inline PTX for mbarriers, TMA bulk copies and memory
// ordering, bounded waits, and the layout workspace description.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

#include "moe_ep.h"

namespace moe {

constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s bound on any device wait

// ----------------------------------------------------------------- workspace

// Header at the start of the layout workspace.  `ticket` hands out scan-tile
// ids in CTA start order; `epoch` numbers layout calls so that progress flags
// of an earlier call never look current; `k1_err` gathers the scan kernel's
// error bits until the finalize kernel moves them into the status word;
// `abort` is set to the current generation once any wait gave up.
struct WsHeader {
    uint32_t ticket;
    uint32_t epoch;
    uint32_t k1_err;
    uint32_t abort;
    uint32_t pad[60];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte line");

struct LayoutWs {
    WsHeader* hdr;
    uint32_t* tile_flag;   // [num_tiles]: (generation << 2) | state
    int32_t*  tile_agg;    // [num_tiles][2E]: this tile's counts (expert, primary)
    int32_t*  tile_incl;   // [num_tiles][2E]: counts of tiles 0..i inclusive
    uint64_t* tile_tagged; // [min(num_tiles, tagged limit)][2E]: (generation << 32) | count, the
                           // aggregates of the look-back without flags (up to 33 tiles, or 16
                           // per thread sharing a column: 65 for E <= 64, 129 for E <= 32)
    int32_t*  erank;       // [T*K]: rank of entry among entries of its expert
    int32_t*  prank;       // [T*K]: rank of a primary entry among its expert's primaries
};

enum : uint32_t { kFlagAgg = 1u, kFlagPrefix = 2u, kFlagError = 3u };
constexpr uint32_t kGenMask = (1u << 30) - 1u;   // generations live in [1, 2^30)

constexpr int kLayoutThreads = 512;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kMaxTileEntries = 2048;                                   // T_tile * K
constexpr int kMaxChunksPerWarp = kMaxTileEntries / (kLayoutWarps * 32);  // 4
constexpr int kFinalizeThreads = 256;
constexpr int kFinalizeTokens = 32;                                     // tokens per finalize block

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}

// 64-bit accesses are single-copy atomic: a reader sees either the old or the
// new word, never a mix, so a generation tag in the upper half validates the
// count in the lower half.
__device__ __forceinline__ uint64_t ld_relaxed_gpu_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// mbarrier (CTA scope) ---------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Plain arrive (count 1) with release semantics at CTA scope.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most `timeout_ns`.
// Returns false if the bound ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// After a timed-out wait: wait (bounded) for the last TMA load issued into
// each stage of a ring whose loads k = 0 .. issued-1 went to stage k % S and
// complete phase k / S of that stage's mbarrier, so that no load lands in
// shared memory after the CTA has exited.  False if one is still outstanding.
__device__ __forceinline__ bool drain_ring_loads(uint64_t* bars, int S, int issued, uint64_t timeout_ns) {
    bool all = true;
    for (int s = 0; s < S && s < issued; ++s) {
        const int j = s + (issued - 1 - s) / S * S;     // the last load issued into stage s
        all &= mbar_wait_bounded(&bars[s], static_cast<uint32_t>(j / S) & 1u, timeout_ns);
    }
    return all;
}

// TMA bulk copies (non-tensor) -------------------------------------------

// global -> shared, completion signalled as transaction bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_addr(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

// shared -> global, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_s2g(void* gdst, const void* smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(smem_addr(smem_src)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" :: "n"(N) : "memory");
}

// Runtime-count form of bulk_wait_read (the PTX operand is an immediate).
__device__ __forceinline__ void bulk_wait_read_n(int n) {
    switch (n) {
        case 0: bulk_wait_read<0>(); break;
        case 1: bulk_wait_read<1>(); break;
        case 2: bulk_wait_read<2>(); break;
        case 3: bulk_wait_read<3>(); break;
        case 4: bulk_wait_read<4>(); break;
        case 5: bulk_wait_read<5>(); break;
        case 6: bulk_wait_read<6>(); break;
        default: bulk_wait_read<7>(); break;
    }
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Streaming 16-byte global accesses --------------------------------------

__device__ __forceinline__ uint4 ld_stream_v4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream_v4(uint4* p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// 32-byte forms (sm_100+; the address must be 32-byte aligned).
__device__ __forceinline__ void ld_stream_v8(uint32_t (&r)[8], const void* p) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_stream_v8(void* p, const uint32_t (&r)[8]) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                    "r"(r[7])
                 : "memory");
}

// Programmatic dependent launch ---------------------------------------------
//
// The layout and dispatch kernels are launched with programmatic stream
// serialization (launch_pdl below), so their CTAs may be scheduled while the
// previous kernel in the stream is still finishing.  Every kernel of the path
// calls pdl_wait() before its first global memory access: it returns once the
// previous grid has completed and its writes are visible (at once when the
// kernel was launched normally or nothing precedes it).
// pdl_trigger() lets the next kernel's launch begin early; it never affects
// correctness, only when the dependent CTAs become resident.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe

// Launch helpers implemented in the per-operator translation units.
namespace moe {
// early_trigger: the kernel after the layout may become resident while the
// scan runs (moe_dispatch_with_layout); x_ready: x was complete before the
// layout's first kernel, so the dispatch may read it before its dependency
// wait (moe_dispatch_with_layout only).
cudaError_t launch_layout(const int32_t* topk_idx, const float* topk_w, const moe_layout* L,
                          cudaStream_t stream, uint64_t timeout_ns, uint32_t debug_flags,
                          bool early_trigger = false);
cudaError_t launch_dispatch(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format,
                            void* recv_x, void* recv_scales, cudaStream_t stream,
                            int32_t num_channels, int32_t stages, int32_t chunk_bytes, int32_t variant,
                            uint64_t timeout_ns, bool x_ready = false);
bool dispatch_wide_supported(const void* x, int32_t hidden, int32_t format, const void* recv_x);
cudaError_t launch_dispatch_wide(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format, void* recv_x,
                                 void* recv_scales, cudaStream_t stream, int32_t num_channels, bool x_ready);
cudaError_t launch_combine(const uint16_t* y, int32_t hidden, const moe_layout* L, const float* topk_w,
                           uint16_t* out, cudaStream_t stream, int32_t num_channels, int32_t variant,
                           uint64_t timeout_ns);
// 32-byte gather (gather_wide.cu): out[t] = bf16(fma chain over the valid
// slots of row t, ascending k, weights w or 1).  Needs y and out 32-byte
// aligned and hidden % 16 == 0 (gather_wide_supported).
bool gather_wide_supported(const void* y, const void* out, int32_t hidden);
cudaError_t launch_gather_wide(const uint16_t* y, const int32_t* slot, const float* w, int32_t T, int32_t K,
                               int64_t n_rows, int32_t hidden, uint16_t* out, uint32_t* status,
                               cudaStream_t stream, int32_t num_channels);
cudaError_t launch_dispatch_backward(const uint16_t* grad_recv, int32_t hidden, const moe_layout* L,
                                     uint16_t* grad_x, cudaStream_t stream, int32_t num_channels);
cudaError_t launch_combine_backward(const uint16_t* grad_out, const uint16_t* y, int32_t hidden, const moe_layout* L,
                                    const float* topk_w, uint16_t* grad_y, float* grad_w, cudaStream_t stream,
                                    int32_t num_channels);
int32_t ll_max_entries();
cudaError_t launch_ll_dispatch(const uint16_t* x, const int32_t* topk_idx, int32_t T, int32_t K, int32_t E,
                               int32_t hidden, int32_t cap, uint16_t* recv, int32_t* tokens_per_expert,
                               int32_t* ll_slot, uint32_t* status, cudaStream_t stream, int32_t num_channels);
cudaError_t launch_ll_combine(const uint16_t* y, const int32_t* ll_slot, const float* topk_w, int32_t T, int32_t K,
                              int64_t n_rows, int32_t hidden, uint16_t* out, uint32_t* status, cudaStream_t stream,
                              int32_t num_channels);
LayoutWs layout_workspace(const moe_layout* L);
size_t layout_workspace_bytes(int32_t T, int32_t K, int32_t E, int32_t num_tiles);
int32_t default_tile_tokens(int32_t T, int32_t K);
int32_t sm_count();
}  // namespace moe
