// noalloc.cu -- moe_dispatch_layout_noalloc: the dispatch layout with its scan
// workspace in a fixed device array compiled into this library, for callers
// that cannot allocate device memory themselves (see moe_ep.h).
//
// The array lives at file scope; host code never uses its name as an address
// (in host code that name is only a stand-in), it asks the runtime for the
// device address once per device and passes that to the same two layout
// kernels that moe_dispatch_layout launches.
#include <mutex>

#include "moe_common.cuh"

namespace {

static_assert(MOE_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size is a whole number of 256-byte lines");

// Zero at module load, like the caller memory moe_layout_init expects.
static __device__ __align__(256) unsigned char g_layout_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;

// The array's device address belongs to the context the library's module was
// loaded into.  A cudaDeviceReset (or any teardown of the primary context)
// and the context the runtime creates afterwards load the module again, at an
// address that may differ, so each cached address is keyed by the identity of
// the context it was looked up in.
struct ScratchEntry {
    unsigned long long ctx_id;
    void* addr;
};
ScratchEntry g_scratch[kMaxDevices] = {};

// Driver calls reached through the runtime (no link against libcuda).
using CtxGetCurrentFn = int (*)(void**);
using CtxGetIdFn = int (*)(void*, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

cudaError_t driver_entry_points() {
    if (g_ctx_get_current && g_ctx_get_id) return cudaSuccess;
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    cudaError_t err = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa);
    if (err != cudaSuccess || qa != cudaDriverEntryPointSuccess || !a) return cudaErrorSymbolNotFound;
    err = cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb);
    if (err != cudaSuccess || qb != cudaDriverEntryPointSuccess || !b) return cudaErrorSymbolNotFound;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
    return cudaSuccess;
}

// Identity of the current context (0 if none is current yet).
cudaError_t current_ctx_id(unsigned long long* id) {
    void* ctx = nullptr;
    *id = 0;
    if (g_ctx_get_current(&ctx) != 0) return cudaErrorDeviceUninitialized;
    if (ctx == nullptr) return cudaSuccess;
    return g_ctx_get_id(ctx, id) == 0 ? cudaSuccess : cudaErrorDeviceUninitialized;
}

// Device address of g_layout_scratch in the current device's context: looked
// up with cudaGetSymbolAddress once per device (with that device current),
// and again whenever the context has been replaced since.
cudaError_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    err = driver_entry_points();
    if (err != cudaSuccess) return err;
    unsigned long long id = 0;
    err = current_ctx_id(&id);
    if (err != cudaSuccess) return err;
    ScratchEntry& e = g_scratch[dev];
    if (id == 0 || e.addr == nullptr || e.ctx_id != id) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_layout_scratch);   // makes the device's context current if needed
        if (err != cudaSuccess) return err;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        err = current_ctx_id(&id);
        if (err != cudaSuccess) return err;
        if (id == 0) return cudaErrorDeviceUninitialized;
        e.ctx_id = id;
        e.addr = p;
    }
    *out = e.addr;
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_dispatch_layout_noalloc(const int32_t* topk_idx, const float* topk_w, int32_t num_experts,
                                                  int32_t num_ranks, moe_layout* L, void* stream,
                                                  const moe_tuning* tuning) {
    if (!L) return MOE_ERR_INVALID_ARG;
    const int32_t T = L->T, K = L->K, E = L->E, R = L->R;
    if (T < 0 || K < 1 || E < 1 || R < 1 || E % R != 0) return MOE_ERR_INVALID_ARG;
    if (num_experts != E || num_ranks != R) return MOE_ERR_INVALID_ARG;
    if (K > MOE_MAX_TOPK || E > MOE_MAX_EXPERTS || R > MOE_MAX_RANKS) return MOE_ERR_UNSUPPORTED;
    const int64_t worst = static_cast<int64_t>(T) * (K < R ? K : R);
    if (L->capacity < worst || L->capacity > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * K > INT32_MAX || static_cast<int64_t>(T) * R > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (T > 0 && !topk_idx) return MOE_ERR_INVALID_ARG;
    if (!L->tokens_per_expert || !L->expert_offset || !L->tokens_per_rank || !L->rank_offset ||
        !L->recv_slot || !L->expert_slot || !L->recv_src_token || !L->expert_src_row ||
        !L->expert_weight || !L->status)
        return MOE_ERR_INVALID_ARG;
    if (L->num_sources == 0) {
        if (!L->recv_expert_offset) return MOE_ERR_INVALID_ARG;
    } else if (L->num_sources < 0 || L->num_sources > MOE_MAX_SOURCES || L->source_tokens < 0 ||
               static_cast<int64_t>(L->num_sources) * L->source_tokens != T ||
               L->capacity != static_cast<int64_t>(T) * R || !L->recv_source_offset) {
        return MOE_ERR_INVALID_ARG;
    }

    moe_layout tmp = *L;
    tmp.tile_tokens = moe::default_tile_tokens(T, K);
    tmp.num_tiles = (T + tmp.tile_tokens - 1) / tmp.tile_tokens;
    if (tmp.num_tiles < 1) tmp.num_tiles = 1;
    const size_t need = moe::layout_workspace_bytes(T, K, E, tmp.num_tiles);
    if (need > MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;

    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    tmp.workspace = scratch;
    tmp.workspace_bytes = need;

    // The array keeps the previous call's contents.  The scan's progress
    // flags carry a generation number and never look current to a later
    // call, but the tile ticket and the gathered error bits must start at
    // zero: clear them (a call interrupted between its two kernels would
    // otherwise leave them set).  No allocation is involved.
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* hdr = static_cast<char*>(scratch);
    if (cudaMemsetAsync(hdr + offsetof(moe::WsHeader, ticket), 0, sizeof(uint32_t), s) != cudaSuccess ||
        cudaMemsetAsync(hdr + offsetof(moe::WsHeader, k1_err), 0, sizeof(uint32_t), s) != cudaSuccess)
        return MOE_ERR_CUDA;

    const uint64_t timeout = (tuning && tuning->wait_timeout_ns) ? tuning->wait_timeout_ns : moe::kDefaultWaitNs;
    const cudaError_t err =
        moe::launch_layout(topk_idx, topk_w, &tmp, s, timeout, tuning ? tuning->debug_flags : 0u);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
