// api.cu -- the C ABI of libmoe_ep.so (declared in include/moe_ep.h): host
// argument checks, carving of caller memory, kernel launches and status
// read-back.  No allocation, no synchronisation inside the operator calls.
#include <climits>
#include <cstring>

#include "moe_common.cuh"

namespace moe {

int32_t sm_count() {
    static thread_local int cached_dev = -1;
    static thread_local int cached = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev != cached_dev) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached = n;
        cached_dev = dev;
    }
    return cached;
}

}  // namespace moe

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool sizes_ok(int32_t T, int32_t K, int32_t E, int32_t R) {
    return T >= 0 && K >= 1 && E >= 1 && R >= 1 && E % R == 0;
}

bool sizes_supported(int32_t K, int32_t E, int32_t R) {
    return K <= MOE_MAX_TOPK && E <= MOE_MAX_EXPERTS && R <= MOE_MAX_RANKS;
}

int32_t num_tiles_for(int32_t T, int32_t tile_tokens) {
    const int32_t n = (T + tile_tokens - 1) / tile_tokens;
    return n < 1 ? 1 : n;
}

// Arrays carved from the caller's memory, in this order.
struct Carve {
    size_t off = 0;
    char* base;
    explicit Carve(void* p) : base(static_cast<char*>(p)) {}
    template <typename T>
    T* take(size_t count) {
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off = moe::align_up(off + sizeof(T) * count, 256);
        return p;
    }
};

// num_sources == 0: single-source layout (recv_expert_offset [E+1]);
// S >= 1: multi-source layout (recv_source_offset [R, S+1] instead).
size_t carve_layout(moe_layout* L, void* mem, int32_t T, int32_t K, int32_t E, int32_t R, int64_t capacity,
                    int32_t num_tiles, int32_t num_sources) {
    Carve c(mem);
    moe_layout tmp;
    moe_layout* o = L ? L : &tmp;
    o->tokens_per_expert = c.take<int32_t>(E);
    o->expert_offset = c.take<int32_t>(E + 1);
    o->tokens_per_rank = c.take<int32_t>(R);
    o->rank_offset = c.take<int32_t>(R + 1);
    if (num_sources == 0) {
        o->recv_expert_offset = c.take<int32_t>(E + 1);
        o->recv_source_offset = nullptr;
    } else {
        o->recv_expert_offset = nullptr;
        o->recv_source_offset = c.take<int32_t>(static_cast<size_t>(R) * (num_sources + 1));
    }
    o->recv_slot = c.take<int32_t>(static_cast<size_t>(T) * R);
    o->expert_slot = c.take<int32_t>(static_cast<size_t>(T) * K);
    o->recv_src_token = c.take<int32_t>(static_cast<size_t>(capacity));
    o->expert_src_row = c.take<int32_t>(static_cast<size_t>(T) * K);
    o->expert_weight = c.take<float>(static_cast<size_t>(T) * K);
    o->status = c.take<uint32_t>(1);
    const size_t ws_bytes = moe::layout_workspace_bytes(T, K, E, num_tiles);
    o->workspace = c.take<char>(ws_bytes);
    o->workspace_bytes = ws_bytes;
    return c.off;
}

moe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// The fields that tell the two layout kinds apart are consistent.
bool layout_mode_ok(const moe_layout* L) {
    if (L->num_sources == 0) return L->recv_expert_offset != nullptr;
    if (L->num_sources < 0 || L->num_sources > MOE_MAX_SOURCES || L->source_tokens < 0) return false;
    return L->recv_source_offset != nullptr &&
           static_cast<int64_t>(L->num_sources) * L->source_tokens == L->T &&
           L->capacity == static_cast<int64_t>(L->T) * L->R;
}

uint64_t timeout_of(const moe_tuning* t) {
    return (t && t->wait_timeout_ns) ? t->wait_timeout_ns : moe::kDefaultWaitNs;
}

moe_status layout_args_ok(const int32_t* topk_idx, int32_t num_experts, int32_t num_ranks, const moe_layout* L) {
    if (!L || !L->workspace || !L->status) return MOE_ERR_INVALID_ARG;
    if (num_experts != L->E || num_ranks != L->R) return MOE_ERR_INVALID_ARG;
    if (!layout_mode_ok(L)) return MOE_ERR_INVALID_ARG;
    if (L->T > 0 && !topk_idx) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status dispatch_args_ok(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format,
                            const void* recv_x, const void* recv_scales, const moe_tuning* tuning) {
    if (!L || !L->status || hidden <= 0 || hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (format != MOE_FORMAT_BF16 && format != MOE_FORMAT_FP8 && format != MOE_FORMAT_MXFP8) return MOE_ERR_INVALID_ARG;
    if (L->T > 0 && (!x || !recv_x)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv_x)) return MOE_ERR_INVALID_ARG;
    if (format != MOE_FORMAT_BF16) {
        if (hidden % 128 != 0 || (L->T > 0 && !recv_scales) || (reinterpret_cast<uintptr_t>(recv_scales) & 3u) != 0)
            return MOE_ERR_INVALID_ARG;
    } else if (recv_scales) {
        return MOE_ERR_INVALID_ARG;
    }
    if (tuning && (tuning->num_channels < 0 || tuning->stages < 0 || tuning->stages > 8 ||
                   (tuning->stages != 0 && tuning->stages < 2) || tuning->chunk_bytes < 0 ||
                   (tuning->chunk_bytes != 0 && (tuning->chunk_bytes < 256 || tuning->chunk_bytes % 256 != 0)) ||
                   tuning->variant < 0 || tuning->variant > 4))
        return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_layout_bytes(int32_t T, int32_t K, int32_t E, int32_t R, int64_t capacity) {
    if (!sizes_ok(T, K, E, R) || capacity < 0) return 0;
    const int32_t tt = moe::default_tile_tokens(T, K);
    return carve_layout(nullptr, nullptr, T, K, E, R, capacity, num_tiles_for(T, tt), 0);
}

moe_status moe_layout_init(moe_layout* L, int32_t T, int32_t K, int32_t E, int32_t R, int64_t capacity,
                           void* device_mem, size_t bytes) {
    if (!L || !device_mem) return MOE_ERR_INVALID_ARG;
    if (!sizes_ok(T, K, E, R)) return MOE_ERR_INVALID_ARG;
    if (!sizes_supported(K, E, R)) return MOE_ERR_UNSUPPORTED;
    const int64_t worst = static_cast<int64_t>(T) * (K < R ? K : R);
    if (capacity < worst || capacity > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (static_cast<int64_t>(T) * K > INT32_MAX || static_cast<int64_t>(T) * R > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(device_mem) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (bytes < moe_layout_bytes(T, K, E, R, capacity)) return MOE_ERR_INVALID_ARG;
    std::memset(L, 0, sizeof(*L));
    L->T = T; L->K = K; L->E = E; L->R = R;
    L->capacity = capacity;
    L->tile_tokens = moe::default_tile_tokens(T, K);
    L->num_tiles = num_tiles_for(T, L->tile_tokens);
    L->num_sources = 0;
    L->source_tokens = T;
    carve_layout(L, device_mem, T, K, E, R, capacity, L->num_tiles, 0);
    return MOE_OK;
}

size_t moe_layout_sources_bytes(int32_t S, int32_t source_tokens, int32_t K, int32_t E, int32_t R) {
    if (S < 1 || S > MOE_MAX_SOURCES || source_tokens < 0) return 0;
    const int64_t T = static_cast<int64_t>(S) * source_tokens;
    if (T > INT32_MAX || !sizes_ok(static_cast<int32_t>(T), K, E, R)) return 0;
    const int64_t cap = T * R;
    if (cap > INT32_MAX) return 0;
    const int32_t t32 = static_cast<int32_t>(T);
    const int32_t tt = moe::default_tile_tokens(t32, K);
    return carve_layout(nullptr, nullptr, t32, K, E, R, cap, num_tiles_for(t32, tt), S);
}

moe_status moe_layout_init_sources(moe_layout* L, int32_t S, int32_t source_tokens, int32_t K, int32_t E, int32_t R,
                                   void* device_mem, size_t bytes) {
    if (!L || !device_mem || S < 1 || source_tokens < 0) return MOE_ERR_INVALID_ARG;
    if (S > MOE_MAX_SOURCES) return MOE_ERR_UNSUPPORTED;
    const int64_t T = static_cast<int64_t>(S) * source_tokens;
    if (T > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    const int32_t t32 = static_cast<int32_t>(T);
    if (!sizes_ok(t32, K, E, R)) return MOE_ERR_INVALID_ARG;
    if (!sizes_supported(K, E, R)) return MOE_ERR_UNSUPPORTED;
    if (T * R > INT32_MAX || T * K > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(device_mem) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (bytes < moe_layout_sources_bytes(S, source_tokens, K, E, R)) return MOE_ERR_INVALID_ARG;
    std::memset(L, 0, sizeof(*L));
    L->T = t32; L->K = K; L->E = E; L->R = R;
    L->capacity = T * R;
    L->tile_tokens = moe::default_tile_tokens(t32, K);
    L->num_tiles = num_tiles_for(t32, L->tile_tokens);
    L->num_sources = S;
    L->source_tokens = source_tokens;
    carve_layout(L, device_mem, t32, K, E, R, L->capacity, L->num_tiles, S);
    return MOE_OK;
}

moe_status moe_dispatch_layout(const int32_t* topk_idx, const float* topk_w, int32_t num_experts,
                               int32_t num_ranks, moe_layout* L, void* stream, const moe_tuning* tuning) {
    const moe_status st = layout_args_ok(topk_idx, num_experts, num_ranks, L);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_layout(topk_idx, topk_w, L, static_cast<cudaStream_t>(stream), timeout_of(tuning),
                                        tuning ? tuning->debug_flags : 0u));
}

moe_status moe_dispatch(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format, void* recv_x,
                        void* recv_scales, void* stream, const moe_tuning* tuning) {
    const moe_status st = dispatch_args_ok(x, hidden, L, format, recv_x, recv_scales, tuning);
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_dispatch(x, hidden, L, format, recv_x, recv_scales,
                                          static_cast<cudaStream_t>(stream), tuning ? tuning->num_channels : 0,
                                          tuning ? tuning->stages : 0, tuning ? tuning->chunk_bytes : 0,
                                          tuning ? tuning->variant : 0, timeout_of(tuning)));
}

moe_status moe_dispatch_with_layout(const int32_t* topk_idx, const float* topk_w, int32_t num_experts,
                                    int32_t num_ranks, moe_layout* L, const uint16_t* x, int32_t hidden,
                                    int32_t format, void* recv_x, void* recv_scales, void* stream,
                                    const moe_tuning* tuning) {
    moe_status st = layout_args_ok(topk_idx, num_experts, num_ranks, L);
    if (st != MOE_OK) return st;
    st = dispatch_args_ok(x, hidden, L, format, recv_x, recv_scales, tuning);
    if (st != MOE_OK) return st;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    // bf16 and MXFP8: the finalize lets the dispatch grid become resident
    // while the scan runs (single-source layout: the dispatch comes right
    // after it), and the dispatch loads and quantises its rows before its
    // dependency wait.  On GB300 that shortened the layout + dispatch +
    // combine step by 1.1-1.9 us (bf16) and 0.4-1.6 us (MXFP8) at three
    // shapes.  FP8 gained nothing from the early loads and lost 0.3-0.8 us
    // with its grid (four CTAs of 63 registers per SM) resident early, so it
    // runs exactly as the two separate calls do.
    const bool early = format != MOE_FORMAT_FP8;
    st = from_cuda(moe::launch_layout(topk_idx, topk_w, L, s, timeout_of(tuning), tuning ? tuning->debug_flags : 0u,
                                      early && L->num_sources == 0));
    if (st != MOE_OK) return st;
    return from_cuda(moe::launch_dispatch(x, hidden, L, format, recv_x, recv_scales, s,
                                          tuning ? tuning->num_channels : 0, tuning ? tuning->stages : 0,
                                          tuning ? tuning->chunk_bytes : 0, tuning ? tuning->variant : 0,
                                          timeout_of(tuning), early));
}

moe_status moe_combine(const uint16_t* y, int32_t hidden, const moe_layout* L, const float* topk_w, uint16_t* out,
                       void* stream, const moe_tuning* tuning) {
    if (!L || !L->status || hidden <= 0 || hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (L->T > 0 && (!y || !topk_w || !out)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out) || (reinterpret_cast<uintptr_t>(topk_w) & 3u) != 0) return MOE_ERR_INVALID_ARG;
    if (tuning && (tuning->num_channels < 0 || tuning->variant < 0 || tuning->variant > 4)) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine(y, hidden, L, topk_w, out, static_cast<cudaStream_t>(stream),
                                         tuning ? tuning->num_channels : 0, tuning ? tuning->variant : 0,
                                         timeout_of(tuning)));
}

moe_status moe_dispatch_backward(const uint16_t* grad_recv, int32_t hidden, const moe_layout* L, uint16_t* grad_x,
                                 void* stream, const moe_tuning* tuning) {
    if (!L || !L->status || hidden <= 0 || hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (L->T > 0 && (!grad_recv || !grad_x)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(grad_recv) || !aligned16(grad_x)) return MOE_ERR_INVALID_ARG;
    if (tuning && tuning->num_channels < 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_dispatch_backward(grad_recv, hidden, L, grad_x, static_cast<cudaStream_t>(stream),
                                                   tuning ? tuning->num_channels : 0));
}

moe_status moe_combine_backward(const uint16_t* grad_out, const uint16_t* y, int32_t hidden, const moe_layout* L,
                                const float* topk_w, uint16_t* grad_y, float* grad_w, void* stream,
                                const moe_tuning* tuning) {
    if (!L || !L->status || hidden <= 0 || hidden % 8 != 0) return MOE_ERR_INVALID_ARG;
    if (L->T > 0 && (!grad_out || !y || !topk_w || !grad_y || !grad_w)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(grad_out) || !aligned16(y) || !aligned16(grad_y) ||
        (reinterpret_cast<uintptr_t>(topk_w) & 3u) != 0 || (reinterpret_cast<uintptr_t>(grad_w) & 3u) != 0)
        return MOE_ERR_INVALID_ARG;
    if (tuning && tuning->num_channels < 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_combine_backward(grad_out, y, hidden, L, topk_w, grad_y, grad_w,
                                                  static_cast<cudaStream_t>(stream), tuning ? tuning->num_channels : 0));
}

moe_status moe_ll_dispatch(const uint16_t* x, const int32_t* topk_idx, int32_t T, int32_t K, int32_t E, int32_t hidden,
                           int32_t cap_per_expert, uint16_t* recv, int32_t* tokens_per_expert, int32_t* ll_slot,
                           uint32_t* status, void* stream, const moe_tuning* tuning) {
    if (T < 0 || K < 1 || E < 1 || hidden <= 0 || hidden % 8 != 0 || cap_per_expert < 0) return MOE_ERR_INVALID_ARG;
    if (K > MOE_MAX_TOPK || E > MOE_MAX_EXPERTS) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(T) * K > moe::ll_max_entries()) return MOE_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(E) * cap_per_expert > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    if (!tokens_per_expert || !status) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !topk_idx || !ll_slot || (cap_per_expert > 0 && !recv))) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(recv)) return MOE_ERR_INVALID_ARG;
    if (tuning && tuning->num_channels < 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_ll_dispatch(x, topk_idx, T, K, E, hidden, cap_per_expert, recv, tokens_per_expert,
                                             ll_slot, status, static_cast<cudaStream_t>(stream),
                                             tuning ? tuning->num_channels : 0));
}

moe_status moe_ll_combine(const uint16_t* y, const int32_t* ll_slot, const float* topk_w, int32_t T, int32_t K,
                          int32_t E, int32_t hidden, int32_t cap_per_expert, uint16_t* out, uint32_t* status,
                          void* stream, const moe_tuning* tuning) {
    if (T < 0 || K < 1 || E < 1 || hidden <= 0 || hidden % 8 != 0 || cap_per_expert < 0) return MOE_ERR_INVALID_ARG;
    if (!status) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!y || !ll_slot || !topk_w || !out)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(out) || (reinterpret_cast<uintptr_t>(topk_w) & 3u) != 0) return MOE_ERR_INVALID_ARG;
    if (tuning && tuning->num_channels < 0) return MOE_ERR_INVALID_ARG;
    return from_cuda(moe::launch_ll_combine(y, ll_slot, topk_w, T, K, static_cast<int64_t>(E) * cap_per_expert, hidden,
                                            out, status, static_cast<cudaStream_t>(stream),
                                            tuning ? tuning->num_channels : 0));
}

moe_status moe_layout_read_status(const moe_layout* L, void* stream, uint32_t* flags_out) {
    if (!L || !L->status) return MOE_ERR_INVALID_ARG;
    uint32_t flags = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&flags, L->status, sizeof(flags), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    if (flags_out) *flags_out = flags;
    // a timed-out scan leaves stale ranks behind, which the later kernels
    // then flag as capacity errors: report the root cause first
    if (flags & MOE_DEVERR_TIMEOUT) return MOE_ERR_TIMEOUT;
    if (flags & MOE_DEVERR_EXPERT_ID) return MOE_ERR_EXPERT_ID;
    if (flags & MOE_DEVERR_CAPACITY) return MOE_ERR_CAPACITY;
    return MOE_OK;
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_CAPACITY: return "slot outside the receive / expert buffers";
        case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_UNSUPPORTED: return "sizes beyond the supported limits";
        case MOE_ERR_EXPERT_ID: return "expert id outside [-1, E)";
    }
    return "unknown status";
}

int32_t moe_device_sm_count(void) { return moe::sm_count(); }

}  // extern "C"
