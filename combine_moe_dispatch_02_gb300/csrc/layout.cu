// layout.cu -- dispatch layout: per-expert / per-rank counts, prefix offsets
// and token <-> slot maps for MoE dispatch and combine.
//
// What is computed follows the problem statement of expert-parallel MoE
// ("Inside the Nebius + PyTorch DeepSeek V3 recipe", section "Mixture-of-
// experts and wide expert parallelism": experts partitioned across ranks,
// tokens dispatched to their top-K experts; Hybrid-EP news article,
// "Availability and Integration": worst-case preallocated receive buffers).
// The definitions (orderings, primary expert) are documented in moe_ep.h.
//
// Two kernels:
//  1. layout_scan_kernel: one CTA per tile of about 2048 (t,k) entries.  When
//     every tile fits on the GPU at once (no more tiles than SMs; a scan CTA
//     needs at most one SM), the tile is the block index and its routing ids
//     are loaded at entry; otherwise tile ids come from an atomic ticket, so a
//     CTA only ever waits on tiles that running CTAs have claimed.  Per tile:
//     warp-aggregated, order-preserving
//     ranks of every entry among the entries of its expert (peer masks from
//     one ballot per id bit + popc inside a warp, per-warp histograms in
//     shared memory, an exclusive scan
//     across warps) and, in the same pass, among the "primary" entries; then
//     a decoupled look-back over the 2E-wide count vectors of earlier tiles
//     (one warp inspects 32 predecessors at a time; the vectors are summed
//     with many loads in flight per thread) gives the tile's prefix.  Every
//     wait is bounded.
//  2. layout_finalize_kernel: one block per 32 tokens derives the expert
//     offsets from the last tile's totals (a block-wide scan), stages the
//     tokens' entries and ranks in shared memory, adds the offsets and writes
//     recv_slot, expert_slot, recv_src_token, expert_src_row and
//     expert_weight with coalesced row writes, plus the tails past the last
//     used row.
// The multi-source layout (S source ranks, one worst-case region per
// destination, rows in (source, token) order) uses the same two kernels with
// the primary pairs counted per destination rank instead of per primary
// expert, and a third, layout_source_offsets_kernel, that reads each source's
// first row per region off the sorted regions by a warp-wide 32-way search.
#include <algorithm>
#include <climits>

#include "moe_common.cuh"

namespace moe {

namespace {

// Tiles whose (token, rank) table fits in this many ints find their primary
// entries with one shared-memory atomicMin per entry; larger ones (many ranks)
// compare every entry with the token's other entries.
constexpr int kMaxPrimSlots = 16384;
// Experts up to this count find equal ids in a warp with a shared-memory
// table of lane masks (one atomicOr per lane); more experts take one ballot
// per bit of the id.
constexpr int kMaxPeerE = 256;
constexpr int kFinalizePerThread = kFinalizeTokens * MOE_MAX_TOPK / kFinalizeThreads;   // entries per thread (4)
static_assert(kFinalizePerThread * kFinalizeThreads == kFinalizeTokens * MOE_MAX_TOPK,
              "a finalize block's threads cover its 32 tokens' entries for every K <= MOE_MAX_TOPK");
constexpr size_t kMaxSmemPerBlock = 227 * 1024;     // opt-in dynamic shared memory per block on sm_100+

struct ScanArgs {
    const int32_t* topk_idx;
    int32_t T, K, E, m, R;
    int32_t tile_tokens, num_tiles;
    int32_t prim_table;          // tile_tokens * R <= kMaxPrimSlots
    LayoutWs ws;
    uint32_t* status;
    uint64_t timeout_ns;
    uint32_t debug_flags;
    int32_t by_block;            // tile = block index (every tile resident at once), else the ticket
};

// Width of a tile's count vector: E expert counts, E primary counts, padded to
// a multiple of 4 so that the look-back can move it in 16-byte pieces.
__host__ __device__ __forceinline__ int vec_width(int E) { return (2 * E + 3) / 4 * 4; }

__host__ __device__ __forceinline__ int round_up4(int n) { return (n + 3) / 4 * 4; }

// Key of a valid entry: (rank << 16) | expert (experts < 2^16); -1 if masked.
// Two keys share a rank iff their upper halves are equal, and then compare like
// their expert ids.
//
// Entry k of a token is primary if no other valid entry of the token on the
// same rank has a smaller id and no earlier entry has the same id.
// The token's keys are read eight at a time (independent loads in flight)
// and compared without early exits.
__device__ __forceinline__ bool is_primary_key(const int32_t* row_keys, int K, int k, int32_t key) {
    bool prim = true;
    for (int k0 = 0; k0 < K; k0 += 8) {
        int32_t kk[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) kk[u] = (k0 + u < K) ? row_keys[k0 + u] : -1;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int k2 = k0 + u;
            const int32_t key2 = kk[u];
            prim &= !(k2 != k && key2 >= 0 && (key2 >> 16) == (key >> 16) && (key2 < key || (key2 == key && k2 < k)));
        }
    }
    return prim;
}

// i / K for i < 2^11 and K <= 32 without an integer division: (i + 0.5) / K is
// at least 1/(2K) >= 2^-6 away from an integer, and the fp32 product's error is
// below 2^11 * 2^-23 = 2^-12, so truncation gives the exact quotient.
__device__ __forceinline__ int div_small(int i, float inv_k) {
    return __float2int_rz((static_cast<float>(i) + 0.5f) * inv_k);
}

constexpr uint32_t kWaitTimedOut = 4u;
constexpr int kLookbackWindow = 32;      // predecessors one look-back step inspects (warp 0's lanes)
constexpr int kTaggedBatch = 16;         // tagged words a thread loads at once (one round for <= 16 predecessors)

// Threads that share a column of the tagged look-back: the largest power of
// two g <= 32 with g * W <= kLayoutThreads (1 where W > kLayoutThreads / 2).
// The g threads of a column are adjacent lanes of one warp.
__host__ __device__ __forceinline__ int lookback_group(int W) {
    int g = 1;
    while (g < 32 && 2 * g * W <= kLayoutThreads) g *= 2;
    return g;
}

// Tiles up to which the look-back uses generation-tagged aggregates: every
// look-back then sums all its predecessors, in at most two rounds of loads
// per thread (one round once kTaggedBatch * g covers them).
__host__ __device__ __forceinline__ int tagged_tile_limit(int E) {
    const int g = lookback_group(vec_width(E));
    return kTaggedBatch * g + 1 > kLookbackWindow + 1 ? kTaggedBatch * g + 1 : kLookbackWindow + 1;
}

// Wait (bounded) until a tile flag carries generation `gen`; return its state,
// kFlagError if another CTA aborted the scan, or kWaitTimedOut.
__device__ uint32_t wait_tile_flag(const uint32_t* flag, uint32_t gen, const uint32_t* abort_word,
                                   uint64_t timeout_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
        const uint32_t v = ld_acquire_gpu(flag);
        if ((v >> 2) == gen && (v & 3u) != 0) return v & 3u;
        if (ld_relaxed_gpu(abort_word) == gen) return kFlagError;
        if (it == 0) {
            t0 = globaltimer_ns();
        } else if (globaltimer_ns() - t0 > timeout_ns) {
            return kWaitTimedOut;
        }
        __nanosleep(it < 32 ? 32 : 256);
    }
}

// SRC = false: primary pairs are counted per primary expert (the single-source
// layout, rows grouped by expert inside each rank).  SRC = true: they are
// counted per destination rank in the column of the rank's first expert (the
// multi-source layout, rows in token order inside each rank's region).
template <bool SRC>
__global__ void __launch_bounds__(kLayoutThreads, 1)
layout_scan_kernel(ScanArgs a) {
    extern __shared__ __align__(16) int32_t smem[];
    const int W = vec_width(a.E);
    const int nvec = W / 4;
    int32_t* s_key = smem;                                            // [kMaxTileEntries]
    int32_t* s_hist = s_key + kMaxTileEntries;                        // [warps][W]
    int32_t* s_prefix = s_hist + kLayoutWarps * W;                    // [W]
    int32_t* s_agg = s_prefix + W;                                    // [W]
    int4* s_part = reinterpret_cast<int4*>(s_agg + W);                // [kLayoutThreads]
    int32_t* s_rank = reinterpret_cast<int32_t*>(s_part + kLayoutThreads);   // [E]
    // [tile_tokens][R] if prim_table: min of (e << 5 | k) per (token, rank)
    int32_t* s_min = s_rank + round_up4(a.E);
    const bool peer_table = a.E <= kMaxPeerE;
    uint32_t* s_peer = reinterpret_cast<uint32_t*>(s_min + (a.prim_table ? round_up4(a.tile_tokens * a.R) : 0));   // [warps][kMaxPeerE]
    __shared__ int s_tile;
    __shared__ uint32_t s_gen;
    __shared__ int s_lb_count, s_lb_final;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();
    pdl_trigger();          // one wave of CTAs: the finalize grid may become resident now
    // Tile = block index: its routing ids are loaded now, all of a thread's
    // loads in flight at once, before the shared-memory setup and without the
    // ticket's round trip (each tile a look-back waits on is sure to get an SM,
    // as they all fit at once).  Otherwise the tile comes from the ticket.
    constexpr int kIdsPerThread = kMaxTileEntries / kLayoutThreads;
    int32_t e_in[kIdsPerThread];
    // by_block: the call counter, needed at the publish.  Every thread loads
    // it, unconditionally: loaded by thread 0 inside a branch of its own, it
    // held that thread for a memory round trip right there (0.6 us measured
    // on GB300), and the whole CTA behind it at the next barrier.  The
    // previous call's finalize wrote it and has completed (the dependency
    // wait above).
    const uint32_t epoch0 = __ldcg(&a.ws.hdr->epoch);
    if (a.by_block) {
        const int64_t base = static_cast<int64_t>(blockIdx.x) * a.tile_tokens * a.K;
        const int nn = min(a.tile_tokens, a.T - static_cast<int>(blockIdx.x) * a.tile_tokens) * a.K;
#pragma unroll
        for (int u = 0; u < kIdsPerThread; ++u) {
            const int i = tid + u * kLayoutThreads;
            e_in[u] = i < nn ? __ldg(a.topk_idx + base + i) : -1;
        }
    } else if (tid == 0) {
        s_tile = static_cast<int>(atomicAdd(&a.ws.hdr->ticket, 1u));
        s_gen = (ld_relaxed_gpu(&a.ws.hdr->epoch) & kGenMask) + 1u;
    }
    // shared-memory set-up in 16-byte stores (every table starts on a 16-byte
    // boundary; W is a multiple of 4)
    for (int i = tid; i < kLayoutWarps * W / 4; i += kLayoutThreads)
        reinterpret_cast<int4*>(s_hist)[i] = make_int4(0, 0, 0, 0);
    for (int i = tid; i < W / 4; i += kLayoutThreads) reinterpret_cast<int4*>(s_agg)[i] = make_int4(0, 0, 0, 0);
    for (int e = tid; e < a.E; e += kLayoutThreads) s_rank[e] = e / a.m;
    if (a.prim_table)
        for (int i = tid; i < round_up4(a.tile_tokens * a.R) / 4; i += kLayoutThreads)
            reinterpret_cast<int4*>(s_min)[i] = make_int4(INT_MAX, INT_MAX, INT_MAX, INT_MAX);
    if (peer_table)
        for (int i = tid; i < kLayoutWarps * kMaxPeerE / 4; i += kLayoutThreads)
            reinterpret_cast<uint4*>(s_peer)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const int tile = a.by_block ? static_cast<int>(blockIdx.x) : s_tile;
    if (tile >= a.num_tiles) return;   // cannot happen: one CTA per tile
    if (tile == 0 && tid == 0) *a.status = 0u;   // the status word covers this call onwards

    const int t0 = tile * a.tile_tokens;
    const int nt = min(a.tile_tokens, a.T - t0);
    const int n = nt * a.K;

    // 1. the tile's entries as keys; ids outside [-1, E) are flagged and masked.
    //    Every valid entry counts itself in the tile aggregate, and, with the
    //    table, bids (e << 5 | k) for the smallest id of its token on its rank
    //    (ties: the first k).
    bool bad = false;
    const float inv_k = 1.0f / static_cast<float>(a.K);
    auto count_entry = [&](int i, int e) {
        int32_t key = -1;
        if (e >= 0 && e < a.E) {
            const int r = s_rank[e];
            key = (r << 16) | e;
            atomicAdd(&s_agg[e], 1);
            if (a.prim_table) {
                const int tl = div_small(i, inv_k);
                atomicMin(&s_min[tl * a.R + r], (e << 5) | (i - tl * a.K));
            }
        } else if (e != -1) {
            bad = true;
        }
        s_key[i] = key;
    };
    if (a.by_block) {
#pragma unroll
        for (int u = 0; u < kIdsPerThread; ++u) {
            const int i = tid + u * kLayoutThreads;
            if (i >= n) break;
            count_entry(i, e_in[u]);
        }
    } else {
        for (int i = tid; i < n; i += kLayoutThreads) count_entry(i, a.topk_idx[static_cast<int64_t>(t0) * a.K + i]);
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(&a.ws.hdr->k1_err, MOE_DEVERR_EXPERT_ID);

    // 1b. primary flags of the entries this lane ranks below (warp w owns a
    //     contiguous segment of 32-entry chunks); primaries complete the tile
    //     aggregate in their column: the primary expert's own or (SRC) the
    //     first expert of the rank
    const int seg = ((n + kLayoutWarps - 1) / kLayoutWarps + 31) / 32 * 32;
    int32_t key[kMaxChunksPerWarp];
    bool prim[kMaxChunksPerWarp];
#pragma unroll
    for (int c = 0; c < kMaxChunksPerWarp; ++c) {
        const int i = warp * seg + c * 32 + lane;
        key[c] = (c * 32 < seg && i < n) ? s_key[i] : -1;
        prim[c] = false;
        if (key[c] >= 0) {
            const int tl = div_small(i, inv_k);
            const int k = i - tl * a.K;
            prim[c] = a.prim_table ? s_min[tl * a.R + (key[c] >> 16)] == (((key[c] & 0xffff) << 5) | k)
                                   : is_primary_key(s_key + tl * a.K, a.K, k, key[c]);
            if (prim[c]) atomicAdd(&s_agg[a.E + (SRC ? (key[c] >> 16) * a.m : (key[c] & 0xffff))], 1);
        }
    }
    if (a.by_block && tid == 0) s_gen = (epoch0 & kGenMask) + 1u;
    __syncthreads();
    const uint32_t gen = s_gen;

    // 1c. publish the tile aggregate now, so that successors find it on their
    //     first look-back poll; tile 0's aggregate is its inclusive prefix
    const bool stall = (a.debug_flags & MOE_DEBUG_STALL_FIRST_TILE) && tile == 0;
    // Up to tagged_tile_limit(E) tiles (33; 65 for E <= 64) every look-back
    // sums all its predecessors' aggregates, published as generation-tagged
    // 64-bit words: no fence, no flag, and a reader validates each word it
    // loads.  More tiles: vectors plus a progress flag (the barrier orders
    // every thread's stores before thread 0's fence and release store, which
    // publish them at GPU scope).
    const bool tagged = a.num_tiles <= tagged_tile_limit(a.E);
    if (tagged) {
        uint64_t* my_words = a.ws.tile_tagged + static_cast<int64_t>(tile) * W;
        if (!stall)
            for (int col = tid; col < W; col += kLayoutThreads)
                st_relaxed_gpu_u64(my_words + col, (static_cast<uint64_t>(gen) << 32) | static_cast<uint32_t>(s_agg[col]));
    } else {
        int32_t* my_vec = (tile == 0 ? a.ws.tile_incl : a.ws.tile_agg) + static_cast<int64_t>(tile) * W;
        for (int col = tid; col < W; col += kLayoutThreads) my_vec[col] = s_agg[col];
        __syncthreads();
        if (tid == 0 && !stall) {
            __threadfence();
            st_release_gpu(&a.ws.tile_flag[tile], (gen << 2) | (tile == 0 ? kFlagPrefix : kFlagAgg));
        }
    }

    // 2. order-preserving ranks inside the tile: each warp keeps its own
    //    histogram.  Lanes with the same expert (peers) come from a table of
    //    lane masks (each lane ORs its bit into its expert's word, reads the
    //    word back, clears it), or, for many experts, from one ballot per bit
    //    of the expert id.  Masked lanes count as peers of each other.
    int lr_e[kMaxChunksPerWarp], lr_p[kMaxChunksPerWarp], ent_e[kMaxChunksPerWarp];
    int32_t* my_hist = s_hist + warp * W;
    uint32_t peers[kMaxChunksPerWarp];
    uint32_t rpeers[kMaxChunksPerWarp];     // SRC: lanes with the same rank
#pragma unroll
    for (int c = 0; c < kMaxChunksPerWarp; ++c) {
        peers[c] = __ballot_sync(0xffffffffu, key[c] >= 0);
        if (key[c] < 0) peers[c] = ~peers[c];
        rpeers[c] = peers[c];
    }
    if (peer_table) {
        uint32_t* tbl = s_peer + warp * kMaxPeerE;
#pragma unroll
        for (int c = 0; c < kMaxChunksPerWarp; ++c) {
            const bool valid = key[c] >= 0;
            const int e = key[c] & 0xffff;
            if (valid) atomicOr(&tbl[e], 1u << lane);
            __syncwarp();
            if (valid) peers[c] = tbl[e];
            __syncwarp();
            if (valid) tbl[e] = 0u;
            __syncwarp();
        }
    } else {
        const int nbits = 32 - __clz(max(a.E - 1, 1));
        for (int b = 0; b < nbits; ++b) {
#pragma unroll
            for (int c = 0; c < kMaxChunksPerWarp; ++c) {
                const bool bit = (key[c] >> b) & 1;
                const uint32_t bb = __ballot_sync(0xffffffffu, bit);
                peers[c] &= bit ? bb : ~bb;
            }
        }
    }
    if constexpr (SRC) {
        const int rbits = 32 - __clz(max(a.R - 1, 1));
        for (int b = 16; b < 16 + rbits; ++b) {
#pragma unroll
            for (int c = 0; c < kMaxChunksPerWarp; ++c) {
                const bool bit = (key[c] >> b) & 1;
                const uint32_t bb = __ballot_sync(0xffffffffu, bit);
                rpeers[c] &= bit ? bb : ~bb;
            }
        }
    }
    // 2b. per-warp histogram updates, chunk by chunk
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int c = 0; c < kMaxChunksPerWarp; ++c) {
        lr_e[c] = -1; lr_p[c] = -1; ent_e[c] = -1;
        if (c * 32 >= seg) continue;            // warp-uniform
        const int e = key[c] >= 0 ? (key[c] & 0xffff) : -1;
        // primary counter column: the expert's own, or (SRC) its rank's first expert's
        const int pcol = a.E + (SRC ? (key[c] >> 16) * a.m : e);
        const uint32_t pmask = __ballot_sync(0xffffffffu, prim[c]) & (SRC ? rpeers[c] : peers[c]);
        int base_e = 0, base_p = 0;
        if (e >= 0) { base_e = my_hist[e]; base_p = my_hist[pcol]; }
        __syncwarp();
        if (e >= 0 && (peers[c] & lt) == 0) {    // lowest lane of its group updates
            my_hist[e] = base_e + __popc(peers[c]);
            if constexpr (!SRC) my_hist[pcol] = base_p + __popc(pmask);
        }
        if constexpr (SRC) {
            if (prim[c] && (pmask & lt) == 0) my_hist[pcol] = base_p + __popc(pmask);
        }
        __syncwarp();
        if (e >= 0) {
            ent_e[c] = e;
            lr_e[c] = base_e + __popc(peers[c] & lt);
            if (prim[c]) lr_p[c] = base_p + __popc(pmask & lt);
        }
    }
    __syncthreads();

    // 3. exclusive scan of the per-warp histograms (each warp's base)
    for (int col = tid; col < W; col += kLayoutThreads) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int v = s_hist[w * W + col];
            s_hist[w * W + col] = run;
            run += v;
        }
        s_prefix[col] = 0;
    }
    __syncthreads();

    // 4. decoupled look-back over the predecessors' aggregates and inclusive
    //    prefixes
    bool failed = false;
    if (tile > 0 && tagged) {
        // g threads share a column, each summing every g-th predecessor: one
        // round of loads for up to kTaggedBatch * g predecessors, a bounded
        // re-load of any word whose tag is not yet current; the g partial
        // sums meet by shuffles (every thread of a column reaches them, also
        // after a timeout, which discards the sums)
        const int g = lookback_group(W);
        const int sub = tid & (g - 1);
        const uint32_t gmask = g == 32 ? 0xffffffffu : ((1u << g) - 1u) << (lane & ~(g - 1));
        bool tmo = false, aborted = false;
        for (int col = tid / g; col < W && !tmo && !aborted; col += kLayoutThreads / g) {
            int32_t sum = 0;
            for (int q0 = sub; q0 < tile && !tmo && !aborted; q0 += kTaggedBatch * g) {
                uint64_t v[kTaggedBatch];
                // every load unconditional (index clamped, the extra words
                // ignored below): a load under a condition made the thread
                // wait for it before issuing the next one
#pragma unroll
                for (int u = 0; u < kTaggedBatch; ++u)
                    v[u] = ld_relaxed_gpu_u64(a.ws.tile_tagged + static_cast<int64_t>(min(q0 + u * g, tile - 1)) * W + col);
#pragma unroll
                for (int u = 0; u < kTaggedBatch; ++u) {
                    const int q = q0 + u * g;
                    if (q >= tile) break;
                    uint64_t t0 = 0;
                    for (uint32_t it = 0; static_cast<uint32_t>(v[u] >> 32) != gen; ++it) {
                        if (ld_relaxed_gpu(&a.ws.hdr->abort) == gen) { aborted = true; break; }
                        if (it == 0) {
                            t0 = globaltimer_ns();
                        } else if (globaltimer_ns() - t0 > a.timeout_ns) {
                            tmo = true;
                            break;
                        }
                        __nanosleep(it < 32 ? 32 : 256);
                        v[u] = ld_relaxed_gpu_u64(a.ws.tile_tagged + static_cast<int64_t>(q) * W + col);
                    }
                    if (tmo || aborted) break;
                    sum += static_cast<int32_t>(static_cast<uint32_t>(v[u]));
                }
            }
            for (int d = 1; d < g; d <<= 1) sum += __shfl_xor_sync(gmask, sum, d);
            if (sub == 0) s_prefix[col] = sum;
        }
        if (tmo) {
            atomicOr(&a.ws.hdr->k1_err, MOE_DEVERR_TIMEOUT);
            atomicExch(&a.ws.hdr->abort, gen);
        }
        if (__syncthreads_or(tmo || aborted)) return;
    } else if (tile > 0) {
        // the window's vectors are summed by `groups` thread groups, each taking
        // every groups-th predecessor, with 16-byte loads: one round of loads
        const int groups = max(1, min(8, kLayoutThreads / nvec));
        const int g = tid / nvec, v = tid - (tid / nvec) * nvec;
        int hi = tile - 1;                      // nearest tile not yet summed
        while (true) {
            if (warp == 0) {
                const int j = hi - lane;
                uint32_t st = kFlagPrefix;     // lanes past tile 0 never matter
                if (j >= 0) st = wait_tile_flag(&a.ws.tile_flag[j], gen, &a.ws.hdr->abort, a.timeout_ns);
                const uint32_t err = __ballot_sync(0xffffffffu, j >= 0 && (st == kFlagError || st == kWaitTimedOut));
                const uint32_t pre = __ballot_sync(0xffffffffu, j >= 0 && st == kFlagPrefix);
                const uint32_t tmo = __ballot_sync(0xffffffffu, st == kWaitTimedOut);
                if (lane == 0) {
                    if (err) {
                        s_lb_count = -1;
                        if (tmo) {
                            atomicOr(&a.ws.hdr->k1_err, MOE_DEVERR_TIMEOUT);
                            atomicExch(&a.ws.hdr->abort, gen);
                        }
                    } else if (pre) {
                        s_lb_count = __ffs(pre);    // lanes 0..nearest prefix tile
                        s_lb_final = 1;
                    } else {
                        s_lb_count = min(kLookbackWindow, hi + 1);
                        s_lb_final = 0;
                    }
                }
            }
            __syncthreads();
            const int cnt = s_lb_count, fin = s_lb_final;
            if (cnt < 0) { failed = true; break; }
            if (g < groups) {
                int4 acc = make_int4(0, 0, 0, 0);
#pragma unroll 8
                for (int q = g; q < cnt; q += groups) {
                    const int64_t j = hi - q;
                    const int32_t* src = (fin && q == cnt - 1) ? a.ws.tile_incl : a.ws.tile_agg;
                    const int4 x = __ldcg(reinterpret_cast<const int4*>(src + j * W) + v);
                    acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
                }
                s_part[g * nvec + v] = acc;
            }
            __syncthreads();
            for (int c4 = tid; c4 < nvec; c4 += kLayoutThreads) {
                int4 sum = s_part[c4];
                for (int gg = 1; gg < groups; ++gg) {
                    const int4 x = s_part[gg * nvec + c4];
                    sum.x += x.x; sum.y += x.y; sum.z += x.z; sum.w += x.w;
                }
                int4* p = reinterpret_cast<int4*>(s_prefix) + c4;
                int4 cur = *p;
                cur.x += sum.x; cur.y += sum.y; cur.z += sum.z; cur.w += sum.w;
                *p = cur;
            }
            hi -= cnt;
            __syncthreads();
            if (fin) break;
            if (hi < 0) { failed = true; break; }   // no prefix found: cannot happen
        }
        if (failed) {
            if (tid == 0) st_release_gpu(&a.ws.tile_flag[tile], (gen << 2) | kFlagError);
            return;
        }
    }

    // 5. per-entry ranks including the tile prefix (prank = -1: not primary)
#pragma unroll
    for (int c = 0; c < kMaxChunksPerWarp; ++c) {
        if (ent_e[c] < 0) continue;
        const int e = ent_e[c];
        const int64_t gi = static_cast<int64_t>(t0) * a.K + warp * seg + c * 32 + lane;
        const int pcol = a.E + (SRC ? s_rank[e] * a.m : e);
        a.ws.erank[gi] = s_prefix[e] + my_hist[e] + lr_e[c];
        a.ws.prank[gi] = lr_p[c] >= 0 ? s_prefix[pcol] + my_hist[pcol] + lr_p[c] : -1;
    }

    // 6. the inclusive prefix.  The last tile's is the totals vector the
    //    finalize pass reads (kernel completion publishes it).  Other tiles
    //    publish theirs, with a flag, only when look-backs use flags (more
    //    tiles than tagged_tile_limit(E)).
    const bool flagged = !tagged && tile > 0;     // (with flags, tile 0 published its prefix above)
    if (flagged || tile == a.num_tiles - 1) {
        int32_t* my_incl = a.ws.tile_incl + static_cast<int64_t>(tile) * W;
        for (int col = tid; col < W; col += kLayoutThreads) my_incl[col] = s_prefix[col] + s_agg[col];
        if (flagged) {
            __syncthreads();
            if (tid == 0) {
                __threadfence();
                st_release_gpu(&a.ws.tile_flag[tile], (gen << 2) | kFlagPrefix);
            }
        }
    }
}

// Block-wide exclusive prefixes of the expert totals (the last tile's
// inclusive count vector, E expert counts then E primary counts): every
// finalize block computes them for itself, s_eoff[0..E] and s_poff[0..E].
__device__ void expert_offsets(const int32_t* totals, int E, int32_t* s_eoff, int32_t* s_poff, int32_t* s_warp) {
    constexpr int kWarps = kFinalizeThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (E + kFinalizeThreads - 1) / kFinalizeThreads;     // <= 4 (E <= 1024)
    const int b = tid * per;
    int ve[4], vp[4];
    int se = 0, sp = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = b + u;
        const bool in = u < per && e < E;
        ve[u] = in ? __ldcg(totals + e) : 0;
        vp[u] = in ? __ldcg(totals + E + e) : 0;
        se += ve[u];
        sp += vp[u];
    }
    int ie = se, ip = sp;                 // inclusive scans across the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int ue = __shfl_up_sync(0xffffffffu, ie, d);
        const int up = __shfl_up_sync(0xffffffffu, ip, d);
        if (lane >= d) { ie += ue; ip += up; }
    }
    if (lane == 31) { s_warp[warp] = ie; s_warp[kWarps + warp] = ip; }
    __syncthreads();
    int be = ie - se, bp = ip - sp;       // exclusive within the warp
    for (int w = 0; w < warp; ++w) { be += s_warp[w]; bp += s_warp[kWarps + w]; }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int e = b + u;
        if (u < per && e < E) { s_eoff[e] = be; s_poff[e] = bp; }
        be += ve[u];
        bp += vp[u];
    }
    if (tid == kFinalizeThreads - 1) { s_eoff[E] = be; s_poff[E] = bp; }
    __syncthreads();
}

// The last scan tile's inclusive counts are read back here (stream order, or
// the programmatic-launch wait, makes them visible).
struct FinalArgs {
    const int32_t* topk_idx;
    const float* topk_w;
    int32_t T, K, E, R, m;
    int32_t src_order;          // multi-source layout: region r*T per destination
    int64_t capacity;
    int32_t num_tiles;
    LayoutWs ws;
    uint32_t* status;
    int32_t *tokens_per_expert, *expert_offset, *recv_expert_offset;
    int32_t *tokens_per_rank, *rank_offset;
    int32_t *recv_slot, *expert_slot, *recv_src_token, *expert_src_row;
    float* expert_weight;
    int32_t early_trigger;      // let the next kernel become resident at once (see below)
};

__global__ void __launch_bounds__(kFinalizeThreads)
layout_finalize_kernel(FinalArgs a) {
    // With early_trigger the next kernel's CTAs may become resident while the
    // scan still runs; they wait for this grid before using its outputs, so
    // this only matters for work they can do without them (the dispatch of
    // moe_dispatch_with_layout loads and quantises its rows meanwhile).
    if (a.early_trigger) pdl_trigger();
    extern __shared__ int32_t sm[];
    const int E1 = a.E + 1;
    int32_t* s_eoff = sm;                                    // [E+1]
    int32_t* s_poff = s_eoff + E1;                           // [E+1]
    int32_t* s_idx = s_poff + E1;                            // [TB*K]
    int32_t* s_er = s_idx + kFinalizeTokens * a.K;           // [TB*K] expert rank -> expert row
    int32_t* s_pr = s_er + kFinalizeTokens * a.K;            // [TB*K] primary rank
    int32_t* s_rs = s_pr + kFinalizeTokens * a.K;            // [TB*R] receive row per (token, rank)
    int32_t* s_rank = s_rs + kFinalizeTokens * a.R;          // [E] rank of expert e
    const int tid = threadIdx.x;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * kFinalizeTokens;
    const int nt = static_cast<int>(max(min(static_cast<int64_t>(kFinalizeTokens), a.T - t0), int64_t{0}));
    const int n = nt * a.K;
    const int64_t e0 = t0 * a.K;

    // The routing and the weights are inputs of the layout call: they were
    // complete before the scan kernel passed its own dependency wait, so they
    // can be fetched before this kernel's wait (which covers the scan's outputs).
    __shared__ int32_t s_warp[2 * (kFinalizeThreads / 32)];
    int32_t e_r[kFinalizePerThread];
    float w_r[kFinalizePerThread];
#pragma unroll
    for (int u = 0; u < kFinalizePerThread; ++u) {
        const int i = tid + u * kFinalizeThreads;
        e_r[u] = i < n ? a.topk_idx[e0 + i] : -1;
        w_r[u] = (i < n && a.topk_w) ? a.topk_w[e0 + i] : 0.0f;
    }
    for (int i = tid; i < a.E; i += kFinalizeThreads) s_rank[i] = i / a.m;
    for (int i = tid; i < nt * a.R; i += kFinalizeThreads) s_rs[i] = -1;
    // the call counter only changes in this kernel (block 0, below); the
    // header words are loaded by every thread, unconditionally, so that no
    // thread waits for them before it uses them
    const bool header = blockIdx.x == 0 && tid == 0;
    const uint32_t epoch = __ldcg(&a.ws.hdr->epoch);

    pdl_wait();
    if (!a.early_trigger) pdl_trigger();    // one wave of CTAs: the dispatch grid may become resident now
    // the scan's per-entry ranks (loaded for every entry, so that they do not
    // wait for the ids) and, inside expert_offsets, its totals
    int32_t er_r[kFinalizePerThread], pr_r[kFinalizePerThread];
#pragma unroll
    for (int u = 0; u < kFinalizePerThread; ++u) {
        const int i = tid + u * kFinalizeThreads;
        er_r[u] = i < n ? __ldcg(a.ws.erank + e0 + i) : 0;
        pr_r[u] = i < n ? __ldcg(a.ws.prank + e0 + i) : 0;
    }
    const uint32_t k1 = __ldcg(&a.ws.hdr->k1_err);   // the scan's error bits (used by the header thread)
    const int32_t* totals = a.ws.tile_incl + static_cast<int64_t>(a.num_tiles - 1) * vec_width(a.E);
    expert_offsets(totals, a.E, s_eoff, s_poff, s_warp);
#pragma unroll
    for (int u = 0; u < kFinalizePerThread; ++u) {
        const int i = tid + u * kFinalizeThreads;
        if (i < n) {
            const int e = (e_r[u] < 0 || e_r[u] >= a.E) ? -1 : e_r[u];
            s_idx[i] = e;
            s_er[i] = e >= 0 ? er_r[u] : 0;
            s_pr[i] = e >= 0 ? pr_r[u] : 0;
        }
    }
    __syncthreads();

    // block 0: the counts and offsets, the status word and the workspace
    // reset, first, so that they overlap the other blocks' scatter writes
    if (blockIdx.x == 0) {
        for (int e = tid; e <= a.E; e += kFinalizeThreads) {
            a.expert_offset[e] = s_eoff[e];
            if (!a.src_order) a.recv_expert_offset[e] = s_poff[e];
            if (e < a.E) a.tokens_per_expert[e] = s_eoff[e + 1] - s_eoff[e];
        }
        for (int r = tid; r <= a.R; r += kFinalizeThreads) {
            a.rank_offset[r] = a.src_order ? r * a.T : s_poff[r * a.m];
            if (r < a.R) a.tokens_per_rank[r] = s_poff[(r + 1) * a.m] - s_poff[r * a.m];
        }
        if (header) {
            // move the scan's error bits into the status word; the next call's
            // scan starts from a fresh ticket and generation (no waits here:
            // both header words were loaded with the other inputs)
            if (k1) {
                atomicOr(a.status, k1);
                a.ws.hdr->k1_err = 0u;
            }
            a.ws.hdr->ticket = 0u;
            a.ws.hdr->epoch = (epoch + 1u) % kGenMask;
        }
    }
    const int64_t n_entries = static_cast<int64_t>(a.T) * a.K;
    // clamped: after a failed scan the offsets may be stale
    const int64_t n_valid = min(max(static_cast<int64_t>(s_eoff[a.E]), int64_t{0}), n_entries);
    const int64_t n_pairs = min(max(static_cast<int64_t>(s_poff[a.E]), int64_t{0}), a.capacity);
    bool bad = false;

    const float inv_k = 1.0f / static_cast<float>(a.K);     // i < 2^10 here: div_small is exact
    // entries: expert row; primaries (prank >= 0) also claim the token's receive row
    for (int i = tid; i < n; i += kFinalizeThreads) {
        const int e = s_idx[i];
        int32_t es = -1;
        if (e >= 0) {
            const int tl = div_small(i, inv_k);
            const int64_t v = static_cast<int64_t>(s_eoff[e]) + s_er[i];
            if (v >= 0 && v < n_valid) es = static_cast<int32_t>(v); else bad = true;
            if (s_pr[i] >= 0) {
                const int64_t rs = a.src_order ? static_cast<int64_t>(s_rank[e]) * a.T + s_pr[i]
                                               : static_cast<int64_t>(s_poff[e]) + s_pr[i];
                const bool in_range = a.src_order ? (s_pr[i] < a.T && rs < a.capacity) : (rs >= 0 && rs < n_pairs);
                if (in_range) {
                    s_rs[tl * a.R + s_rank[e]] = static_cast<int32_t>(rs);
                    a.recv_src_token[rs] = static_cast<int32_t>(t0 + tl);
                } else {
                    bad = true;
                }
            }
        }
        s_er[i] = es;
        a.expert_slot[e0 + i] = es;
    }
    __syncthreads();
    for (int i = tid; i < nt * a.R; i += kFinalizeThreads) a.recv_slot[t0 * a.R + i] = s_rs[i];
#pragma unroll
    for (int u = 0; u < kFinalizePerThread; ++u) {
        const int i = tid + u * kFinalizeThreads;
        if (i >= n) continue;
        const int e = s_idx[i];
        const int32_t es = s_er[i];
        if (e < 0 || es < 0) continue;
        const int tl = div_small(i, inv_k);
        a.expert_src_row[es] = s_rs[tl * a.R + s_rank[e]];
        a.expert_weight[es] = w_r[u];
    }

    // tails past the last used rows, spread over all blocks
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kFinalizeThreads + tid;
    const int64_t gstride = static_cast<int64_t>(gridDim.x) * kFinalizeThreads;
    if (a.src_order) {
        // the unused tail of every destination region
        for (int r = 0; r < a.R; ++r) {
            const int64_t used = min(max(static_cast<int64_t>(s_poff[(r + 1) * a.m] - s_poff[r * a.m]), int64_t{0}),
                                     static_cast<int64_t>(a.T));
            int32_t* region = a.recv_src_token + static_cast<int64_t>(r) * a.T;
            for (int64_t i = used + gtid; i < a.T; i += gstride) region[i] = -1;
        }
    } else {
        for (int64_t i = n_pairs + gtid; i < a.capacity; i += gstride) a.recv_src_token[i] = -1;
    }
    for (int64_t i = n_valid + gtid; i < n_entries; i += gstride) {
        a.expert_src_row[i] = -1;
        a.expert_weight[i] = 0.0f;
    }
    if (!a.src_order && s_poff[a.E] > a.capacity) bad = true;
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

// Multi-source layout: per destination r and source s, the first row of
// region r holding a token of source s or later.  Each region's used rows
// hold ascending token ids, so this is a lower bound of s * Ts in them.
struct SourceOffsetArgs {
    const int32_t* recv_src_token;
    const int32_t* tokens_per_rank;
    int32_t* recv_source_offset;     // [R, S+1]
    int32_t T, R, S, Ts;
};

// One warp per (destination r, source s): the first row of region r whose
// token is at least s * Ts, by a 32-way search.  Each step the lanes probe 32
// evenly spaced rows of the remaining range; the rows ascend, so the lanes
// below the target form a prefix and a ballot keeps the gap that holds the
// boundary: about log32 of the region's length dependent loads, not log2.
__global__ void __launch_bounds__(256)
layout_source_offsets_kernel(SourceOffsetArgs a) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t n = static_cast<int64_t>(a.R) * (a.S + 1);
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; i < n; i += warps) {
        const int r = static_cast<int>(i / (a.S + 1));
        const int s = static_cast<int>(i - static_cast<int64_t>(r) * (a.S + 1));
        const int32_t* rows = a.recv_src_token + static_cast<int64_t>(r) * a.T;
        const int32_t target = s * a.Ts;           // <= T
        // the first row >= target lies in [lo, hi] (hi: none of the rows is)
        int lo = 0, hi = min(max(a.tokens_per_rank[r], 0), a.T);
        while (hi > lo) {                          // warp-uniform
            const int len = hi - lo;
            if (len <= 32) {
                const bool below = lane < len && rows[lo + lane] < target;
                lo += __popc(__ballot_sync(0xffffffffu, below));
                break;
            }
            // 32 probes, strictly increasing, in [lo, hi)
            const int p = lo + static_cast<int>(static_cast<int64_t>(len) * (lane + 1) / 33);
            const int c = __popc(__ballot_sync(0xffffffffu, rows[p] < target));
            const int p_below = __shfl_sync(0xffffffffu, p, c > 0 ? c - 1 : 0);
            const int p_at = __shfl_sync(0xffffffffu, p, c < 32 ? c : 31);
            if (c > 0) lo = p_below + 1;           // rows[p_below] < target
            if (c < 32) hi = p_at;                 // rows[p_at] >= target
        }
        if (lane == 0) a.recv_source_offset[i] = lo;
    }
}

}  // namespace

int32_t default_tile_tokens(int32_t T, int32_t K) {
    int32_t tt = kMaxTileEntries / K;       // about 2048 entries per scan tile
    if (tt < 1) tt = 1;
    if (T > 0 && tt > T) tt = T;
    return tt;
}

size_t layout_workspace_bytes(int32_t T, int32_t K, int32_t E, int32_t num_tiles) {
    size_t b = sizeof(WsHeader);
    b = align_up(b + sizeof(uint32_t) * num_tiles, 256);
    b = align_up(b + sizeof(int32_t) * static_cast<size_t>(num_tiles) * vec_width(E), 256);
    b = align_up(b + sizeof(int32_t) * static_cast<size_t>(num_tiles) * vec_width(E), 256);
    b = align_up(b + sizeof(uint64_t) * static_cast<size_t>(min(num_tiles, tagged_tile_limit(E))) * vec_width(E), 256);
    b = align_up(b + sizeof(int32_t) * static_cast<size_t>(T) * K, 256);
    b = align_up(b + sizeof(int32_t) * static_cast<size_t>(T) * K, 256);
    return b;
}

LayoutWs layout_workspace(const moe_layout* L) {
    char* p = static_cast<char*>(L->workspace);
    LayoutWs ws;
    size_t off = 0;
    ws.hdr = reinterpret_cast<WsHeader*>(p + off);
    off += sizeof(WsHeader);
    ws.tile_flag = reinterpret_cast<uint32_t*>(p + off);
    off = align_up(off + sizeof(uint32_t) * L->num_tiles, 256);
    ws.tile_agg = reinterpret_cast<int32_t*>(p + off);
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(L->num_tiles) * vec_width(L->E), 256);
    ws.tile_incl = reinterpret_cast<int32_t*>(p + off);
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(L->num_tiles) * vec_width(L->E), 256);
    ws.tile_tagged = reinterpret_cast<uint64_t*>(p + off);
    off = align_up(off + sizeof(uint64_t) * static_cast<size_t>(min(L->num_tiles, tagged_tile_limit(L->E))) *
                             vec_width(L->E), 256);
    ws.erank = reinterpret_cast<int32_t*>(p + off);
    off = align_up(off + sizeof(int32_t) * static_cast<size_t>(L->T) * L->K, 256);
    ws.prank = reinterpret_cast<int32_t*>(p + off);
    return ws;
}

// SMs of the current device (0 if the query fails).
static int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

cudaError_t launch_layout(const int32_t* topk_idx, const float* topk_w, const moe_layout* L,
                          cudaStream_t stream, uint64_t timeout_ns, uint32_t debug_flags, bool early_trigger) {
    const LayoutWs ws = layout_workspace(L);
    ScanArgs sa;
    sa.topk_idx = topk_idx;
    sa.T = L->T; sa.K = L->K; sa.E = L->E; sa.m = L->E / L->R; sa.R = L->R;
    sa.tile_tokens = L->tile_tokens; sa.num_tiles = L->num_tiles;
    sa.ws = ws; sa.status = L->status;
    sa.timeout_ns = timeout_ns; sa.debug_flags = debug_flags;
    // Block-index tiles when all of them fit on the GPU at once.  In-process
    // A/B on GB300 (graph-replayed layout + dispatch + combine, flushed):
    // 150.4 -> 149.5 us at the DeepSeek-V3 shape, 135.3 -> 133.2 us Qwen-like,
    // 158.8 -> 156.1 us DeepSeek-16B-like.
    sa.by_block = L->num_tiles <= device_sm_count() ? 1 : 0;
    const bool src = L->num_sources > 0;
    size_t smem1 = sizeof(int32_t) * (kMaxTileEntries + (kLayoutWarps + 2) * static_cast<size_t>(vec_width(L->E)) +
                                      static_cast<size_t>(round_up4(L->E))) + sizeof(int4) * kLayoutThreads;
    if (L->E <= kMaxPeerE) smem1 += sizeof(uint32_t) * kLayoutWarps * kMaxPeerE;   // lane-mask tables
    const size_t table_bytes = sizeof(int32_t) * static_cast<size_t>(round_up4(L->tile_tokens * L->R));
    sa.prim_table = (static_cast<int64_t>(L->tile_tokens) * L->R <= kMaxPrimSlots &&
                     smem1 + table_bytes <= kMaxSmemPerBlock) ? 1 : 0;
    if (sa.prim_table) smem1 += table_bytes;
    const void* scan_fn = src ? reinterpret_cast<const void*>(layout_scan_kernel<true>)
                              : reinterpret_cast<const void*>(layout_scan_kernel<false>);
    cudaError_t err = cudaFuncSetAttribute(scan_fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem1));
    if (err != cudaSuccess) return err;
    err = src ? launch_pdl(layout_scan_kernel<true>, dim3(L->num_tiles), dim3(kLayoutThreads), smem1, stream, sa)
              : launch_pdl(layout_scan_kernel<false>, dim3(L->num_tiles), dim3(kLayoutThreads), smem1, stream, sa);
    if (err != cudaSuccess) return err;

    FinalArgs fa;
    fa.topk_idx = topk_idx; fa.topk_w = topk_w;
    fa.T = L->T; fa.K = L->K; fa.E = L->E; fa.R = L->R; fa.m = L->E / L->R;
    fa.src_order = src ? 1 : 0;
    fa.capacity = L->capacity; fa.num_tiles = L->num_tiles; fa.ws = ws; fa.status = L->status;
    fa.tokens_per_expert = L->tokens_per_expert;
    fa.expert_offset = L->expert_offset; fa.recv_expert_offset = L->recv_expert_offset;
    fa.tokens_per_rank = L->tokens_per_rank; fa.rank_offset = L->rank_offset;
    fa.recv_slot = L->recv_slot; fa.expert_slot = L->expert_slot; fa.recv_src_token = L->recv_src_token;
    fa.expert_src_row = L->expert_src_row; fa.expert_weight = L->expert_weight;
    fa.early_trigger = early_trigger ? 1 : 0;
    int64_t blocks = (static_cast<int64_t>(L->T) + kFinalizeTokens - 1) / kFinalizeTokens;
    if (blocks < 1) blocks = 1;
    const size_t smem2 = sizeof(int32_t) * (2 * (static_cast<size_t>(L->E) + 1) +
                                            3 * static_cast<size_t>(kFinalizeTokens) * L->K +
                                            static_cast<size_t>(kFinalizeTokens) * L->R + L->E);
    err = cudaFuncSetAttribute(layout_finalize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem2));
    if (err != cudaSuccess) return err;
    err = launch_pdl(layout_finalize_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kFinalizeThreads), smem2,
                     stream, fa);
    if (err != cudaSuccess || !src) return err;

    SourceOffsetArgs oa;
    oa.recv_src_token = L->recv_src_token;
    oa.tokens_per_rank = L->tokens_per_rank;
    oa.recv_source_offset = L->recv_source_offset;
    oa.T = L->T; oa.R = L->R; oa.S = L->num_sources; oa.Ts = L->source_tokens;
    const int64_t n = static_cast<int64_t>(L->R) * (L->num_sources + 1);    // one warp each
    const unsigned g3 = static_cast<unsigned>(std::min<int64_t>((n + 7) / 8, 1024));
    return launch_pdl(layout_source_offsets_kernel, dim3(g3), dim3(256), 0, stream, oa);
}

}  // namespace moe
