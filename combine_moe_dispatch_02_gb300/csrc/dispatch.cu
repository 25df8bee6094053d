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
//   * FP8 (TMA variant): the CTA's warps compute block amax, scale and E4M3
//     codes into an output stage, which TMA bulk stores send to every
//     destination row; the scales go out with plain stores.
// All three formats default to the 32-byte vector kernel of dispatch_wide.cu
// (no staging: each warp moves -- and for FP8 / MXFP8 quantises -- one
// 1024-column segment in registers and stores it straight to every
// destination row), which measured fastest for every format and shape on
// GB300.  Where the pointers are only 16-byte aligned, bf16 takes the TMA
// kernel below (variant 1) and FP8 / MXFP8 the 16-byte vector kernel
// (variant 2).  A warp-specialised TMA variant (one copy warp, eight
// quantiser warps) is kept as variant 3.
// x is read from HBM once; the receive rows are written once each.
#include <climits>

#include "fp8_quant.cuh"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kMaxStages = 8;
constexpr int kSlotBatchInts = 2048;     // recv_slot entries staged per batch
constexpr int kFp8Threads = 256;

struct DispatchArgs {
    const uint8_t* x;            // bf16 [T, H]
    uint8_t* recv;               // bf16 or E4M3 [capacity, H]
    uint32_t* recv_scales;       // [capacity, H/128] 32-bit scale words (FP8: fp32, MXFP8: 4 x E8M0)
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
    pdl_wait();
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
    int issued = min(S, rg.n);                  // warp-uniform

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
            ++issued;
        }
    }
    pdl_trigger();          // many waves: let the next kernel launch only as channels finish
    // Exit once the stores have read the stages (and, after a timeout, once
    // the loads still in flight have landed): the shared memory goes away with
    // the CTA, while kernel completion makes the global writes visible.
    bulk_wait_read<0>();
    if (timed_out) drain_ring_loads(bars, S, issued, a.timeout_ns);
    const uint32_t any_bad = __ballot_sync(0xffffffffu, bad);
    const uint32_t any_tmo = __ballot_sync(0xffffffffu, timed_out);
    if (lane == 0) {
        if (any_bad) atomicOr(a.status, MOE_DEVERR_CAPACITY);
        if (any_tmo) atomicOr(a.status, MOE_DEVERR_TIMEOUT);
    }
}

// FP8 E4M3 ------------------------------------------------------------------

// One item = one column chunk of one token.  A 128-column block is 256 bytes of
// bf16: sixteen lanes hold 16 bytes each, so a warp quantises two blocks at a
// time; the block amax is reduced across the half-warp.
// FMT 1: FP8 with one fp32 scale per 1x128 block; FMT 2: MXFP8 with four
// E8M0 bytes per 128 columns.  Either way one 32-bit scale word per 128-column
// group goes to each destination row.
template <int FMT>
__global__ void __launch_bounds__(kFp8Threads)
dispatch_fp8_kernel(DispatchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    const ItemRange rg = channel_items(a);
    if (rg.n <= 0) return;
    uint64_t* bars;
    int32_t* s_slots;
    uint8_t* rest;
    smem_carve(smem, a, &bars, &s_slots, &rest);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kWarps = kFp8Threads / 32;
    const int S = a.stages;
    const int nbc = a.chunk_elems / 128;                   // blocks per chunk
    const int nb_row = a.H / 128;
    uint32_t* s_scale = reinterpret_cast<uint32_t*>(rest);  // [S][nbc] scale words
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
    int issued = min(S, rg.n);                  // CTA-uniform

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

        // quantise: each group of eight lanes takes one 128-column block per
        // pass; lane li holds columns li*8.. and 64+li*8.. of the block
        const uint8_t* in = stage_in + static_cast<size_t>(s) * in_bytes;
        uint8_t* out = stage_out + static_cast<size_t>(s) * out_bytes;
        const int li = lane & 7;
        for (int base = warp * 4; base < nb; base += 4 * kWarps) {
            const int b = base + (lane >> 3);
            const bool active = b < nb;
            uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
            if (active) {
                va = *reinterpret_cast<const uint4*>(in + b * 256 + li * 16);
                vb = *reinterpret_cast<const uint4*>(in + b * 256 + 128 + li * 16);
            }
            uint2 q0, q1;
            uint32_t word;
            if constexpr (FMT == 1) {
                const BlockQuant bq = quantize_block_share(va, vb);
                q0 = bq.q0; q1 = bq.q1; word = __float_as_uint(bq.scale);
            } else {
                const MxQuant mq = quantize_group_share_mx(va, vb);
                q0 = mq.q0; q1 = mq.q1; word = mq.scales;
            }
            if (active) {
                *reinterpret_cast<uint2*>(out + b * 128 + li * 8) = q0;
                *reinterpret_cast<uint2*>(out + b * 128 + 64 + li * 8) = q1;
                if (li == 0) s_scale[s * nbc + b] = word;
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        // the input stage is free again: fetch item k+S into it
        if (k + S < rg.n) {
            if (tid == 0) issue_load(k + S);
            ++issued;
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
            a.recv_scales[static_cast<int64_t>(slot) * nb_row + c * nbc + b] = s_scale[s * nbc + b];   // 32-bit word
        }
    }
    pdl_trigger();
    if (warp == 0) bulk_wait_read<0>();     // stages read; completion publishes the writes
    if (timed_out) drain_ring_loads(bars, S, issued, a.timeout_ns);   // loads still in flight
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
    if (timed_out && tid == 0) atomicOr(a.status, MOE_DEVERR_TIMEOUT);
}

// Warp-specialised FP8 path --------------------------------------------------
//
// Roles inside one CTA, linked by mbarriers only (no CTA-wide barrier per
// item, so a slow warp delays only the store of its own item):
//   warp 0 (producer): TMA bulk loads of items into an input ring of
//     kWsInStages stages, and -- once an item is quantised -- one TMA bulk
//     store of the code row per destination plus the scale words; it prefetches
//     the next token's recv_slot row into a register while the current one is
//     being stored;
//   warps 1..kWsQuant (quantisers): each takes every kWsQuant-th group of four
//     128-column blocks of an item, reads the bf16 input stage, writes the code
//     stage and the scale words.
// Barriers per stage: in_full (TMA bytes), in_empty (one arrive per quantiser
// warp), out_full (one arrive per quantiser warp), out_empty (producer, after
// the bulk stores have read the stage).  Every wait is bounded.
constexpr int kWsQuant = 8;
constexpr int kWsThreads = 32 * (1 + kWsQuant);
constexpr int kWsInStages = 4;
constexpr int kWsOutStages = 3;

template <int FMT>
__global__ void __launch_bounds__(kWsThreads)
dispatch_fp8_ws_kernel(DispatchArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    pdl_wait();
    const ItemRange rg = channel_items(a);
    if (rg.n <= 0) return;
    uint64_t* in_full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* in_empty = in_full + kWsInStages;
    uint64_t* out_full = in_empty + kWsInStages;
    uint64_t* out_empty = out_full + kWsOutStages;
    const int nbc = a.chunk_elems / 128;                      // 128-column groups per chunk
    uint32_t* s_scale = reinterpret_cast<uint32_t*>(smem + 256);            // [kWsOutStages][nbc]
    uint8_t* stage_in = smem + 256 + align_up(sizeof(uint32_t) * kWsOutStages * nbc, 128);
    const uint32_t in_bytes = static_cast<uint32_t>(a.chunk_elems) * 2u;
    uint8_t* stage_out = stage_in + static_cast<size_t>(kWsInStages) * in_bytes;
    const uint32_t out_bytes = static_cast<uint32_t>(a.chunk_elems);
    const int64_t x_row_bytes = static_cast<int64_t>(a.H) * 2;
    const int nb_row = a.H / 128;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int s = 0; s < kWsInStages; ++s) { mbar_init(&in_full[s], 1); mbar_init(&in_empty[s], kWsQuant); }
        for (int s = 0; s < kWsOutStages; ++s) { mbar_init(&out_full[s], kWsQuant); mbar_init(&out_empty[s], 1); }
        fence_mbar_init();
    }
    __syncthreads();

    auto item_of = [&](int k, int64_t* t, int* c, int* elems) {
        const int64_t i = rg.i0 + k;
        *t = i / a.nchunk;
        *c = static_cast<int>(i - *t * a.nchunk);
        *elems = min(a.chunk_elems, a.H - *c * a.chunk_elems);
    };
    bool timed_out = false, bad = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        auto issue_load = [&](int k) {           // lane 0 only
            int64_t t; int c, elems;
            item_of(k, &t, &c, &elems);
            const int s = k % kWsInStages;
            mbar_arrive_expect_tx(&in_full[s], static_cast<uint32_t>(elems) * 2u);
            bulk_g2s(stage_in + static_cast<size_t>(s) * in_bytes,
                     a.x + t * x_row_bytes + static_cast<int64_t>(c) * a.chunk_elems * 2,
                     static_cast<uint32_t>(elems) * 2u, &in_full[s]);
        };
        if (lane == 0)
            for (int k = 0; k < kWsInStages - 1 && k < rg.n; ++k) issue_load(k);
        int issued = min(kWsInStages - 1, rg.n);               // warp-uniform
        int64_t t_cur; int c_cur, e_cur;
        item_of(0, &t_cur, &c_cur, &e_cur);
        int32_t slot_next = (a.R <= 32 && lane < a.R) ? __ldg(a.recv_slot + t_cur * a.R + lane) : -1;
        int64_t slot_tok = t_cur;
        for (int k = 0; k < rg.n; ++k) {
            int64_t t; int c, elems;
            item_of(k, &t, &c, &elems);
            // keep the input ring kWsInStages - 1 items ahead
            const int kl = k + kWsInStages - 1;
            if (kl < rg.n) {
                bool ok = true;
                if (kl >= kWsInStages)
                    ok = mbar_wait_bounded(&in_empty[kl % kWsInStages],
                                           static_cast<uint32_t>(kl / kWsInStages - 1) & 1u, a.timeout_ns);
                if (__any_sync(0xffffffffu, !ok)) { timed_out = true; break; }
                if (lane == 0) { fence_proxy_async_smem(); issue_load(kl); }
                ++issued;
            }
            // slots of this item's token (prefetched when the token started)
            int32_t my_slot = slot_next;
            if (t != slot_tok) {
                my_slot = (a.R <= 32 && lane < a.R) ? __ldg(a.recv_slot + t * a.R + lane) : -1;
            }
            // prefetch the slots of the next item's token
            if (k + 1 < rg.n) {
                int64_t tn; int cn, en;
                item_of(k + 1, &tn, &cn, &en);
                if (tn != t) slot_next = (a.R <= 32 && lane < a.R) ? __ldg(a.recv_slot + tn * a.R + lane) : -1;
                else slot_next = my_slot;
                slot_tok = tn;
            }
            const int o = k % kWsOutStages;
            const bool got = mbar_wait_bounded(&out_full[o], static_cast<uint32_t>(k / kWsOutStages) & 1u, a.timeout_ns);
            if (__any_sync(0xffffffffu, !got)) { timed_out = true; break; }
            const int nb = elems / 128;
            const uint8_t* outp = stage_out + static_cast<size_t>(o) * out_bytes;
            for (int rbase = 0; rbase < a.R; rbase += 32) {
                const int32_t sl = (a.R <= 32) ? my_slot
                                               : (rbase + lane < a.R ? __ldg(a.recv_slot + t * a.R + rbase + lane) : -1);
                if (sl >= a.capacity) bad = true;
                if (sl >= 0 && sl < a.capacity)
                    bulk_s2g(a.recv + static_cast<int64_t>(sl) * a.H + static_cast<int64_t>(c) * a.chunk_elems, outp,
                             static_cast<uint32_t>(elems));
                // scale words of this chunk to every destination
                const int nr = min(32, a.R - rbase);
                for (int r = 0; r < nr; ++r) {
                    const int32_t sr = __shfl_sync(0xffffffffu, sl, r);
                    if (sr < 0 || sr >= a.capacity) continue;
                    for (int b = lane; b < nb; b += 32)
                        a.recv_scales[static_cast<int64_t>(sr) * nb_row + c * nbc + b] = s_scale[o * nbc + b];
                }
            }
            bulk_commit();
            // release the output stage of the previous item once its stores have read it
            if (k >= 1) {
                bulk_wait_read<1>();
                __syncwarp();
                if (lane == 0) mbar_arrive(&out_empty[(k - 1) % kWsOutStages]);
            }
        }
        bulk_wait_read<0>();                 // stages read; completion publishes the writes
        // After a timeout, loads may still be landing in the input ring: wait
        // (bounded) for the last load issued into each stage before exiting.
        if (!drain_ring_loads(in_full, kWsInStages, issued, a.timeout_ns)) timed_out = true;
    } else {
        // ----------------------------------------------------------- quantisers
        const int q = warp - 1;
        const int li = lane & 7;
        for (int k = 0; k < rg.n; ++k) {
            int64_t t; int c, elems;
            item_of(k, &t, &c, &elems);
            const int s = k % kWsInStages, o = k % kWsOutStages;
            bool ok = mbar_wait_bounded(&in_full[s], static_cast<uint32_t>(k / kWsInStages) & 1u, a.timeout_ns);
            if (ok && k >= kWsOutStages)
                ok = mbar_wait_bounded(&out_empty[o], static_cast<uint32_t>(k / kWsOutStages - 1) & 1u, a.timeout_ns);
            if (__any_sync(0xffffffffu, !ok)) { timed_out = true; break; }
            const int nb = elems / 128;
            const uint8_t* in = stage_in + static_cast<size_t>(s) * in_bytes;
            uint8_t* out = stage_out + static_cast<size_t>(o) * out_bytes;
            for (int base = q * 4; base < nb; base += 4 * kWsQuant) {
                const int b = base + (lane >> 3);
                const bool active = b < nb;
                uint4 va = make_uint4(0u, 0u, 0u, 0u), vb = va;
                if (active) {
                    va = *reinterpret_cast<const uint4*>(in + b * 256 + li * 16);
                    vb = *reinterpret_cast<const uint4*>(in + b * 256 + 128 + li * 16);
                }
                uint2 q0, q1;
                uint32_t word;
                if constexpr (FMT == 1) {
                    const BlockQuant bq = quantize_block_share(va, vb);
                    q0 = bq.q0; q1 = bq.q1; word = __float_as_uint(bq.scale);
                } else {
                    const MxQuant mq = quantize_group_share_mx(va, vb);
                    q0 = mq.q0; q1 = mq.q1; word = mq.scales;
                }
                if (active) {
                    *reinterpret_cast<uint2*>(out + b * 128 + li * 8) = q0;
                    *reinterpret_cast<uint2*>(out + b * 128 + 64 + li * 8) = q1;
                    if (li == 0) s_scale[o * nbc + b] = word;
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&in_empty[s]);
                mbar_arrive(&out_full[o]);
            }
        }
    }
    pdl_trigger();
    if (__syncthreads_or(bad) && tid == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
    if (__syncthreads_or(timed_out) && tid == 0) atomicOr(a.status, MOE_DEVERR_TIMEOUT);
}

// 16-byte vector path ------------------------------------------------------

// No shared-memory staging: a warp moves one 512-column segment of one token
// per item.  Each lane loads two 16-byte vectors.  bf16: lane l takes columns
// l*8 and 256 + l*8 of the segment.  FP8 / MXFP8: the eight lanes 8g..8g+7
// hold 128-column block g of the segment, lane li its columns li*16 ..
// li*16+15, and reduce the block amax with shuffles; each lane then writes its
// 16 codes with one 16-byte store per destination row (eight lanes fill a
// whole 128-byte line).  U items (2 or 4) are in flight per warp (all
// their loads are issued before any store).  The destination rows come from
// recv_slot: lane r holds the slot of rank r and the warp walks the ranks with
// shuffles.
constexpr int kLsuThreads = 256;
constexpr int kLsuWaves = 4;
constexpr int kSegElems = 512;

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

template <int FMT>
__device__ __forceinline__ int lsu_col(int col0, int lane, int j) {
    if constexpr (FMT != 0) return col0 + (lane >> 3) * 128 + (lane & 7) * 16 + j * 8;
    return col0 + j * 256 + lane * 8;
}

// One batch: U items of a warp (item = one 512-column segment of one token),
// their source vectors and the lane's recv_slot entry.
template <int U>
struct LsuBatch {
    uint4 v[U][2];
    int32_t slot_lane[U];
    int64_t tok[U];
    int col0[U];
    bool live[U];
};

template <int FMT, int U>
__device__ __forceinline__ void lsu_load(LsuBatch<U>& b, const DispatchArgs& a, int64_t item0, int64_t n_warps,
                                         int64_t n_items, int nseg, int lane) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t item = item0 + u * n_warps;
        b.live[u] = item < n_items;                      // warp-uniform
        const int64_t t = b.live[u] ? item / nseg : 0;
        const int g = b.live[u] ? static_cast<int>(item - t * nseg) : 0;
        b.tok[u] = t;
        b.col0[u] = g * kSegElems;
        b.slot_lane[u] = (b.live[u] && lane < a.R) ? __ldg(a.recv_slot + t * a.R + lane) : -1;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int col = lsu_col<FMT>(b.col0[u], lane, j);
            b.v[u][j] = (b.live[u] && col < a.H) ? ld_nc_v4(a.x + (t * a.H + col) * 2) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

template <int FMT, int U>
__device__ __forceinline__ void lsu_store(const LsuBatch<U>& b, const DispatchArgs& a, int nb_row, int lane,
                                          bool& bad) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        if (!b.live[u]) continue;
        const int64_t t = b.tok[u];
        uint2 q0 = make_uint2(0u, 0u), q1 = q0;
        uint32_t word = 0;
        if constexpr (FMT == 1) {
            const BlockQuant bq = quantize_block_share(b.v[u][0], b.v[u][1]);
            q0 = bq.q0; q1 = bq.q1; word = __float_as_uint(bq.scale);
        } else if constexpr (FMT == 2) {
            const MxQuant mq = quantize_group_share_mx16(b.v[u][0], b.v[u][1]);
            q0 = mq.q0; q1 = mq.q1; word = mq.scales;
        }
        const uint4 q = make_uint4(q0.x, q0.y, q1.x, q1.y);     // the lane's 16 consecutive codes
        // this lane's two column offsets (the same for every destination row)
        const int c0 = lsu_col<FMT>(b.col0[u], lane, 0), c1 = lsu_col<FMT>(b.col0[u], lane, 1);
        const bool in0 = c0 < a.H, in1 = c1 < a.H;
        const bool scale_lane = FMT != 0 && in0 && (lane & 7) == 0;
        for (int rbase = 0; rbase < a.R; rbase += 32) {
            const int32_t my_slot = rbase == 0 ? b.slot_lane[u]
                                               : (lane + rbase < a.R ? __ldg(a.recv_slot + t * a.R + rbase + lane) : -1);
            if (my_slot >= a.capacity) bad = true;          // flagged, never written
            // walk only the ranks this token goes to
            uint32_t dests = __ballot_sync(0xffffffffu, my_slot >= 0 && my_slot < a.capacity);
            while (dests) {
                const int r = __ffs(dests) - 1;
                dests &= dests - 1;
                const int64_t slot = __shfl_sync(0xffffffffu, my_slot, r);
                if constexpr (FMT != 0) {
                    uint8_t* row = a.recv + slot * a.H;
                    if (in0) *reinterpret_cast<uint4*>(row + c0) = q;     // c1 = c0 + 8: one 16-byte store
                    if (scale_lane) a.recv_scales[slot * nb_row + (c0 >> 7)] = word;
                } else {
                    uint8_t* row = a.recv + slot * a.H * 2;
                    if (in0) *reinterpret_cast<uint4*>(row + c0 * 2) = b.v[u][0];
                    if (in1) *reinterpret_cast<uint4*>(row + c1 * 2) = b.v[u][1];
                }
            }
        }
    }
}

// FMT 0: bf16 rows; 1: FP8 with fp32 1x128 scales; 2: MXFP8 (E8M0 1x32 scales).
// Software-pipelined in batches of U items per warp: the next batch's loads
// are issued before the current batch is quantised and stored, so the load
// latency overlaps the arithmetic and the stores (2U items in flight).
// Registers for U = 1 (the default): MXFP8 is held to five CTAs per SM (48
// registers, 4 bytes of spill), which on GB300 beat four CTAs (60 registers) by
// 0.5-1.0 us on all three full-size shapes; FP8 and bf16 are held to four (FP8:
// 64 registers, as fast as before; at five it spills 16 bytes and measured up
// to 0.8 us slower).  Deeper batches keep their registers (bounded to four or
// five CTAs they spill hundreds of bytes).
template <int FMT, int U>
__global__ void __launch_bounds__(kLsuThreads, U == 1 ? (FMT == 2 ? 5 : 4) : 1)
dispatch_lsu_kernel(DispatchArgs a) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = (static_cast<int64_t>(blockIdx.x) * kLsuThreads + threadIdx.x) >> 5;
    const int64_t n_warps = (static_cast<int64_t>(gridDim.x) * kLsuThreads) >> 5;
    const int nseg = (a.H + kSegElems - 1) / kSegElems;
    const int64_t n_items = static_cast<int64_t>(a.T) * nseg;
    const int nb_row = a.H / 128;
    const int64_t stride = U * n_warps;
    bool bad = false;
    LsuBatch<U> cur, nxt;
    int64_t item0 = warp_id;
    lsu_load<FMT, U>(cur, a, item0, n_warps, n_items, nseg, lane);
    while (item0 < n_items) {
        // two batches per trip, so that the buffers swap roles without copies
        lsu_load<FMT, U>(nxt, a, item0 + stride, n_warps, n_items, nseg, lane);
        lsu_store<FMT, U>(cur, a, nb_row, lane, bad);
        item0 += stride;
        if (item0 >= n_items) break;
        lsu_load<FMT, U>(cur, a, item0 + stride, n_warps, n_items, nseg, lane);
        lsu_store<FMT, U>(nxt, a, nb_row, lane, bad);
        item0 += stride;
    }
    pdl_trigger();
    if (__syncthreads_or(bad) && threadIdx.x == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

}  // namespace

cudaError_t launch_dispatch(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format,
                            void* recv_x, void* recv_scales, cudaStream_t stream,
                            int32_t num_channels, int32_t stages, int32_t chunk_bytes, int32_t variant,
                            uint64_t timeout_ns, bool x_ready) {
    if (L->T == 0) return cudaSuccess;
    // The default and variant 4: the 32-byte vector kernel (dispatch_wide.cu);
    // where the pointers or the row pitch do not keep 32-byte alignment, the
    // 16-byte kernels: TMA staging for bf16 (variant 1), the 16-byte vector
    // kernel for FP8 / MXFP8 (variant 2)
    if (variant == 4 || variant == 0) {
        if (dispatch_wide_supported(x, hidden, format, recv_x))
            return launch_dispatch_wide(x, hidden, L, format, recv_x, recv_scales, stream, num_channels, x_ready);
        variant = format == MOE_FORMAT_BF16 ? 1 : 2;
    }
    DispatchArgs a;
    a.x = reinterpret_cast<const uint8_t*>(x);
    a.recv = static_cast<uint8_t*>(recv_x);
    a.recv_scales = static_cast<uint32_t*>(recv_scales);
    a.recv_slot = L->recv_slot;
    const bool fp8 = format != MOE_FORMAT_BF16;
    a.T = L->T; a.H = hidden; a.R = L->R;
    a.capacity = L->capacity;
    a.status = L->status;
    a.timeout_ns = timeout_ns;
    // column chunks: at most chunk_bytes (default 16 KB) of bf16 input per stage
    const int32_t max_elems = (chunk_bytes > 0 ? chunk_bytes : 16384) / 2;
    const int32_t gran = fp8 ? 128 : 8;
    a.nchunk = (hidden + max_elems - 1) / max_elems;
    a.chunk_elems = ((hidden + a.nchunk - 1) / a.nchunk + gran - 1) / gran * gran;
    a.nchunk = (hidden + a.chunk_elems - 1) / a.chunk_elems;   // every chunk non-empty
    // Channels: by default many short ones (one item each for bf16, about 4
    // for FP8): each CTA issues the loads of all its items at once, and the
    // scheduler keeps every SM full while earlier channels drain their stores
    // (measured on GB300: one item per channel beats two by ~3 us at the
    // DeepSeek-V3 shape).
    const int64_t n_items = static_cast<int64_t>(L->T) * a.nchunk;
    int64_t grid = num_channels > 0 ? num_channels : (fp8 ? (n_items + 3) / 4 : n_items);
    if (grid > n_items) grid = n_items;
    if (grid < 1) grid = 1;
    const int64_t items_per_channel = (n_items + grid - 1) / grid;
    int S = stages > 0 ? stages : (fp8 ? 3 : 4);
    if (S > items_per_channel) S = static_cast<int>(items_per_channel);   // no unused stages
    // one stage only when every channel holds exactly one item (no refill)
    if (S < 2 && items_per_channel > 1) S = 2;
    if (S > kMaxStages) S = kMaxStages;
    a.stages = S;
    // recv_slot rows staged per batch: at most the tokens one channel spans
    int64_t slot_tokens = items_per_channel / a.nchunk + 2;
    if (slot_tokens > kSlotBatchInts / L->R) slot_tokens = kSlotBatchInts / L->R;
    a.slot_batch = slot_tokens < 1 ? 1 : static_cast<int32_t>(slot_tokens);

    size_t smem = align_up(8 * kMaxStages + sizeof(int32_t) * static_cast<size_t>(a.slot_batch) * a.R, 128);
    if (fp8) {
        const int nbc = a.chunk_elems / 128;
        smem += align_up(sizeof(float) * S * nbc, 128) + static_cast<size_t>(S) * a.chunk_elems * 3;
    } else {
        smem += static_cast<size_t>(S) * a.chunk_elems * 2;
    }
    if (variant == 2 || (fp8 && variant == 0)) {
        // 16-byte vector path (the FP8 / MXFP8 default): persistent grid, occupancy-limited.
        // Items in flight per warp = 2U (two pipelined batches of U): stages 2 -> U = 1,
        // 4 -> U = 2, 8 -> U = 4; the default is U = 1.
        const int U = stages >= 8 ? 4 : stages >= 4 ? 2 : 1;
        const void* fn = U == 4 ? (format == MOE_FORMAT_MXFP8 ? reinterpret_cast<const void*>(dispatch_lsu_kernel<2, 4>)
                                   : fp8 ? reinterpret_cast<const void*>(dispatch_lsu_kernel<1, 4>)
                                         : reinterpret_cast<const void*>(dispatch_lsu_kernel<0, 4>))
                       : U == 2 ? (format == MOE_FORMAT_MXFP8 ? reinterpret_cast<const void*>(dispatch_lsu_kernel<2, 2>)
                                   : fp8 ? reinterpret_cast<const void*>(dispatch_lsu_kernel<1, 2>)
                                         : reinterpret_cast<const void*>(dispatch_lsu_kernel<0, 2>))
                                : (format == MOE_FORMAT_MXFP8 ? reinterpret_cast<const void*>(dispatch_lsu_kernel<2, 1>)
                                   : fp8 ? reinterpret_cast<const void*>(dispatch_lsu_kernel<1, 1>)
                                         : reinterpret_cast<const void*>(dispatch_lsu_kernel<0, 1>));
        int per_sm = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kLsuThreads, 0);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        const int64_t nseg = (hidden + kSegElems - 1) / kSegElems;
        const int64_t warps_needed = (static_cast<int64_t>(L->T) * nseg + U - 1) / U;
        // four waves of resident CTAs by default (GB300: FP8 and MXFP8 as fast as
        // or faster than one persistent wave on all three full-size shapes)
        int64_t lsu_grid = num_channels > 0 ? num_channels : static_cast<int64_t>(sm_count()) * per_sm * kLsuWaves;
        const int64_t need = (warps_needed * 32 + kLsuThreads - 1) / kLsuThreads;
        if (lsu_grid > need) lsu_grid = need;
        if (lsu_grid < 1) lsu_grid = 1;
        const dim3 g(static_cast<unsigned>(lsu_grid)), b(kLsuThreads);
        if (U == 4) {
            if (format == MOE_FORMAT_MXFP8) return launch_pdl(dispatch_lsu_kernel<2, 4>, g, b, 0, stream, a);
            if (fp8) return launch_pdl(dispatch_lsu_kernel<1, 4>, g, b, 0, stream, a);
            return launch_pdl(dispatch_lsu_kernel<0, 4>, g, b, 0, stream, a);
        }
        if (U == 2) {
            if (format == MOE_FORMAT_MXFP8) return launch_pdl(dispatch_lsu_kernel<2, 2>, g, b, 0, stream, a);
            if (fp8) return launch_pdl(dispatch_lsu_kernel<1, 2>, g, b, 0, stream, a);
            return launch_pdl(dispatch_lsu_kernel<0, 2>, g, b, 0, stream, a);
        }
        if (format == MOE_FORMAT_MXFP8) return launch_pdl(dispatch_lsu_kernel<2, 1>, g, b, 0, stream, a);
        if (fp8) return launch_pdl(dispatch_lsu_kernel<1, 1>, g, b, 0, stream, a);
        return launch_pdl(dispatch_lsu_kernel<0, 1>, g, b, 0, stream, a);
    }
    if (fp8 && variant == 3) {
        const int nbc = a.chunk_elems / 128;
        const size_t smem_ws = 256 + align_up(sizeof(uint32_t) * kWsOutStages * nbc, 128) +
                               static_cast<size_t>(kWsInStages) * a.chunk_elems * 2 +
                               static_cast<size_t>(kWsOutStages) * a.chunk_elems;
        const void* fnw = format == MOE_FORMAT_MXFP8 ? reinterpret_cast<const void*>(dispatch_fp8_ws_kernel<2>)
                                                     : reinterpret_cast<const void*>(dispatch_fp8_ws_kernel<1>);
        cudaError_t e = cudaFuncSetAttribute(fnw, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem_ws));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fnw, kWsThreads, smem_ws);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        int64_t g = num_channels > 0 ? num_channels : static_cast<int64_t>(sm_count()) * per_sm;
        if (g > n_items) g = n_items;
        if (g < 1) g = 1;
        if (format == MOE_FORMAT_MXFP8)
            return launch_pdl(dispatch_fp8_ws_kernel<2>, dim3(static_cast<unsigned>(g)), dim3(kWsThreads), smem_ws,
                              stream, a);
        return launch_pdl(dispatch_fp8_ws_kernel<1>, dim3(static_cast<unsigned>(g)), dim3(kWsThreads), smem_ws,
                          stream, a);
    }
    const void* fn = format == MOE_FORMAT_MXFP8 ? reinterpret_cast<const void*>(dispatch_fp8_kernel<2>)
                     : fp8 ? reinterpret_cast<const void*>(dispatch_fp8_kernel<1>)
                           : reinterpret_cast<const void*>(dispatch_bf16_kernel);
    const int threads = fp8 ? kFp8Threads : 32;
    cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    if (format == MOE_FORMAT_MXFP8)
        return launch_pdl(dispatch_fp8_kernel<2>, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, a);
    if (fp8) return launch_pdl(dispatch_fp8_kernel<1>, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, a);
    return launch_pdl(dispatch_bf16_kernel, dim3(static_cast<unsigned>(grid)), dim3(threads), smem, stream, a);
}

}  // namespace moe
