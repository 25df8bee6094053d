// dispatch_wide.cu -- MoE token dispatch with 32-byte vector accesses.
//
// The operator is the one of dispatch.cu ("Inside the Nebius + PyTorch
// DeepSeek V3 recipe", section "Mixture-of-experts and wide expert
// parallelism": every token row goes once to each virtual rank that holds one
// of its experts; "MoE / Hybrid-EP Validation", section "FP8 dispatch
// restriction": optionally quantised to FP8 in the same pass), with a work
// split shaped by what the quantised formats cost on GB300:
//
//   * an item is one 1024-column segment of one token; lane l of the warp
//     owns the 32 consecutive columns 32l .. 32l+31 of the segment and loads
//     them with two 32-byte loads (each load instruction of the warp touches
//     32 whole sectors, every sector of the 2 KB of bf16 exactly once);
//   * FP8 1x128: a block is four lanes (two shuffles for its amax); MXFP8
//     1x32: a block is one lane (no shuffle at all);
//   * a lane's 32 codes leave in ONE 32-byte store per destination row, so a
//     warp instruction writes 1 KB of one receive row; the block scales of
//     the segment (32 bytes) leave in one more store instruction;
//   * bf16 (no quantisation): the lane's 64 bytes leave in two 32-byte
//     stores per destination row;
//   * by default every warp takes one item (many short-lived CTAs, which the
//     block scheduler balances); with fewer channels (moe_tuning) each warp
//     takes a contiguous run of items (token-major), whose token / segment
//     indices advance by increments (no per-item division) and whose
//     destination list (the recv_slot row, one ballot) is reused by all of a
//     token's segments the warp holds;
//   * the next item's loads are issued once the current item is quantised,
//     before its stores.
//
// The block arithmetic is that of fp8_quant.cuh (IEEE-exact scale and
// quotients).  Magnitudes are quantised and the sign bits of the bf16 inputs
// are OR'ed into the code bytes afterwards: E4M3 is sign-magnitude and
// round-to-nearest-even with saturation is symmetric, so code(-v) =
// code(v) | 0x80 for every v, signed zero included.
//
// Alignment: every 32-byte access needs a 32-byte aligned address.  The
// launcher takes this kernel only when x and recv_x are 32-byte aligned and
// the row pitches keep them so (FP8 / MXFP8: hidden % 128 == 0; bf16:
// hidden % 16 == 0); otherwise it falls back to the 16-byte vector kernel.
#include <climits>

#include "fastdiv.h"
#include "fp8_quant.cuh"
#include "moe_common.cuh"

namespace moe {

namespace {

constexpr int kWideThreads = 256;
constexpr int kWideWarps = kWideThreads / 32;
constexpr int kWideSeg = 1024;          // columns per item
constexpr int kWideLaneCols = 32;       // columns per lane

struct WideArgs {
    const uint8_t* x;            // bf16 [T, H]
    uint8_t* recv;               // bf16 or E4M3 [capacity, H]
    uint8_t* recv_scales;        // FP8: fp32 [capacity, H/128]; MXFP8: E8M0 bytes [capacity, H/32]
    const int32_t* recv_slot;    // [T, R]
    int32_t T, H, R;
    int64_t capacity;
    int32_t nseg;                // segments per row
    int64_t n_items;             // T * nseg
    uint32_t* status;
    FastDiv seg_div;             // division by nseg
    int32_t items_fit_u32;       // every warp index of the one-item grid is below 2^32
};

// Token and segment of item i (one-item grids).
__device__ __forceinline__ void item_coords(const WideArgs& a, int64_t i, int32_t& t, int32_t& seg) {
    if (a.items_fit_u32) {
        const uint32_t q = fastdiv(static_cast<uint32_t>(i), a.seg_div);
        t = static_cast<int32_t>(q);
        seg = static_cast<int32_t>(static_cast<uint32_t>(i) - q * static_cast<uint32_t>(a.nseg));
    } else {
        t = static_cast<int32_t>(i / a.nseg);
        seg = static_cast<int32_t>(i - static_cast<int64_t>(t) * a.nseg);
    }
}

__device__ __forceinline__ void ld_v8(uint32_t* r, const void* p) {
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "l"(p));
}

__device__ __forceinline__ void st_v8(void* p, const uint32_t* r) {
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                 :: "l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                    "r"(r[7])
                 : "memory");
}

// One item in registers: the lane's 32 bf16 values (16 words, column order)
// and its entry of the token's recv_slot row (rank = lane; -1 past R).
struct WideItem {
    uint32_t w[16];
    int32_t slot;
    int32_t t;
    int32_t seg;
};

// The item's source columns only (x is an input of the call; the slots are
// the layout's output).
__device__ __forceinline__ void wide_load_x(WideItem& it, const WideArgs& a, int32_t t, int32_t seg, int lane) {
    it.t = t;
    it.seg = seg;
    const int col = seg * kWideSeg + lane * kWideLaneCols;
    const uint8_t* src = a.x + (static_cast<int64_t>(t) * a.H + col) * 2;
    if (col < a.H) {
        ld_v8(it.w, src);
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) it.w[j] = 0u;
    }
    if (col + 16 < a.H) {
        ld_v8(it.w + 8, src + 32);
    } else {
#pragma unroll
        for (int j = 8; j < 16; ++j) it.w[j] = 0u;
    }
}

// The lane's entry of the token's recv_slot row (rank = lane; -1 past R).
__device__ __forceinline__ int32_t wide_slot(const WideArgs& a, int32_t t, int lane) {
    return lane < a.R ? __ldg(a.recv_slot + static_cast<int64_t>(t) * a.R + lane) : -1;
}

__device__ __forceinline__ void wide_load(WideItem& it, const WideArgs& a, int32_t t, int32_t seg, int lane,
                                          int32_t prev_t, int32_t prev_slot) {
    // the slot row is fetched once per token the warp meets (warp-uniform test)
    it.slot = t == prev_t ? prev_slot : wide_slot(a, t, lane);
    wide_load_x(it, a, t, seg, lane);
}

// Largest magnitude of the lane's 32 values as a bf16 bit pattern; clears
// the sign bits of the words in place.
__device__ __forceinline__ uint32_t lane_absmax_inplace(uint32_t (&w)[16]) {
    uint32_t acc = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        w[j] &= 0x7fff7fffu;
        acc = __vmaxu2(acc, w[j]);
    }
    return max(acc & 0xffffu, acc >> 16);
}

// Sign bits of the four bf16 values in words (w0, w1) moved to bit 7 of the
// four code bytes (value order: w0 low, w0 high, w1 low, w1 high).
__device__ __forceinline__ uint32_t sign_bytes(uint32_t w0, uint32_t w1) {
    return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// FP8 1x128: the block of this lane is lanes 4b .. 4b+3.  `w` holds the
// lane's 32 values and is consumed (its sign bits are cleared); the codes
// replace it in codes[0..7].  Returns the scale.
__device__ __forceinline__ float wide_quant_fp8(uint32_t (&w)[16], uint32_t (&codes)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) codes[i] = sign_bytes(w[2 * i], w[2 * i + 1]);
    uint32_t mb = lane_absmax_inplace(w);
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float amax = __uint_as_float(mb << 16);
    const float s = block_scale(amax);
    if (mb == 0) {                       // an all-zero block: scale 0, codes 0x00
#pragma unroll
        for (int i = 0; i < 8; ++i) codes[i] = 0u;
        return s;
    }
    if (!amax_in_fast_range(amax)) {
        // rare: IEEE division, out of line (magnitudes; the signs are in codes)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint2 q = quantize8_ieee(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3], s);
            codes[2 * i] |= q.x;
            codes[2 * i + 1] |= q.y;
        }
        return s;
    }
    const float r = block_recip(s);
    const uint64_t r2 = pack_f32x2(r, r), ns2 = pack_f32x2(-s, -s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {     // the quotients two at a time (packed fp32)
        float v0, v1, v2, v3;
        unpack_f32x2(div_mag_by_scale_x2(bf16x2_to_f32x2(w[2 * i]), r2, ns2), v0, v1);
        unpack_f32x2(div_mag_by_scale_x2(bf16x2_to_f32x2(w[2 * i + 1]), r2, ns2), v2, v3);
        codes[i] |= e4m3x2(v0, v1) | (e4m3x2(v2, v3) << 16);
    }
    return s;
}

// MXFP8 1x32: the block is this lane's 32 values (`w`, consumed).  Returns
// the E8M0 byte.
__device__ __forceinline__ uint32_t wide_quant_mx(uint32_t (&w)[16], uint32_t (&codes)[8]) {
    uint32_t acc = 0;
#pragma unroll
    for (int j = 0; j < 16; ++j) acc = __vmaxu2(acc, w[j] & 0x7fff7fffu);
    const int se = mx_shared_exp(max(acc & 0xffffu, acc >> 16));
    const float mul = mx_inv_scale(se);
    const uint64_t mul2 = pack_f32x2(mul, mul);
#pragma unroll
    for (int i = 0; i < 8; ++i) {     // the products two at a time (packed fp32)
        float v0, v1, v2, v3;
        unpack_f32x2(mul_f32x2(bf16x2_to_f32x2(w[2 * i]), mul2), v0, v1);
        unpack_f32x2(mul_f32x2(bf16x2_to_f32x2(w[2 * i + 1]), mul2), v2, v3);
        codes[i] = e4m3x2(v0, v1) | (e4m3x2(v2, v3) << 16);
    }
    return static_cast<uint32_t>(se + 127);
}

// Quantise the item in place: FP8 / MXFP8 codes go to `codes` and the scale
// word (FP8: fp32 bits; MXFP8: the E8M0 byte) is returned; `it.w` is
// consumed.  bf16 items stay as they are.
template <int FMT>
__device__ __forceinline__ uint32_t wide_quant(WideItem& it, uint32_t (&codes)[8]) {
    if constexpr (FMT == 1) return __float_as_uint(wide_quant_fp8(it.w, codes));
    if constexpr (FMT == 2) return wide_quant_mx(it.w, codes);
    return 0u;
}

// Store one item to every destination row of token t: bf16 rows from `w`,
// or the codes and the scale word.
template <int FMT>
__device__ __forceinline__ void wide_emit(const WideArgs& a, int32_t t, int32_t seg, int32_t slot_lane,
                                          const uint32_t* w, const uint32_t (&codes)[8], uint32_t scale_word,
                                          int lane, bool& bad) {
    const int col = seg * kWideSeg + lane * kWideLaneCols;
    const bool in0 = col < a.H;
    const bool in1 = col + 16 < a.H;      // bf16 only: the lane's second 16 columns
    for (int rbase = 0; rbase < a.R; rbase += 32) {
        const int32_t my_slot =
            rbase == 0 ? slot_lane
                       : (lane + rbase < a.R ? __ldg(a.recv_slot + static_cast<int64_t>(t) * a.R + rbase + lane)
                                             : -1);
        if (my_slot >= a.capacity) bad = true;          // flagged, never written
        // walk only the ranks this token goes to
        uint32_t dests = __ballot_sync(0xffffffffu, my_slot >= 0 && my_slot < a.capacity);
        while (dests) {
            const int r = __ffs(dests) - 1;
            dests &= dests - 1;
            const int64_t slot = __shfl_sync(0xffffffffu, my_slot, r);
            if constexpr (FMT == 0) {
                uint8_t* dst = a.recv + (slot * a.H + col) * 2;
                if (in0) st_v8(dst, w);
                if (in1) st_v8(dst + 32, w + 8);
            } else {
                if (in0) st_v8(a.recv + slot * a.H + col, codes);
                if constexpr (FMT == 1) {
                    // scale of block col / 128, held by the block's first lane
                    if (in0 && (lane & 3) == 0)
                        reinterpret_cast<uint32_t*>(a.recv_scales)[slot * (a.H >> 7) + (col >> 7)] = scale_word;
                } else {
                    if (in0) a.recv_scales[slot * (a.H >> 5) + (col >> 5)] = static_cast<uint8_t>(scale_word);
                }
            }
        }
    }
}

// FMT 0: bf16 rows; 1: FP8 with fp32 1x128 scales; 2: MXFP8 (E8M0 1x32
// scales).  ONE: the default grid, exactly one item per warp (warp w takes
// item w), straight-line code: FP8 in 63 registers (four CTAs of 256 threads
// per SM; bounded to five it spills 28 bytes and measured 1-2 us slower at
// two of three shapes), MXFP8 and bf16 bounded to six CTAs per SM (40
// registers, no spill; MXFP8 0.5 us faster at the DeepSeek-V3 shape than at
// four, the same elsewhere).  Otherwise each
// warp takes a contiguous run of items with one item in registers: the next
// item's loads are issued as soon as the current one is quantised (bf16: once
// it is stored), before its stores, so the load latency overlaps the stores
// and the other warps' work; registers bounded to four CTAs per SM (FP8: 64
// registers and 12 bytes of spill).  Two items in registers per warp measured
// slower on GB300 at every shape: the registers they need cost occupancy or
// spill.
//
// EARLY (with ONE; moe_dispatch_with_layout only): x was complete before the
// layout's first kernel, so the warp loads its item -- and quantises it --
// before the dependency wait, while the layout still runs; only the slots
// and the stores wait for it.
template <int FMT, bool ONE, bool EARLY>
__global__ void __launch_bounds__(kWideThreads, (ONE && FMT != 1) ? 6 : 4)
dispatch_wide_kernel(WideArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * kWideWarps + (threadIdx.x >> 5);
    bool bad = false;
    if constexpr (EARLY) {
        static_assert(ONE, "early loads take the one-item grid");
        const bool live = warp_id < a.n_items;
        int32_t t = 0, seg = 0;
        if (live) item_coords(a, warp_id, t, seg);
        uint32_t codes[8];
        uint32_t sw = 0;
        WideItem it;
        if (live) {
            wide_load_x(it, a, t, seg, lane);
            sw = wide_quant<FMT>(it, codes);
        }
        pdl_wait();
        if (live) wide_emit<FMT>(a, t, seg, wide_slot(a, t, lane), it.w, codes, sw, lane, bad);
    } else if constexpr (ONE) {
        pdl_wait();
        if (warp_id < a.n_items) {
            int32_t t, seg;
            item_coords(a, warp_id, t, seg);
            uint32_t codes[8];
            WideItem it;
            wide_load(it, a, t, seg, lane, -1, -1);
            const uint32_t sw = wide_quant<FMT>(it, codes);
            wide_emit<FMT>(a, t, seg, it.slot, it.w, codes, sw, lane, bad);
        }
    } else {
        pdl_wait();
        const int64_t n_warps = static_cast<int64_t>(gridDim.x) * kWideWarps;
        const int64_t i0 = a.n_items * warp_id / n_warps;
        const int64_t i1 = a.n_items * (warp_id + 1) / n_warps;
        if (i0 < i1) {
            int n = static_cast<int>(i1 - i0);
            int32_t t = static_cast<int32_t>(i0 / a.nseg);
            int32_t seg = static_cast<int32_t>(i0 - static_cast<int64_t>(t) * a.nseg);
            uint32_t codes[8];
            WideItem it;
            wide_load(it, a, t, seg, lane, -1, -1);
            while (true) {
                const int32_t ct = it.t, cseg = it.seg, cslot = it.slot;
                if constexpr (FMT == 0) {
                    wide_emit<FMT>(a, ct, cseg, cslot, it.w, codes, 0u, lane, bad);
                    if (--n == 0) break;
                    if (++seg == a.nseg) { seg = 0; ++t; }
                    wide_load(it, a, t, seg, lane, ct, cslot);
                } else {
                    const uint32_t sw = wide_quant<FMT>(it, codes);
                    const bool more = n > 1;
                    if (more) {
                        if (++seg == a.nseg) { seg = 0; ++t; }
                        wide_load(it, a, t, seg, lane, ct, cslot);
                    }
                    wide_emit<FMT>(a, ct, cseg, cslot, nullptr, codes, sw, lane, bad);
                    if (--n == 0) break;
                }
            }
        }
    }
    pdl_trigger();
    // per warp, no CTA-wide barrier: a warp that is done leaves at once
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(a.status, MOE_DEVERR_CAPACITY);
}

}  // namespace

bool dispatch_wide_supported(const void* x, int32_t hidden, int32_t format, const void* recv_x) {
    const bool aligned = ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(recv_x)) & 31u) == 0;
    return aligned && (format == MOE_FORMAT_BF16 ? hidden % 16 == 0 : hidden % 128 == 0);
}

cudaError_t launch_dispatch_wide(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format, void* recv_x,
                                 void* recv_scales, cudaStream_t stream, int32_t num_channels, bool x_ready) {
    if (L->T == 0) return cudaSuccess;
    WideArgs a;
    a.x = reinterpret_cast<const uint8_t*>(x);
    a.recv = static_cast<uint8_t*>(recv_x);
    a.recv_scales = static_cast<uint8_t*>(recv_scales);
    a.recv_slot = L->recv_slot;
    a.T = L->T; a.H = hidden; a.R = L->R;
    a.capacity = L->capacity;
    a.nseg = (hidden + kWideSeg - 1) / kWideSeg;
    a.n_items = static_cast<int64_t>(L->T) * a.nseg;
    a.status = L->status;
    a.seg_div = make_fastdiv(static_cast<uint32_t>(a.nseg));
    a.items_fit_u32 = a.n_items + kWideWarps <= (int64_t{1} << 32) ? 1 : 0;
    // Default grid: one item per warp (the last CTA may hold fewer).  The
    // block scheduler then balances the tokens' unequal destination counts
    // CTA by CTA, and no warp of a CTA waits for a sibling with more items.
    // On GB300 (back-to-back launches over buffers larger than L2) this beat
    // four waves of CTAs holding about 1.5 items per warp by 1.2 us at the
    // DeepSeek-V3 shape (FP8 35.1 -> 33.9 us) and 1.7 us at the DeepSeek-16B-
    // like shape, and one persistent wave by 5-7 us; at the Zipf-skewed
    // Qwen-like shape two items per warp were 1.4 us faster.  CTAs of one or
    // two warps measured the same except where their sheer number (32,768
    // one-warp CTAs in 24 us) outran the CTA launch rate.
    const int64_t need = (a.n_items + kWideWarps - 1) / kWideWarps;     // one item per warp
    int64_t grid = num_channels > 0 ? num_channels : need;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    if (grid > INT32_MAX) return cudaErrorInvalidConfiguration;
    const dim3 g(static_cast<unsigned>(grid)), b(kWideThreads);
    if (grid == need && x_ready) {        // one item per warp, loaded before the dependency wait
        if (format == MOE_FORMAT_MXFP8) return launch_pdl(dispatch_wide_kernel<2, true, true>, g, b, 0, stream, a);
        if (format == MOE_FORMAT_FP8) return launch_pdl(dispatch_wide_kernel<1, true, true>, g, b, 0, stream, a);
        return launch_pdl(dispatch_wide_kernel<0, true, true>, g, b, 0, stream, a);
    }
    if (grid == need) {                   // one item per warp
        if (format == MOE_FORMAT_MXFP8) return launch_pdl(dispatch_wide_kernel<2, true, false>, g, b, 0, stream, a);
        if (format == MOE_FORMAT_FP8) return launch_pdl(dispatch_wide_kernel<1, true, false>, g, b, 0, stream, a);
        return launch_pdl(dispatch_wide_kernel<0, true, false>, g, b, 0, stream, a);
    }
    if (format == MOE_FORMAT_MXFP8) return launch_pdl(dispatch_wide_kernel<2, false, false>, g, b, 0, stream, a);
    if (format == MOE_FORMAT_FP8) return launch_pdl(dispatch_wide_kernel<1, false, false>, g, b, 0, stream, a);
    return launch_pdl(dispatch_wide_kernel<0, false, false>, g, b, 0, stream, a);
}

}  // namespace moe
