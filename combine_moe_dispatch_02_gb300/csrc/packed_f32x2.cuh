// packed_f32x2.cuh -- two fp32 values in one 64-bit register pair, for the
// packed instructions of sm_100+ (mul.rn.f32x2, fma.rn.f32x2).  Each packed
// instruction performs two independent IEEE round-to-nearest operations, so
// a packed step gives bit for bit what the scalar step gives on each half,
// in one instruction instead of two.
#pragma once

#include <cstdint>

namespace moe {

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// The two bf16 values of a word (low half first) as an fp32 pair (exact).
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
    return pack_f32x2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// a * b + c per half, one rounding each.
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

}  // namespace moe
