// Test-only kernel: checks the dispatch kernels' fast FP8 arithmetic against
// CUDA's IEEE operations, for a list of bf16 block maxima amax:
//   scale:      moe::block_scale(amax)  vs __fdiv_rn(amax, 448)  (every amax)
//   reciprocal: moe::block_recip(s)     vs __frcp_rn(s)          (fast range)
//   quotient:   moe::div_by_scale(x, s, r) vs __fdiv_rn(x, s) for every bf16
//               x with |x| <= amax, bit for bit where |x| >= 2^-100 and
//               |x/s| >= 2^-100 (the claimed exact range),
//   codes:      their E4M3 codes, everywhere;
//   magnitude:  moe::div_mag_by_scale(|x|, s, r) vs __fdiv_rn(|x|, s) under
//               the same exactness condition, and the E4M3 code of that
//               quotient with the sign bit of x OR'ed in vs the code of
//               __fdiv_rn(x, s), everywhere;
//   packed:     moe::div_mag_by_scale_x2 on the pair (|x|, |x'|), x' another
//               bf16 value, vs moe::div_mag_by_scale on each half, bit for
//               bit everywhere (the packed fp32 instructions round each half
//               like the scalar ones).
// The first few quotient and code mismatches are recorded.  Every index is
// bounded by the array sizes.
#include <cstdint>

#include "fp8_quant.cuh"

namespace {

__device__ void record(unsigned long long* counter, uint32_t* examples, int max_examples, uint32_t a,
                       uint32_t b, uint32_t c, uint32_t d) {
    const unsigned long long slot = atomicAdd(counter, 1ull);
    if (slot < static_cast<unsigned long long>(max_examples)) {
        examples[4 * slot + 0] = a;
        examples[4 * slot + 1] = b;
        examples[4 * slot + 2] = c;
        examples[4 * slot + 3] = d;
    }
}

__global__ void div_check_kernel(const uint16_t* amax_bits, int n_amax, unsigned long long* counters,
                                 uint32_t* examples, int max_examples) {
    const int a_idx = blockIdx.y;
    if (a_idx >= n_amax) return;
    const float amax = __uint_as_float(static_cast<uint32_t>(amax_bits[a_idx]) << 16);
    const float s = __fdiv_rn(amax, 448.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if (__float_as_uint(moe::block_scale(amax)) != __float_as_uint(s)) atomicAdd(&counters[3], 1ull);
        if (moe::amax_in_fast_range(amax) && __float_as_uint(moe::block_recip(s)) != __float_as_uint(__frcp_rn(s)))
            atomicAdd(&counters[4], 1ull);
    }
    if (!moe::amax_in_fast_range(amax)) return;
    const float r = moe::block_recip(s);
    unsigned local_n = 0;
    for (uint32_t xb = blockIdx.x * blockDim.x + threadIdx.x; xb < 65536u; xb += gridDim.x * blockDim.x) {
        const float x = __uint_as_float(xb << 16);
        if (!(fabsf(x) <= amax)) continue;            // skips NaN and values beyond the block max
        ++local_n;
        const float q_fast = moe::div_by_scale(x, s, r);
        const float q_ieee = __fdiv_rn(x, s);
        const bool in_range = x == 0.0f || (fabsf(x) >= 0x1p-100f && fabsf(q_ieee) >= 0x1p-100f);
        if (in_range && __float_as_uint(q_fast) != __float_as_uint(q_ieee))
            record(&counters[0], examples, max_examples, amax_bits[a_idx], xb, __float_as_uint(q_fast),
                   __float_as_uint(q_ieee));
        const uint32_t c_fast = moe::e4m3x2(q_fast, 0.0f) & 0xffu;
        const uint32_t c_ieee = moe::e4m3x2(q_ieee, 0.0f) & 0xffu;
        if (c_fast != c_ieee)
            record(&counters[1], examples + 4 * max_examples, max_examples, amax_bits[a_idx], xb, c_fast, c_ieee);
        const float m = fabsf(x);
        const float qm_fast = moe::div_mag_by_scale(m, s, r);
        if (in_range && __float_as_uint(qm_fast) != __float_as_uint(__fdiv_rn(m, s))) atomicAdd(&counters[5], 1ull);
        const uint32_t cm = (moe::e4m3x2(qm_fast, 0.0f) & 0xffu) | ((xb >> 8) & 0x80u);
        if (cm != c_ieee) atomicAdd(&counters[6], 1ull);
        float m2 = fabsf(__uint_as_float(((xb * 40503u) & 0xffffu) << 16));   // another bf16 value
        if (!(m2 <= 0x1.fffffep127f)) m2 = m;                                   // finite ones only
        float p0, p1;
        moe::unpack_f32x2(moe::div_mag_by_scale_x2(moe::pack_f32x2(m, m2), moe::pack_f32x2(r, r),
                                                   moe::pack_f32x2(-s, -s)), p0, p1);
        if (__float_as_uint(p0) != __float_as_uint(qm_fast) ||
            __float_as_uint(p1) != __float_as_uint(moe::div_mag_by_scale(m2, s, r)))
            atomicAdd(&counters[7], 1ull);
    }
    const unsigned warp_n = __reduce_add_sync(0xffffffffu, local_n);
    if ((threadIdx.x & 31) == 0) atomicAdd(&counters[2], static_cast<unsigned long long>(warp_n));
}

}  // namespace

// counters: [quotient mismatches, code mismatches, pairs checked, scale mismatches,
//            reciprocal mismatches, magnitude-quotient mismatches, sign-OR code mismatches,
//            packed-quotient mismatches];
// examples: 2 * max_examples records of 4 words.
extern "C" int fp8_div_check(const uint16_t* amax_bits, int n_amax, unsigned long long* counters,
                             uint32_t* examples, int max_examples) {
    if (n_amax <= 0 || n_amax > 65535) return 1;
    dim3 grid(64, static_cast<unsigned>(n_amax));
    div_check_kernel<<<grid, 256>>>(amax_bits, n_amax, counters, examples, max_examples);
    if (cudaGetLastError() != cudaSuccess) return 2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
