// Test-only kernel: compares the dispatch kernel's quotient
// (moe::scaled_quotient with r = __frcp_rn(s)) against CUDA's IEEE division
// __fdiv_rn(x, s) for every bf16 value x with |x| <= amax, over a list of
// block maxima amax (s = __fdiv_rn(amax, 448)).  Counts bitwise mismatches
// and records the first few.  Every index is bounded by the array sizes.
#include <cstdint>

#include "fp8_quant.cuh"

namespace {

__global__ void div_check_kernel(const uint16_t* amax_bits, int n_amax, unsigned long long* mismatches,
                                 uint32_t* examples, int max_examples, unsigned long long* checked) {
    const int a_idx = blockIdx.y;
    if (a_idx >= n_amax) return;
    const float amax = __uint_as_float(static_cast<uint32_t>(amax_bits[a_idx]) << 16);
    const float s = __fdiv_rn(amax, 448.0f);
    if (!moe::scale_is_normal(s)) return;
    const float r = __frcp_rn(s);
    unsigned long long local_bad = 0, local_n = 0;
    for (uint32_t xb = blockIdx.x * blockDim.x + threadIdx.x; xb < 65536u; xb += gridDim.x * blockDim.x) {
        const float x = __uint_as_float(xb << 16);
        if (!(fabsf(x) <= amax)) continue;            // skips NaN and values beyond the block max
        ++local_n;
        const float q_fast = moe::scaled_quotient(x, s, r, true);
        const float q_ieee = __fdiv_rn(x, s);
        if (__float_as_uint(q_fast) != __float_as_uint(q_ieee)) {
            ++local_bad;
            const unsigned long long slot = atomicAdd(mismatches, 1ull);
            if (slot < static_cast<unsigned long long>(max_examples)) {
                examples[4 * slot + 0] = amax_bits[a_idx];
                examples[4 * slot + 1] = xb;
                examples[4 * slot + 2] = __float_as_uint(q_fast);
                examples[4 * slot + 3] = __float_as_uint(q_ieee);
            }
        }
    }
    (void)local_bad;
    const unsigned warp_n = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(local_n));
    if ((threadIdx.x & 31) == 0) atomicAdd(checked, static_cast<unsigned long long>(warp_n));
}

}  // namespace

extern "C" int fp8_div_check(const uint16_t* amax_bits, int n_amax, unsigned long long* mismatches,
                             uint32_t* examples, int max_examples, unsigned long long* checked) {
    if (n_amax <= 0 || n_amax > 65535) return 1;
    dim3 grid(64, static_cast<unsigned>(n_amax));
    div_check_kernel<<<grid, 256>>>(amax_bits, n_amax, mismatches, examples, max_examples, checked);
    if (cudaGetLastError() != cudaSuccess) return 2;
    return cudaDeviceSynchronize() == cudaSuccess ? 0 : 3;
}
