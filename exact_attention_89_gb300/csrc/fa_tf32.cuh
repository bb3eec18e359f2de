// fa_tf32.cuh -- pieces shared by the fp32 passes on the tensor cores (three TF32 products).
//
// An fp32 value x is split as x = hi + lo: hi keeps the sign, the exponent and the top 10
// mantissa bits (exactly a TF32 value) and lo = x - hi is exact in fp32.  A product A B is then
// formed as hi(A) hi(B) + hi(A) lo(B) + lo(A) hi(B) in an fp32 accumulator (tcgen05 kind::tf32);
// the dropped lo(A) lo(B) and the TF32 rounding of lo leave a relative error near 2^-21 per
// product.  Operands are K-major only.
#pragma once

#include <cstdint>

namespace fa {

constexpr uint32_t TF32_HI_MASK = 0xFFFFE000u;

__device__ __forceinline__ float tf32_hi(float x) {
    return __uint_as_float(__float_as_uint(x) & TF32_HI_MASK);
}

// Instruction descriptor, kind::tf32: TF32 A and B (format 2), fp32 D, both K-major, dense.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((static_cast<uint32_t>(N) >> 3) << 17) |
           ((static_cast<uint32_t>(M) >> 4) << 24);
}

// D(tmem) (+)= A(smem desc) * B(smem desc), TF32.
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem) (+)= A(tmem) * B(smem desc), TF32: row m of A is TMEM lane m, one element per column.
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

}  // namespace fa
