// MXFP8 (OCP Microscaling formats, MXFP8 with E4M3 elements) to bf16, on
// the device. An E4M3 code is a sign, a 4-bit exponent with bias 7 and a
// 3-bit mantissa (exponent 0: subnormals m * 2^-9); a UE8M0 scale code s
// stands for 2^(s - 127). Every product of the two has at most 4 significant
// bits, so it is exactly a bf16 number whenever it lies in bf16's range
// (scale codes 3..246 for every E4M3 value); the conversion below is exact
// there. NaN codes (S.1111.111) and the NaN scale (255) give unspecified
// values.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace moe {

// Two E4M3 codes given as the 16-bit halves 0x00bb of a word -> a bf16 pair
// whose values are the codes' values times 2^-120: the sign moves to bit 15
// and the 7 exponent/mantissa bits to bits 4..10, so the E4M3 exponent field
// becomes the bf16 exponent field (bias 127 instead of 7) and an E4M3
// subnormal becomes the bf16 subnormal with the same mantissa bits.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2_scaled_down(uint32_t m16) {
    return (m16 << 4) + (m16 & 0x00800080u) * 0xF0u;
}

// 16 E4M3 codes (bytes of v, lowest first) with scale code s -> 8 bf16 pairs
// (out[i] holds values 2i and 2i + 1, the lower index in the low half).
// The factor 2^120 * 2^(s - 127) = 2^(s - 7) is one bf16 multiplier when it
// is a normal bf16 number (s <= 134), else the two exact multipliers 2^120
// and 2^(s - 127). Every product is exact (a power of two times a value that
// bf16 holds, with an exact result whenever that lies in bf16's range).
__device__ __forceinline__ void mx_dequant16(const uint4& v, uint32_t s, uint32_t (&out)[8]) {
    const bool one = s <= 134u;
    const uint32_t c1 = ((one ? s + 120u : 247u) << 7) * 0x10001u;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = ptx::mul_bf16x2(e4m3x2_to_bf16x2_scaled_down(__byte_perm(w[i], 0u, 0x4140)), c1);
        out[2 * i + 1] =
            ptx::mul_bf16x2(e4m3x2_to_bf16x2_scaled_down(__byte_perm(w[i], 0u, 0x4342)), c1);
    }
    if (!one) {
        const uint32_t c2 = (s << 7) * 0x10001u;
#pragma unroll
        for (int i = 0; i < 8; ++i) out[i] = ptx::mul_bf16x2(out[i], c2);
    }
}

}  // namespace moe
