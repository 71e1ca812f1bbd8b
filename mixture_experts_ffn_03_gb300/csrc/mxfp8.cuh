// MXFP8 (OCP Microscaling formats, MXFP8 with E4M3 elements) and NVFP4 (FP4
// E2M1 elements, E4M3 block scales) to bf16, on the device. An E4M3 code is a sign, a 4-bit exponent with bias 7 and a
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

// One byte permute in the generic mode of prmt, where bit 3 of a selector
// nibble replicates bit 7 of the selected byte (a sign) instead of copying it.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// bf16 pair (v, v) of the E4M3 value of `code`: the bit pattern of
// e4m3x2_to_bf16x2_scaled_down is the value x 2^-120, and one exact multiply
// by 2^120 restores it (every E4M3 value is a normal bf16 number).
__device__ __forceinline__ uint32_t e4m3_to_bf16x2(uint32_t code) {
    return ptx::mul_bf16x2(e4m3x2_to_bf16x2_scaled_down(code * 0x10001u), (247u << 7) * 0x10001u);
}

// 32 E2M1 codes (the nibbles of v, lowest first: value 2j in the low nibble of
// byte j) -> 16 bf16 pairs, values 0-15 scaled by the bf16 pair c0 and values
// 16-31 by c1 (the block scales). The magnitude's two bf16 bytes come from two
// 8-entry byte tables (0, 0.5, 1, 1.5, 2, 3, 4, 6); prmt's sign-replicate mode
// moves each nibble's sign bit to bit 7 of its high byte. An E2M1 value times
// an E4M3 scale has at most 6 significant bits and lies in [2^-10, 2688], so
// the multiply is exact.
__device__ __forceinline__ void nv_dequant32(const uint4& v, uint32_t c0, uint32_t c1,
                                             uint32_t (&out)[16]) {
    constexpr uint32_t kHi0 = 0x3F3F3F00u, kHi1 = 0x40404040u;  // high bytes, magnitudes 0-3, 4-7
    constexpr uint32_t kLo0 = 0xC0800000u, kLo1 = 0xC0804000u;  // low bytes
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t wi = w[i], w4 = wi << 4;
        const uint32_t c = i < 2 ? c0 : c1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // values 8i + 4h .. 8i + 4h + 3
            const uint32_t sel = (h ? wi >> 16 : wi) & 0x7777u;
            const uint32_t lo = prmt(kLo0, kLo1, sel);
            // value j's sign (bit 3 of its nibble) sits at bit 7 of a byte of w4
            // (even j) or of w (odd j): replicate it into byte j, keep bit 7
            const uint32_t sgn = prmt(w4, wi, h ? 0xFBEAu : 0xD9C8u);
            const uint32_t hi = prmt(kHi0, kHi1, sel) | (sgn & 0x80808080u);
            out[4 * i + 2 * h] = ptx::mul_bf16x2(prmt(lo, hi, 0x5140u), c);
            out[4 * i + 2 * h + 1] = ptx::mul_bf16x2(prmt(lo, hi, 0x7362u), c);
        }
    }
}

}  // namespace moe
