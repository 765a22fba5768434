// pair_rows.cuh -- the storage format of the per-pair weighted expert
// outputs w * Expert(x) between the down GEMM and the combine: a bf16 value
// hi = bf16(v) plus an int8 residual r, three bytes a value instead of four.
//
// Why: the layer's output tolerance leaves little room above the bf16
// rounding of the exact result, so the k contributions of a token must reach
// the combine with well over bf16's 8 significant bits (an fp16 rounding of
// each, 11 bits, was already too coarse at prefill size); but at prefill size
// the pair outputs are the largest intermediate in memory (N*k rows of H),
// written once and read once.  hi + residual keeps 16 significant bits in
// three bytes: with e the binary exponent of hi, hi's spacing is 2^(e-7), so
// |v - hi| <= 2^(e-8), and r = round((v - hi) * 2^(15-e)) in [-127, 127]
// resolves it in steps of 2^(e-15); the decoded hi + r * 2^(e-15) is within
// 2^(e-16) <= 2^-16 |v| of v.  The scale is a power of two taken from hi's
// own exponent field, so encoding and decoding need no extra storage and
// are exact apart from the one rounding of r.  Exponents are clamped below
// at 2^-111 (values that small are decoded to within 2^-127 absolute).
//
// Layout: two planes, hi [rows, H] (bf16) and r [rows, H] (int8), rows in
// pair order.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace moe {

// 2^(15 - e') and 2^(e' - 15) as float bit patterns, e' the biased exponent
// field of hi clamped to >= 16 (both stay normal floats for every e').
__device__ __forceinline__ int pair_exp_field(float hi) {
    const int f = static_cast<int>((__float_as_uint(hi) >> 23) & 0xFF);
    return f < 16 ? 16 : f;
}

// The residual of v against hi = bf16(v) (hi given widened to fp32).
__device__ __forceinline__ int pair_residual(float v, float hi) {
    const int f = pair_exp_field(hi);
    const float up = __uint_as_float(static_cast<uint32_t>(269 - f) << 23);  // 2^(142 - f)
    float r = rintf((v - hi) * up);
    r = fminf(fmaxf(r, -127.f), 127.f);
    return static_cast<int>(r);
}

// Four residuals (of v[i] against hi[i]) packed as bytes 0..3 of a word,
// with the arithmetic kept off the conversion pipe: (v - hi) * 2^(142 - f)
// is exact (a difference of v and its own rounding, times a power of two)
// and lies within [-128, 128], so one fused add of 1.5 * 2^23 rounds it to
// the nearest integer, ties to even, exactly as rint does, and leaves that
// integer in the low mantissa bits (1.5 * 2^23 has a zero low byte); the
// clamp to [-127, 127] is taken on the sum, and the low bytes are gathered
// with byte permutes.  Equal, byte for byte, to pair_residual.
__device__ __forceinline__ uint32_t pair_residual_sum_bits(float v, float hi) {
    constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
    // 2^(142 - f) built from hi's exponent bits in place: (269 << 23) minus
    // max(exponent bits, 16 << 23), the same value as pair_residual's
    const uint32_t e_bits = max(__float_as_uint(hi) & 0x7F800000u, 16u << 23);
    const float up = __uint_as_float((269u << 23) - e_bits);
    float t = fmaf(v - hi, up, kMagic);
    t = fminf(fmaxf(t, kMagic - 127.f), kMagic + 127.f);
    return __float_as_uint(t);
}

__device__ __forceinline__ uint32_t pair_residual4(float v0, float h0, float v1, float h1,
                                                   float v2, float h2, float v3, float h3) {
    const uint32_t a = __byte_perm(pair_residual_sum_bits(v0, h0), pair_residual_sum_bits(v1, h1),
                                   0x0040);
    const uint32_t b = __byte_perm(pair_residual_sum_bits(v2, h2), pair_residual_sum_bits(v3, h3),
                                   0x0040);
    return __byte_perm(a, b, 0x5410);
}

// hi + r * 2^(f - 142): the decoded value.
__device__ __forceinline__ float pair_decode(float hi, int r) {
    const int f = pair_exp_field(hi);
    const float down = __uint_as_float(static_cast<uint32_t>(f - 15) << 23);  // 2^(f - 142)
    return fmaf(static_cast<float>(r), down, hi);
}

}  // namespace moe
