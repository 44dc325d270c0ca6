// Device helpers for the fp8 KV publication kernels (sm_103a).
//
// One warp owns one token row.  Lane l holds:
//   latent elements [16 l, 16 l + 16)  -> 2 x 16-byte loads, tile = lanes 8j..8j+7
//   Indexer-K elements [4 l, 4 l + 4)  -> 1 x 8-byte load, the tile is the warp
//   rope chunk l-1 (8 values) for lanes 1..8 -> 1 x 16-byte load
// so every amax is a 3-step (latent) or 5-step (Indexer-K) xor-shuffle
// reduction, and every lane quantises 20 values.
//
// Quantisation rule (the cache format's reading): per 128-element tile
// amax = max |x|, scale = max(amax, 1e-4f) / 448 (correctly rounded fp32),
// code = E4M3(x / scale) with round-to-nearest-even and saturation; a NaN in
// the tile gives the scale 0x7FFFFFFF and codes 0x7F.
//
// The quotient x / scale must be the correctly rounded fp32 quotient.  It is
// computed with Markstein's correction (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with y = RN(1/scale) per tile, q0 = RN(x * y),
// r = x - scale * q0 (exact in one fma) and q = RN(q0 + r * y) (one fma).
// Per element that is one multiply and two fmas, issued two elements at a
// time as packed f32x2 operations, then the input's sign bit is ORed into
// each code (see quant4_markstein).  A tile whose scale is not finite (an
// Inf or NaN in the tile) takes IEEE division.
//
// The per-tile scale and reciprocal are themselves exact without an IEEE
// division: the scale by the same correction with the constant RN(1/448)
// (tile_scale), the reciprocal by one Newton-Raphson step from the hardware
// approximation (tile_divisor).  Both are correctly rounded on every input
// the kernel can meet: a tile maximum is one of 32,768 bf16 magnitudes, so
// GPU tests compare them, and the codes of every (x, amax) pair, with
// CUDA's __fdiv_rn and __frcp_rn.
#pragma once

#include <cuda_fp8.h>
#include <stdint.h>

namespace kvpub {

constexpr unsigned kFullMask = 0xffffffffu;

// |bf16| bit patterns order like their magnitudes (NaN patterns above
// +Inf), so the tile amax is an unsigned 16-bit max over x & 0x7fff.
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t a, uint32_t b) {
    return __vmaxu2(a & 0x7fff7fffu, b & 0x7fff7fffu);
}

__device__ __forceinline__ uint32_t halves_max(uint32_t v) {
    return max(v & 0xffffu, v >> 16);
}

// RN(max(amax, 1e-4f) / 448) in fp32.  For a finite maximum, m is 1e-4f
// or a bf16 magnitude above it, and Markstein's correction with the
// constant c = RN(1/448) gives the correctly rounded quotient for every one
// of those 18,095 values: q0 = RN(m c), r = m - 448 q0 (exact), RN(q0 + r c).
// An Inf maximum gives Inf (as IEEE division would), a NaN maximum the
// canonical quiet NaN.
__device__ __forceinline__ float tile_scale(uint32_t amax_bits16) {
    if (amax_bits16 >= 0x7f80u)
        return __uint_as_float(amax_bits16 == 0x7f80u ? 0x7f800000u : 0x7fffffffu);
    const float amax = __uint_as_float(amax_bits16 << 16);
    const float m = (amax < 1e-4f) ? 1e-4f : amax;
    constexpr float c = 1.0f / 448.0f;
    const float q0 = __fmul_rn(m, c);
    const float r = __fmaf_rn(-448.0f, q0, m);
    return __fmaf_rn(r, c, q0);
}

// Everything a lane needs to divide by one tile's scale.
struct TileDivisor {
    float scale;
    unsigned long long y2;        // {RN(1/scale), RN(1/scale)}
    unsigned long long neg_s2;    // {-scale, -scale}
    bool ieee;                    // scale is Inf or NaN: use IEEE division
};

// RN(1/scale) for the finite scales tile_scale returns (2.2e-7 .. 7.6e35,
// all normal, as are their reciprocals): the hardware's approximate
// reciprocal y0, then one Newton-Raphson step in fma form,
// y = y0 + y0 (1 - scale y0).  Non-finite scales take IEEE division and do
// not use y.
__device__ __forceinline__ TileDivisor tile_divisor(float scale) {
    TileDivisor d;
    d.scale = scale;
    d.ieee = !(fabsf(scale) <= 3.402823466e38f);
    float y0;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y0) : "f"(scale));
    const float y = __fmaf_rn(__fmaf_rn(-scale, y0, 1.0f), y0, y0);
    asm("mov.b64 %0, {%1, %1};" : "=l"(d.y2) : "f"(y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(d.neg_s2) : "f"(-scale));
    return d;
}

// Two bf16 words (4 values) -> 4 E4M3 codes, low byte = first value, using
// Markstein's correction on packed f32x2.  For x = -0 the residual
// fma(-scale, q0, x) is (+0) + (-0) = +0 and the corrected quotient comes
// out +0, so the sign of each input is ORed into its code afterwards: for
// every finite x the correctly rounded quotient carries the sign of x, and
// for x != -0 the code already has it.
__device__ __forceinline__ uint32_t quant4_markstein(uint32_t w0, uint32_t w1,
                                                     unsigned long long y2,
                                                     unsigned long long neg_s2) {
    uint32_t out;
    asm("{\n\t"
        ".reg .b32 l0, h0, l1, h1;\n\t"
        ".reg .b64 x0, x1, a0, a1, r0, r1;\n\t"
        ".reg .f32 p0, p1, p2, p3;\n\t"
        ".reg .b16 c0, c1;\n\t"
        ".reg .b32 codes, signs;\n\t"
        "shl.b32 l0, %1, 16;\n\t"
        "and.b32 h0, %1, 0xffff0000;\n\t"
        "shl.b32 l1, %2, 16;\n\t"
        "and.b32 h1, %2, 0xffff0000;\n\t"
        "mov.b64 x0, {l0, h0};\n\t"
        "mov.b64 x1, {l1, h1};\n\t"
        "mul.rn.f32x2 a0, x0, %3;\n\t"
        "mul.rn.f32x2 a1, x1, %3;\n\t"
        "fma.rn.f32x2 r0, %4, a0, x0;\n\t"
        "fma.rn.f32x2 r1, %4, a1, x1;\n\t"
        "fma.rn.f32x2 a0, r0, %3, a0;\n\t"
        "fma.rn.f32x2 a1, r1, %3, a1;\n\t"
        "mov.b64 {p0, p1}, a0;\n\t"
        "mov.b64 {p2, p3}, a1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 c0, p1, p0;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 c1, p3, p2;\n\t"
        "mov.b32 codes, {c0, c1};\n\t"
        // sign bits of the four inputs (bits 15 and 31 of each word) into
        // bit 7 of their codes
        "prmt.b32 signs, %1, %2, 0x7531;\n\t"
        "lop3.b32 %0, codes, signs, 0x80808080, 0xF8;\n\t"
        "}"
        : "=r"(out)
        : "r"(w0), "r"(w1), "l"(y2), "l"(neg_s2));
    return out;
}

// The same four codes through IEEE division (non-finite scales only).
__device__ __forceinline__ uint32_t quant4_ieee(uint32_t w0, uint32_t w1, float scale) {
    const float2 a = make_float2(__fdiv_rn(__uint_as_float(w0 << 16), scale),
                                 __fdiv_rn(__uint_as_float(w0 & 0xffff0000u), scale));
    const float2 b = make_float2(__fdiv_rn(__uint_as_float(w1 << 16), scale),
                                 __fdiv_rn(__uint_as_float(w1 & 0xffff0000u), scale));
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(a, __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(b, __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t quant4(uint32_t w0, uint32_t w1, const TileDivisor &d) {
    if (d.ieee) return quant4_ieee(w0, w1, d.scale);
    return quant4_markstein(w0, w1, d.y2, d.neg_s2);
}

}  // namespace kvpub
