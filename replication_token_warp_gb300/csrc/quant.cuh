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
// amax = max |x|, scale = max(amax, 1e-4f) / 448 (one IEEE fp32 division),
// code = E4M3(x / scale) with round-to-nearest-even and saturation; a NaN in
// the tile gives the scale 0x7FFFFFFF and codes 0x7F.
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

// max(amax, 1e-4f) / 448 in fp32.  The comparison is false for NaN, so a
// NaN amax passes through and becomes the canonical quiet NaN.
__device__ __forceinline__ float tile_scale(uint32_t amax_bits16) {
    const float amax = __uint_as_float(amax_bits16 << 16);
    const float m = (amax < 1e-4f) ? 1e-4f : amax;
    float s = __fdiv_rn(m, 448.0f);
    if (s != s) s = __uint_as_float(0x7fffffffu);
    return s;
}

// Two bf16 (one 32-bit word) -> two E4M3 codes (low byte = low element).
__device__ __forceinline__ uint32_t quant_bf16x2(uint32_t w, float scale) {
    const float lo = __uint_as_float(w << 16);
    const float hi = __uint_as_float(w & 0xffff0000u);
    const float2 q = make_float2(__fdiv_rn(lo, scale), __fdiv_rn(hi, scale));
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3));
}

// Four bf16 words (8 values) -> 8 codes packed in two 32-bit words.
__device__ __forceinline__ uint2 quant_bf16x8(uint4 v, float scale) {
    uint2 out;
    out.x = quant_bf16x2(v.x, scale) | (quant_bf16x2(v.y, scale) << 16);
    out.y = quant_bf16x2(v.z, scale) | (quant_bf16x2(v.w, scale) << 16);
    return out;
}

}  // namespace kvpub
