// Exhaustive check of the store kernel's quotient against IEEE division.
//
// For every finite tile maximum M (as a bf16 bit pattern) and every bf16 x
// with |x| <= M, quant4() from the library's quant.cuh (Markstein's
// correction on packed f32x2, IEEE division for non-finite scales) must
// give the same E4M3 codes as CUDA's correctly rounded __fdiv_rn followed
// by the saturating conversion.  Those are all the (value, scale) pairs the
// store kernel can meet, since a tile's scale comes from its own maximum.
// A second sweep checks the per-tile scale and reciprocal that quant4()
// receives: tile_scale() against __fdiv_rn(max(amax, 1e-4f), 448) and
// tile_divisor()'s reciprocal against __frcp_rn, over all 32,768 tile
// maxima (every non-negative bf16 pattern, Inf and NaN included).
// Test infrastructure: built and run by tests/test_gpu_division.py.
#include <cuda_runtime.h>

#include "quant.cuh"

using namespace kvpub;

__device__ unsigned long long g_mismatch;
__device__ unsigned long long g_checked;
__device__ unsigned int g_examples[16];   // [0] = count, then (M, x) pairs

__global__ void sweep_kernel(unsigned int m_begin, unsigned int m_end) {
    for (unsigned int mb = m_begin + blockIdx.x; mb < m_end; mb += gridDim.x) {
        const float scale = tile_scale(mb);
        const TileDivisor d = tile_divisor(scale);
        unsigned long long mism = 0, checked = 0;
        for (unsigned int xb = 2 * threadIdx.x; xb <= mb; xb += 2 * blockDim.x) {
            const unsigned int x1 = (xb + 1 <= mb) ? xb + 1 : xb;
            const uint32_t w0 = xb | (x1 << 16);                               // +x
            const uint32_t w1 = (xb | 0x8000u) | ((x1 | 0x8000u) << 16);       // -x
            const uint32_t fast = quant4(w0, w1, d);
            const uint32_t ref = quant4_ieee(w0, w1, scale);
            checked += 4;
            if (fast != ref) {
                ++mism;
                const unsigned int k = atomicAdd(&g_examples[0], 1u);
                if (k < 7) {
                    g_examples[1 + 2 * k] = mb;
                    g_examples[2 + 2 * k] = xb;
                }
            }
        }
        atomicAdd(&g_mismatch, mism);
        atomicAdd(&g_checked, checked);
    }
}

// out[0] = mismatching words, out[1] = values checked, out[2..16] = examples.
extern "C" int kvpub_test_division_sweep(unsigned long long *out) {
    const unsigned long long zero = 0;
    unsigned int zeros[16] = {0};
    cudaError_t e;
    if ((e = cudaMemcpyToSymbol(g_mismatch, &zero, sizeof zero)) != cudaSuccess) return (int)e;
    if ((e = cudaMemcpyToSymbol(g_checked, &zero, sizeof zero)) != cudaSuccess) return (int)e;
    if ((e = cudaMemcpyToSymbol(g_examples, zeros, sizeof zeros)) != cudaSuccess) return (int)e;
    sweep_kernel<<<4096, 256>>>(0u, 0x7F80u);   // every finite non-negative bf16 maximum
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return (int)e;
    unsigned int ex[16];
    if ((e = cudaMemcpyFromSymbol(&out[0], g_mismatch, 8)) != cudaSuccess) return (int)e;
    if ((e = cudaMemcpyFromSymbol(&out[1], g_checked, 8)) != cudaSuccess) return (int)e;
    if ((e = cudaMemcpyFromSymbol(ex, g_examples, sizeof ex)) != cudaSuccess) return (int)e;
    for (int i = 0; i < 15; ++i) out[2 + i] = ex[i];
    return 0;
}

__device__ unsigned int g_scale_bad[2];       // scale, reciprocal mismatches
__device__ unsigned int g_scale_examples[8];  // first maxima that differ

__device__ float ieee_tile_scale(uint32_t amax_bits16) {
    const float amax = __uint_as_float(amax_bits16 << 16);
    const float m = (amax < 1e-4f) ? 1e-4f : amax;
    const float s = __fdiv_rn(m, 448.0f);
    return (s != s) ? __uint_as_float(0x7fffffffu) : s;
}

__global__ void scale_sweep_kernel() {
    const uint32_t a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a > 0x7fffu) return;
    const float ref = ieee_tile_scale(a);
    if (__float_as_uint(tile_scale(a)) != __float_as_uint(ref)) {
        const unsigned int k = atomicAdd(&g_scale_bad[0], 1u);
        if (k < 4) g_scale_examples[k] = a;
    }
    if (!(fabsf(ref) <= 3.402823466e38f)) return;     // IEEE path, no reciprocal
    const TileDivisor d = tile_divisor(ref);
    const uint32_t y = static_cast<uint32_t>(d.y2 & 0xffffffffull);
    if (y != __float_as_uint(__frcp_rn(ref))) {
        const unsigned int k = atomicAdd(&g_scale_bad[1], 1u);
        if (k < 4) g_scale_examples[4 + k] = a;
    }
}

// out[0] = scale mismatches, out[1] = reciprocal mismatches,
// out[2..5] / out[6..9] = the first maxima of each.
extern "C" int kvpub_test_scale_sweep(unsigned long long *out) {
    unsigned int zeros[8] = {0};
    cudaError_t e;
    if ((e = cudaMemcpyToSymbol(g_scale_bad, zeros, 2 * sizeof(unsigned int))) != cudaSuccess)
        return (int)e;
    if ((e = cudaMemcpyToSymbol(g_scale_examples, zeros, sizeof zeros)) != cudaSuccess)
        return (int)e;
    scale_sweep_kernel<<<128, 256>>>();   // 32,768 threads, one per maximum
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
    if ((e = cudaDeviceSynchronize()) != cudaSuccess) return (int)e;
    unsigned int bad[2], ex[8];
    if ((e = cudaMemcpyFromSymbol(bad, g_scale_bad, sizeof bad)) != cudaSuccess) return (int)e;
    if ((e = cudaMemcpyFromSymbol(ex, g_scale_examples, sizeof ex)) != cudaSuccess) return (int)e;
    out[0] = bad[0];
    out[1] = bad[1];
    for (int i = 0; i < 8; ++i) out[2 + i] = ex[i];
    return 0;
}
