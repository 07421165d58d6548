// MXFP8 (E4M3 elements, E8M0 block scales) encoding on fp32 registers.
//
// Scale rule: the exponent of a 32-element block is the smallest integer e
// with amax <= 448 * 2^e, clamped to [-127, 127], stored as the byte e + 127;
// elements are v * 2^-e rounded to nearest-even E4M3 with saturation (the
// hardware cvt.rn.satfinite). A block holding NaN or Inf gets scale 0xFF and
// NaN codes (0x7F with each element's sign).
#pragma once
#include <cstdint>

namespace mlaq {

// Exponent from the bits of a non-negative finite fp32 amax:
// amax = 1.m * 2^E with 448 = 1.75 * 2^8, so amax <= 448 * 2^(E-8) exactly
// when the 23-bit mantissa field is <= 0x600000 (1.75), else one more.
// Zero and fp32 subnormals (< 2^-126 < 448 * 2^-127) clamp to -127.
__device__ __forceinline__ int e8m0_exponent_f32(float amax) {
    const uint32_t bits = __float_as_uint(amax);
    const int be = (int)((bits >> 23) & 0xFFu);
    if (be == 0) return -127;
    int e = (be - 127) - 8 + ((bits & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    e = e < -127 ? -127 : e;
    e = e > 127 ? 127 : e;
    return e;
}

// 2^-e as an fp32 (e in [-127, 120] for finite fp32 amax: always a normal).
__device__ __forceinline__ float exp2_neg(int e) {
    return __uint_as_float((uint32_t)(127 - e) << 23);
}

// Two fp32 -> two E4M3 bytes (lo in bits 0..7, hi in bits 8..15), RNE, saturating.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    return cvt_e4m3x2(a, b) | (cvt_e4m3x2(c, d) << 16);
}

// NaN code keeping the element's sign.
__device__ __forceinline__ uint32_t nan_code(float v) {
    return 0x7Fu | ((__float_as_uint(v) >> 24) & 0x80u);
}

// Round two fp32 to bf16 (RNE) and pack (lo in bits 0..15).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t packed) { return __uint_as_float(packed << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t packed) {
    return __uint_as_float(packed & 0xFFFF0000u);
}

// max(m, |v|) that returns NaN when either input is NaN (so a block amax taken
// with it is NaN or Inf exactly when the block holds a non-finite element;
// for finite inputs it equals the largest magnitude).
__device__ __forceinline__ float amax_nan(float m, float v) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(m), "f"(fabsf(v)));
    return r;
}

// max.NaN of two magnitudes (both already non-negative or NaN).
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// The NaN-propagating amax of v[0..n) (n a compile-time bound after
// unrolling) as a tree: eight independent running maxima, then three
// levels. max is exact and NaN-propagating in any order, so the result is
// the serial chain's, with a quarter of its dependent latency.
template <int NV>
__device__ __forceinline__ float amax_tree(const float (&v)[NV], int n) {
    float m[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
        if (i < n) m[i % 8] = amax_nan(m[i % 8], v[i]);
#pragma unroll
    for (int w = 4; w >= 1; w /= 2)
#pragma unroll
        for (int j = 0; j < w; ++j) m[j] = max_nan(m[j], m[j + w]);
    return m[0];
}

// Quantize n <= 32 fp32 values held by ONE thread (a whole block) into codes
// (packed little-endian, 4 per word) and return the scale byte. Entries past
// n are ignored for the amax and encoded anyway (callers do not store them).
// The amax is a NaN-propagating float max of the magnitudes: its bits are
// >= 0x7F800000 exactly when the block holds an Inf or a NaN.
template <int NV>
__device__ __forceinline__ uint32_t quantize_block_regs(const float (&v)[NV], int n,
                                                        uint32_t (&codes)[(NV + 3) / 4]) {
    const float am = amax_tree<NV>(v, n);
    const uint32_t mbits = __float_as_uint(am);
    if (mbits >= 0x7F800000u) {
#pragma unroll
        for (int w = 0; w < (NV + 3) / 4; ++w) {
            uint32_t c = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (4 * w + j < NV) c |= nan_code(v[4 * w + j]) << (8 * j);
            codes[w] = c;
        }
        return 0xFFu;
    }
    const int e = e8m0_exponent_f32(__uint_as_float(mbits));
    const float s = exp2_neg(e);
#pragma unroll
    for (int w = 0; w < (NV + 3) / 4; ++w) {
        float a = v[4 * w] * s;
        float b = (4 * w + 1 < NV) ? v[4 * w + 1] * s : 0.f;
        float c = (4 * w + 2 < NV) ? v[4 * w + 2] * s : 0.f;
        float d = (4 * w + 3 < NV) ? v[4 * w + 3] * s : 0.f;
        codes[w] = pack_e4m3x4(a, b, c, d);
    }
    return (uint32_t)(e + 127);
}

// A whole 32-element block held by one thread: the rule of
// quantize_block_regs, with the amax by amax_nan.
__device__ __forceinline__ uint32_t quantize_block32(const float (&v)[32], uint32_t (&codes)[8]) {
    const float am = amax_tree<32>(v, 32);
    const uint32_t mbits = __float_as_uint(am);
    if (mbits >= 0x7F800000u) {
#pragma unroll
        for (int w = 0; w < 8; ++w)
            codes[w] = nan_code(v[4 * w]) | (nan_code(v[4 * w + 1]) << 8) | (nan_code(v[4 * w + 2]) << 16) |
                       (nan_code(v[4 * w + 3]) << 24);
        return 0xFFu;
    }
    const int e = e8m0_exponent_f32(am);
    const float s = exp2_neg(e);
#pragma unroll
    for (int w = 0; w < 8; ++w)
        codes[w] = pack_e4m3x4(v[4 * w] * s, v[4 * w + 1] * s, v[4 * w + 2] * s, v[4 * w + 3] * s);
    return (uint32_t)(e + 127);
}

// Quantize 8 values of a 32-element block whose other 24 elements are held by
// three other lanes; mbits is the block's amax magnitude bits already reduced
// over all 32 (the same rule as quantize_block_regs). Returns the scale byte.
__device__ __forceinline__ uint32_t quantize8_block_scale(const float (&v)[8], uint32_t mbits,
                                                          uint32_t (&codes)[2]) {
    if (mbits >= 0x7F800000u) {
#pragma unroll
        for (int w = 0; w < 2; ++w)
            codes[w] = nan_code(v[4 * w]) | (nan_code(v[4 * w + 1]) << 8) | (nan_code(v[4 * w + 2]) << 16) |
                       (nan_code(v[4 * w + 3]) << 24);
        return 0xFFu;
    }
    const int e = e8m0_exponent_f32(__uint_as_float(mbits));
    const float s = exp2_neg(e);
#pragma unroll
    for (int w = 0; w < 2; ++w)
        codes[w] = pack_e4m3x4(v[4 * w] * s, v[4 * w + 1] * s, v[4 * w + 2] * s, v[4 * w + 3] * s);
    return (uint32_t)(e + 127);
}

// E8M0 scales in the order the block-scaled GEMM loads them: rows of one
// operand (its M or N axis) in groups of G rows (the GEMM's tile height along
// that axis); a group is padded to whole 128-row chunks and each chunk stored
// as tiles of 128 rows x 4 scale columns (one 128-element K step), 512 bytes,
// in the layout tcgen05.cp replicates into TMEM: row rr of the chunk, column
// c at (rr % 32) * 16 + (rr / 32) * 4 + (c % 4). Chunk i of group g, K step
// kt is tile ((g * ceil(G/128) + i) * nkt + kt), nkt = ceil(cols / 4). With
// G = 128 this is the GEMM scale swizzle of the whole [rows, cols] matrix.
__host__ __device__ __forceinline__ int64_t sf_tiled_offset(int64_t r, int64_t c, int64_t G, int64_t nkt) {
    const int64_t nsub = (G + 127) / 128;
    const int64_t g = r / G, rg = r - g * G;
    const int64_t i = rg / 128, rr = rg - i * 128;
    return ((g * nsub + i) * nkt + c / 4) * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4);
}
__host__ __device__ __forceinline__ int64_t sf_tiled_bytes(int64_t rows, int64_t cols, int64_t G) {
    return (rows + G - 1) / G * ((G + 127) / 128) * ((cols + 3) / 4) * 512;
}

}  // namespace mlaq
