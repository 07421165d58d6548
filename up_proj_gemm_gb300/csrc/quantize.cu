// Standalone rowwise MXFP8 quantizer (HBM-bound streaming kernel).
//
// TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant":
// the separable ("two-phase") MXFP8 quantization helper, mxfp8_quantize_only
// in its review thread. One pass: each 32-element block's amax -> E8M0 scale
// -> E4M3 codes, no intermediate written to memory.
//
// Work split: a warp-iteration covers 32 lanes x 16 bytes of input per
// unrolled step (256 bf16 or 128 fp32 elements, i.e. 8 or 4 whole blocks);
// the lanes of one block (4 for bf16, 8 for fp32) combine their amax with
// shuffles. Each thread keeps UNROLL 16-byte loads in flight. The grid is
// persistent (a multiple of the SM count) and strides over (row, segment)
// tasks. Rows that are contiguous with C % 32 == 0 are folded into one long
// row, which leaves codes and scales in the same places.
#include <cuda_bf16.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kUnroll = 4;
constexpr int kThreads = 256;

template <typename Tin>
struct VecTraits;
template <>
struct VecTraits<float> {
    static constexpr int kElems = 4;
};
template <>
struct VecTraits<__nv_bfloat16> {
    static constexpr int kElems = 8;
};

__device__ __forceinline__ void unpack(const uint4& v, float (&f)[4], float) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float (&f)[8], __nv_bfloat16) {
    f[0] = bf16lo_to_f32(v.x);
    f[1] = bf16hi_to_f32(v.x);
    f[2] = bf16lo_to_f32(v.y);
    f[3] = bf16hi_to_f32(v.y);
    f[4] = bf16lo_to_f32(v.z);
    f[5] = bf16hi_to_f32(v.z);
    f[6] = bf16lo_to_f32(v.w);
    f[7] = bf16hi_to_f32(v.w);
}

__device__ __forceinline__ float load_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p) {
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
}

// VEC: rows start 16-byte aligned and C % kElems == 0, so every 16-byte
// vector is either wholly inside a row or wholly past its end.
template <typename Tin, bool VEC>
__global__ void __launch_bounds__(kThreads) mxfp8_quantize_kernel(const Tin* __restrict__ in,
                                                                  int64_t R, int64_t C, int64_t ld,
                                                                  uint8_t* __restrict__ codes,
                                                                  uint8_t* __restrict__ scales) {
    constexpr int E = VecTraits<Tin>::kElems;  // elements per 16-byte vector
    constexpr int TPB = 32 / E;                // lanes per 32-element block
    constexpr int STEP = 32 * E;               // elements per warp per unrolled step
    constexpr int SEG = STEP * kUnroll;        // elements per warp task
    const int lane = threadIdx.x & 31;
    const int64_t nb = (C + 31) / 32;
    const int64_t segs = (C + SEG - 1) / SEG;
    const int64_t tasks = R * segs;
    const int64_t warp0 = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kThreads) >> 5;

    for (int64_t task = warp0; task < tasks; task += nwarps) {
        const int64_t r = task / segs;
        const int64_t c_base = (task - r * segs) * SEG;
        const Tin* row = in + r * ld;
        float v[kUnroll][E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c0 = c_base + (int64_t)u * STEP + (int64_t)lane * E;
            if (VEC) {
                uint4 raw = make_uint4(0, 0, 0, 0);
                if (c0 < C) raw = __ldg(reinterpret_cast<const uint4*>(row + c0));
                unpack(raw, v[u], Tin());
            } else {
#pragma unroll
                for (int j = 0; j < E; ++j) v[u][j] = (c0 + j < C) ? load_elem(row + c0 + j) : 0.f;
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c0 = c_base + (int64_t)u * STEP + (int64_t)lane * E;
            float amax = 0.f;
            uint32_t bad = 0;
#pragma unroll
            for (int j = 0; j < E; ++j) {
                // elements past C were loaded as 0 and cannot raise the amax
                bad |= not_finite(v[u][j]) ? 1u : 0u;
                amax = fmaxf(amax, fabsf(v[u][j]));
            }
#pragma unroll
            for (int off = 1; off < TPB; off <<= 1) {
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
                bad |= __shfl_xor_sync(0xffffffffu, bad, off);
            }
            uint32_t w[E / 4];
            uint32_t sbyte;
            if (bad) {
                sbyte = 0xFFu;
#pragma unroll
                for (int q = 0; q < E / 4; ++q)
                    w[q] = nan_code(v[u][4 * q]) | (nan_code(v[u][4 * q + 1]) << 8) |
                           (nan_code(v[u][4 * q + 2]) << 16) | (nan_code(v[u][4 * q + 3]) << 24);
            } else {
                const int e = e8m0_exponent_f32(amax);
                const float s = exp2_neg(e);
                sbyte = (uint32_t)(e + 127);
#pragma unroll
                for (int q = 0; q < E / 4; ++q)
                    w[q] = pack_e4m3x4(v[u][4 * q] * s, v[u][4 * q + 1] * s, v[u][4 * q + 2] * s,
                                       v[u][4 * q + 3] * s);
            }
            if (c0 < C) {
                uint8_t* dst = codes + r * C + c0;
                if (VEC) {
                    if (E == 8)
                        *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[E / 4 - 1]);
                    else
                        *reinterpret_cast<uint32_t*>(dst) = w[0];
                } else {
#pragma unroll
                    for (int j = 0; j < E; ++j)
                        if (c0 + j < C) dst[j] = (uint8_t)(w[j / 4] >> (8 * (j % 4)));
                }
                if ((lane % TPB) == 0) scales[r * nb + c0 / 32] = (uint8_t)sbyte;
            }
        }
    }
}

template <typename Tin>
int launch_typed(int64_t R, int64_t C, const void* in, int64_t ld, uint8_t* codes, uint8_t* scales,
                 cudaStream_t stream) {
    constexpr int E = VecTraits<Tin>::kElems;
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    // Contiguous rows whose blocks never straddle a row end: one long row.
    if (ld == C && C % 32 == 0) {
        C = R * C;
        ld = C;
        R = 1;
    }
    const bool vec = (reinterpret_cast<uintptr_t>(in) % 16 == 0) &&
                     ((ld * (int64_t)sizeof(Tin)) % 16 == 0) && (C % E == 0) &&
                     (reinterpret_cast<uintptr_t>(codes) % 8 == 0);
    const int64_t seg = 32LL * E * kUnroll;
    const int64_t tasks = R * ((C + seg - 1) / seg);
    const int64_t warps_per_block = kThreads / 32;
    int64_t blocks = (tasks + warps_per_block - 1) / warps_per_block;
    const int64_t cap = (int64_t)di.num_sms * (2048 / kThreads);
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    const Tin* p = static_cast<const Tin*>(in);
    if (vec)
        mxfp8_quantize_kernel<Tin, true><<<(unsigned)blocks, kThreads, 0, stream>>>(p, R, C, ld, codes,
                                                                                   scales);
    else
        mxfp8_quantize_kernel<Tin, false><<<(unsigned)blocks, kThreads, 0, stream>>>(p, R, C, ld,
                                                                                    codes, scales);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

int launch_mxfp8_quantize(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                          uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
    if (in_dtype == MLA_IN_F32) return launch_typed<float>(R, C, in, ld_in, codes, scales, stream);
    return launch_typed<__nv_bfloat16>(R, C, in, ld_in, codes, scales, stream);
}

}  // namespace mlaq
