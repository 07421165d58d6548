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
// TILED: the scale of (row r, block c) goes to the GEMM's tiled order
// with row groups of sf_group (sf_tiled_offset, sf_nkt = ceil(nb / 4)); the
// host zero-fills the buffer first when it has padding.
template <typename Tin, bool VEC, bool TILED>
__global__ void __launch_bounds__(kThreads) mxfp8_quantize_kernel(const Tin* __restrict__ in,
                                                                  int64_t R, int64_t C, int64_t ld,
                                                                  uint8_t* __restrict__ codes,
                                                                  uint8_t* __restrict__ scales, int64_t sf_group,
                                                                  int64_t sf_nkt) {
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
            // NaN-propagating amax: Inf or NaN in the block leaves it non-finite;
            // elements past C were loaded as 0 and cannot raise it
            float amax = 0.f;
#pragma unroll
            for (int j = 0; j < E; ++j) amax = amax_nan(amax, v[u][j]);
#pragma unroll
            for (int off = 1; off < TPB; off <<= 1) amax = amax_nan(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const bool bad = __float_as_uint(amax) >= 0x7F800000u;
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
                if ((lane % TPB) == 0)
                    scales[TILED ? sf_tiled_offset(r, c0 / 32, sf_group, sf_nkt) : r * nb + c0 / 32] =
                        (uint8_t)sbyte;
            }
        }
    }
}

template <typename Tin>
int launch_typed(int64_t R, int64_t C, const void* in, int64_t ld, uint8_t* codes, uint8_t* scales,
                 cudaStream_t stream, int64_t sf_group = 0) {
    constexpr int E = VecTraits<Tin>::kElems;
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const int64_t nb = (C + 31) / 32, nkt = (nb + 3) / 4;
    if (sf_group > 0 && (sf_group % 128 || R % sf_group || nb % 4)) {
        // the tiled order has padding rows or columns: they read as 0
        if (cudaMemsetAsync(scales, 0, (size_t)sf_tiled_bytes(R, nb, sf_group), stream) != cudaSuccess)
            return MLA_ERR_CUDA;
    }
    // Contiguous rows whose blocks never straddle a row end: one long row
    // (scale positions unchanged only in the row-major order).
    if (sf_group == 0 && ld == C && C % 32 == 0) {
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
    const unsigned g = (unsigned)blocks;
    if (sf_group > 0) {
        if (vec) mxfp8_quantize_kernel<Tin, true, true><<<g, kThreads, 0, stream>>>(p, R, C, ld, codes, scales, sf_group, nkt);
        else mxfp8_quantize_kernel<Tin, false, true><<<g, kThreads, 0, stream>>>(p, R, C, ld, codes, scales, sf_group, nkt);
    } else {
        if (vec) mxfp8_quantize_kernel<Tin, true, false><<<g, kThreads, 0, stream>>>(p, R, C, ld, codes, scales, 0, 0);
        else mxfp8_quantize_kernel<Tin, false, false><<<g, kThreads, 0, stream>>>(p, R, C, ld, codes, scales, 0, 0);
    }
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// ------------------------------------------------------- columnwise copy
// The MXFP8 copy along the other axis (TransformerEngine PR "Add support for
// fused Q Up-Proj GEMM/RoPE/Quant", Greptile summary: the transpose helper
// among the MXFP8 quantization helpers), for GEMM operands that are reduced
// over their rows: codes_t [C, R] and scales_t [C, ceil(R/32)] are the
// rowwise quantization of in^T, i.e. blocks of 32 consecutive rows of one
// column.
//
// A CTA tile is 128 rows x 512 columns; each thread owns two adjacent
// columns and walks the tile's four 32-row blocks: for every row it loads
// its two elements (the warp reads 128 contiguous bytes of bf16 per row),
// keeps the block's 32 values of each column in registers, quantizes them
// and writes each column's 32 codes as one contiguous run of the output row.
constexpr int kColThreads = 256;
constexpr int kColTileR = 128;
constexpr int kColTileC = 2 * kColThreads;

__device__ __forceinline__ void load_pair(const float* p, bool both, float& a, float& b) {
    if (both) {
        const float2 v = __ldg(reinterpret_cast<const float2*>(p));
        a = v.x;
        b = v.y;
    } else {
        a = __ldg(p);
        b = 0.f;
    }
}
__device__ __forceinline__ void load_pair(const __nv_bfloat16* p, bool both, float& a, float& b) {
    if (both) {
        const uint32_t v = __ldg(reinterpret_cast<const unsigned int*>(p));
        a = bf16lo_to_f32(v);
        b = bf16hi_to_f32(v);
    } else {
        a = load_elem(p);
        b = 0.f;
    }
}

// One column's block: n valid codes to dst (32-byte run when whole and aligned).
// V32: dst 32-byte aligned; a whole block leaves in one 32-byte store
// (`st.global.v8.b32`, sm_100 and later), one full sector per instruction.
template <bool V32 = false>
__device__ __forceinline__ void store_codes(uint8_t* dst, const uint32_t (&w)[8], int n, bool vec) {
    if (V32 && n == 32) {
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
    } else if (vec && n == 32) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)  // unrolled: w stays in registers
            if (j < n) dst[j] = (uint8_t)(w[j / 4] >> (8 * (j % 4)));
    }
}

// PAIR: rows start 4-byte (bf16) / 8-byte (fp32) aligned, so a thread's two
// columns load as one vector when both exist. VEC: ldc % 16 == 0 and codes_t
// 16-byte aligned, so whole blocks store as two 16-byte vectors.
template <typename Tin, bool PAIR, bool VEC>
__global__ void __launch_bounds__(kColThreads) mxfp8_quantize_cols_kernel(const Tin* __restrict__ in, int64_t R,
                                                                      int64_t C, int64_t ld,
                                                                      uint8_t* __restrict__ codes, int64_t ldc,
                                                                      uint8_t* __restrict__ scales, int64_t nbr) {
    const int64_t tiles_r = (R + kColTileR - 1) / kColTileR;
    const int64_t tiles = tiles_r * ((C + kColTileC - 1) / kColTileC);
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t tr = tile % tiles_r, tc = tile / tiles_r;
        const int64_t c = tc * kColTileC + 2 * (int64_t)threadIdx.x;  // first of this thread's columns
        const bool has0 = c < C, has1 = c + 1 < C;
#pragma unroll 1
        for (int blk = 0; blk < kColTileR / 32; ++blk) {
            const int64_t r0 = tr * kColTileR + 32 * blk;
            if (r0 >= R) break;
            const int n = (R - r0) < 32 ? (int)(R - r0) : 32;
            float a[32], b[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                a[i] = 0.f;
                b[i] = 0.f;
                if (i < n && has0) {
                    const Tin* src = in + (r0 + i) * ld + c;
                    if (PAIR) {
                        load_pair(src, has1, a[i], b[i]);
                    } else {
                        a[i] = load_elem(src);
                        if (has1) b[i] = load_elem(src + 1);
                    }
                }
            }
            uint32_t wa[8], wb[8];
            const uint32_t sa = quantize_block_regs<32>(a, n, wa);
            const uint32_t sb = quantize_block_regs<32>(b, n, wb);
            if (has0) {
                store_codes(codes + c * ldc + r0, wa, n, VEC);
                scales[c * nbr + r0 / 32] = (uint8_t)sa;
            }
            if (has1) {
                store_codes(codes + (c + 1) * ldc + r0, wb, n, VEC);
                scales[(c + 1) * nbr + r0 / 32] = (uint8_t)sb;
            }
        }
    }
}

// Fast path: rows 16-byte aligned and C a multiple of the 16-byte vector.
// A tile is 128 rows x 256 columns, loaded as four 32-row blocks with
// 16-byte cp.async into a ring of shared-memory buffers (every warp load is
// 512 contiguous bytes of a row). Each thread then takes CPT adjacent
// columns of a block (bf16: two, read together by one 4-byte shared load per
// row; fp32: one), quantizes each column's 32 values and writes its 32
// codes as one run; a column's 4 scale bytes of the tile leave as one 4-byte
// word when the scale rows allow it.
constexpr int kColTC = 256;
template <typename Tin>
__host__ __device__ constexpr int cols_nbuf() { return sizeof(Tin) == 2 ? 4 : 2; }
template <typename Tin>
__host__ __device__ constexpr uint32_t cols_buf_bytes() { return 32u * kColTC * (uint32_t)sizeof(Tin); }
template <typename Tin>
__host__ __device__ constexpr int cols_cpt() { return sizeof(Tin) == 2 ? 2 : 1; }  // columns per thread
template <typename Tin>
__host__ __device__ constexpr int cols_threads() { return kColTC / cols_cpt<Tin>(); }

// V32: ldc % 32 == 0 and codes 32-byte aligned (every block's run is 32-byte aligned)
template <typename Tin, bool VEC, bool V32 = false>
__global__ void __launch_bounds__(cols_threads<Tin>()) mxfp8_quantize_cols_tiled(
    const Tin* __restrict__ in, int64_t R, int64_t C, int64_t ld, uint8_t* __restrict__ codes, int64_t ldc,
    uint8_t* __restrict__ scales, int64_t nbr, int64_t sf_group) {
    extern __shared__ __align__(16) uint8_t smem[];
    constexpr int NBUF = cols_nbuf<Tin>();
    constexpr uint32_t BUF = cols_buf_bytes<Tin>();
    constexpr int CPT = cols_cpt<Tin>();
    constexpr int NT = cols_threads<Tin>();
    constexpr int EPV = 16 / (int)sizeof(Tin);      // elements per 16-byte vector
    constexpr int VPR = kColTC / EPV;                // vectors per tile row
    constexpr int VPT = 32 * VPR / NT;               // vectors per thread per block
    constexpr int NB = kColTileR / 32;               // blocks per tile
    constexpr uint32_t ROWB = (uint32_t)kColTC * (uint32_t)sizeof(Tin);  // bytes per staged row
    const uint32_t sbase = smem_u32(smem);
    const int t = threadIdx.x;
    const int64_t tiles_r = (R + kColTileR - 1) / kColTileR;
    const int64_t tiles = tiles_r * ((C + kColTC - 1) / kColTC);
    // a row's scale pitch holds whole 4-byte words for every tile (bytes of blocks past R are 0);
    // always so in the GEMM's tiled order (sf_group > 0), where a tile's 4 bytes are one word
    const bool word_scales = sf_group > 0 || ((nbr % 4) == 0 && nbr >= 4 * tiles_r &&
                                              (reinterpret_cast<uintptr_t>(scales) % 4) == 0);
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
        const int64_t tr = tile % tiles_r, tc = tile / tiles_r;
        const int64_t c0 = tc * kColTC;
        auto issue = [&](int b) {
            const int64_t r0 = tr * kColTileR + 32 * b;
            const uint32_t buf = sbase + (uint32_t)(b % NBUF) * BUF;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int idx = t + k * NT;
                const int row = idx / VPR, vc = idx % VPR;
                const int64_t r = r0 + row, c = c0 + (int64_t)vc * EPV;
                const bool ok = r < R && c < C;
                const Tin* src = ok ? in + r * ld + c : in;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(buf + (uint32_t)row * ROWB + (uint32_t)(vc * 16)),
                             "l"(src), "r"(ok ? 16 : 0)
                             : "memory");
            }
        };
        for (int b = 0; b < NBUF - 1; ++b) {
            if (b < NB) issue(b);
            cp_async_commit();
        }
        const int64_t c = c0 + (int64_t)CPT * t;  // this thread's first column (C % EPV == 0: all CPT exist or none)
        uint32_t sword[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) sword[j] = 0;
        for (int blk = 0; blk < NB; ++blk) {
            if (blk + NBUF - 1 < NB) issue(blk + NBUF - 1);
            cp_async_commit();
            asm volatile("cp.async.wait_group %0;" ::"n"(NBUF - 1) : "memory");
            __syncthreads();
            const int64_t r0 = tr * kColTileR + 32 * blk;
            if (r0 < R && c < C) {
                const int n = (R - r0) < 32 ? (int)(R - r0) : 32;
                const uint32_t buf = sbase + (uint32_t)(blk % NBUF) * BUF + (uint32_t)(t * CPT * (int)sizeof(Tin));
                float v[CPT][32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t w = lds_b32(buf + (uint32_t)i * ROWB);
                    if (sizeof(Tin) == 2) {
                        v[0][i] = bf16lo_to_f32(w);
                        v[CPT - 1][i] = bf16hi_to_f32(w);
                    } else {
                        v[0][i] = __uint_as_float(w);
                    }
                }
                // rows past R were zero-filled by the loads: they leave the amax unchanged
#pragma unroll
                for (int j = 0; j < CPT; ++j) {
                    uint32_t w[8];
                    const uint32_t sb = quantize_block32(v[j], w);
                    store_codes<V32>(codes + (c + j) * ldc + r0, w, n, VEC);
                    if (word_scales) sword[j] |= sb << (8 * blk);
                    else scales[(c + j) * nbr + r0 / 32] = (uint8_t)sb;
                }
            }
            __syncthreads();  // the buffer may be refilled now
        }
        if (word_scales && c < C && tr * kColTileR < R) {
#pragma unroll
            for (int j = 0; j < CPT; ++j)
                *reinterpret_cast<uint32_t*>(scales + (sf_group > 0 ? sf_tiled_offset(c + j, tr * NB, sf_group, tiles_r)
                                                                    : (c + j) * nbr + tr * NB)) = sword[j];
        }
    }
}

// ------------------------------------------------------- scale swizzle
// Row-major E8M0 scales [rows, cols] -> the tiled order block-scaled GEMMs
// read (TransformerEngine PR "Add support for fused Q Up-Proj
// GEMM/RoPE/Quant": the GEMM scale swizzle among its MXFP8 helpers): rows in
// groups of G (the GEMM's tile height along that operand), each group padded
// to whole 128-row chunks; chunk i of group g and column tile j (4 scale
// columns) is the 512-byte tile ((g * ceil(G/128) + i) * ceil(cols/4) + j);
// inside it, row r of the chunk and column c at byte
// (r % 32) * 16 + (r / 32) * 4 + (c % 4). Bytes past the rows of a group or
// past cols are 0. With G = 128 this is the plain swizzle of the matrix.
// One thread writes the 16 bytes of one (tile, r % 32) pair.
__global__ void __launch_bounds__(256) mxfp8_swizzle_kernel(const uint8_t* __restrict__ in, int64_t rows,
                                                            int64_t cols, int64_t ld, int64_t group, int64_t nsub,
                                                            uint8_t* __restrict__ out, int64_t tiles_c,
                                                            int64_t nthreads) {
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < nthreads;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t tile = g / 32;
        const int r32 = (int)(g % 32);
        const int64_t ti = tile / tiles_c, tj = tile % tiles_c;
        const int64_t grp = ti / nsub, chunk = ti % nsub;
        uint32_t w[4];
#pragma unroll
        for (int rb = 0; rb < 4; ++rb) {
            const int64_t rg = chunk * 128 + rb * 32 + r32;  // row within the group
            const int64_t r = grp * group + rg;
            uint32_t word = 0;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                const int64_t c = tj * 4 + cc;
                if (rg < group && r < rows && c < cols) word |= (uint32_t)__ldg(in + r * ld + c) << (8 * cc);
            }
            w[rb] = word;
        }
        *reinterpret_cast<uint4*>(out + tile * 512 + r32 * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

template <typename Tin>
int launch_cols_typed(int64_t R, int64_t C, const void* in, int64_t ld, uint8_t* codes, int64_t ldc,
                      uint8_t* scales, int64_t lds, cudaStream_t stream, int64_t sf_group = 0) {
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const bool pair = (reinterpret_cast<uintptr_t>(in) % (2 * sizeof(Tin)) == 0) && (ld % 2 == 0);
    const bool vec = (ldc % 16 == 0) && (reinterpret_cast<uintptr_t>(codes) % 16 == 0);
    constexpr int EPV = 16 / (int)sizeof(Tin);
    if (reinterpret_cast<uintptr_t>(in) % 16 == 0 && (ld * (int64_t)sizeof(Tin)) % 16 == 0 && C % EPV == 0) {
        const size_t smem = (size_t)cols_nbuf<Tin>() * cols_buf_bytes<Tin>();
        const int64_t tiles = ((R + kColTileR - 1) / kColTileR) * ((C + kColTC - 1) / kColTC);
        int64_t blocks = tiles;
        const int64_t cap = (int64_t)di.num_sms * 3;
        if (blocks > cap) blocks = cap;
        const Tin* p = static_cast<const Tin*>(in);
        const bool v32 = vec && (ldc % 32 == 0) && (reinterpret_cast<uintptr_t>(codes) % 32 == 0);
        const void* k = v32   ? (const void*)mxfp8_quantize_cols_tiled<Tin, true, true>
                        : vec ? (const void*)mxfp8_quantize_cols_tiled<Tin, true>
                              : (const void*)mxfp8_quantize_cols_tiled<Tin, false>;
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return MLA_ERR_CUDA;
        constexpr int NT = cols_threads<Tin>();
        if (v32)
            mxfp8_quantize_cols_tiled<Tin, true, true><<<(unsigned)blocks, NT, smem, stream>>>(p, R, C, ld, codes, ldc, scales, lds, sf_group);
        else if (vec)
            mxfp8_quantize_cols_tiled<Tin, true><<<(unsigned)blocks, NT, smem, stream>>>(p, R, C, ld, codes, ldc, scales, lds, sf_group);
        else
            mxfp8_quantize_cols_tiled<Tin, false><<<(unsigned)blocks, NT, smem, stream>>>(p, R, C, ld, codes, ldc, scales, lds, sf_group);
        return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
    }
    if (sf_group > 0) return MLA_ERR_UNSUPPORTED;  // the tiled scale order needs the fast path
    const int64_t tiles = ((R + kColTileR - 1) / kColTileR) * ((C + kColTileC - 1) / kColTileC);
    int64_t blocks = tiles;
    const int64_t cap = (int64_t)di.num_sms * (2048 / kColThreads);
    if (blocks > cap) blocks = cap;
    const Tin* p = static_cast<const Tin*>(in);
    const unsigned g = (unsigned)blocks;
    if (pair && vec) mxfp8_quantize_cols_kernel<Tin, true, true><<<g, kColThreads, 0, stream>>>(p, R, C, ld, codes, ldc, scales, lds);
    else if (pair) mxfp8_quantize_cols_kernel<Tin, true, false><<<g, kColThreads, 0, stream>>>(p, R, C, ld, codes, ldc, scales, lds);
    else if (vec) mxfp8_quantize_cols_kernel<Tin, false, true><<<g, kColThreads, 0, stream>>>(p, R, C, ld, codes, ldc, scales, lds);
    else mxfp8_quantize_cols_kernel<Tin, false, false><<<g, kColThreads, 0, stream>>>(p, R, C, ld, codes, ldc, scales, lds);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

int launch_mxfp8_quantize(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                          uint8_t* codes, uint8_t* scales, cudaStream_t stream, int64_t sf_group) {
    if (in_dtype == MLA_IN_F32) return launch_typed<float>(R, C, in, ld_in, codes, scales, stream, sf_group);
    return launch_typed<__nv_bfloat16>(R, C, in, ld_in, codes, scales, stream, sf_group);
}

}  // namespace mlaq

namespace mlaq {
int launch_mxfp8_quantize_cols(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                               uint8_t* codes_t, uint8_t* scales_t, cudaStream_t stream) {
    return launch_mxfp8_quantize_cols_ld(R, C, in_dtype, in, ld_in, codes_t, R, scales_t, (R + 31) / 32, stream);
}

int launch_mxfp8_quantize_cols_tiled_sf(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                        uint8_t* codes_t, int64_t ld_codes, uint8_t* scales_t, int64_t sf_group,
                                        cudaStream_t stream) {
    if (sf_group <= 0) return MLA_ERR_INVALID_ARG;
    if (in_dtype == MLA_IN_F32)
        return launch_cols_typed<float>(R, C, in, ld_in, codes_t, ld_codes, scales_t, 0, stream, sf_group);
    return launch_cols_typed<__nv_bfloat16>(R, C, in, ld_in, codes_t, ld_codes, scales_t, 0, stream, sf_group);
}

int launch_mxfp8_quantize_cols_ld(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                  uint8_t* codes_t, int64_t ld_codes, uint8_t* scales_t, int64_t ld_scales,
                                  cudaStream_t stream) {
    if (in_dtype == MLA_IN_F32)
        return launch_cols_typed<float>(R, C, in, ld_in, codes_t, ld_codes, scales_t, ld_scales, stream);
    return launch_cols_typed<__nv_bfloat16>(R, C, in, ld_in, codes_t, ld_codes, scales_t, ld_scales, stream);
}
}  // namespace mlaq

namespace mlaq {
int launch_mxfp8_swizzle(int64_t rows, int64_t cols, int64_t group, const uint8_t* in, int64_t ld, uint8_t* out,
                         cudaStream_t stream) {
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const int64_t tiles_c = (cols + 3) / 4;
    const int64_t nsub = (group + 127) / 128;
    const int64_t n = ((rows + group - 1) / group) * nsub * tiles_c * 32;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)di.num_sms * 8;
    if (blocks > cap) blocks = cap;
    mxfp8_swizzle_kernel<<<(unsigned)blocks, 256, 0, stream>>>(in, rows, cols, ld, group, nsub, out, tiles_c, n);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
}  // namespace mlaq
