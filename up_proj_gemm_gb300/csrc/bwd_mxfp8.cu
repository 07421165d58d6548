// MXFP8 backward: the low-precision backward beyond the fused bf16 one.
//
// TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant"
// names the MXFP8 quantization helpers (rowwise, the transpose copy, the
// GEMM scale swizzle) such a backward is built from; the pages give no
// formula. The reading implemented here: dq_pre = the inverse rotation of dq
// in float32 (each product and sum rounded once, in a fixed order), each GEMM
// operand quantized to MXFP8 along its reduction dimension, and the GEMMs run
// on the block-scaled tensor cores:
//   dgrad  dx = Q_rows(dq_pre) [T x N] . Q_cols(W)^T [K x N]   (blocks along N)
//   wgrad  dW = Q_cols(dq_pre) [N x T] . Q_cols(x)^T  [K x T]  (blocks along T)
//   bgrad  db = sum_t dq_pre (float32 partial sums per 32-token block, fixed order)
//
// This file holds the pass that rotates dq and writes both MXFP8 copies of
// dq_pre plus the db partials in one read of dq, and the db reduction. The
// GEMMs are the forward kernel's block-scaled main loop with a plain bf16
// epilogue (no rotation); the W and x copies come from the columnwise
// quantizer.
#include <cuda_bf16.h>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kRqThreads = 256;

__device__ __forceinline__ void load8_f32(const float* src, bool vec, float (&o)[8]) {
    if (vec) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(src));
        const float4 b = __ldg(reinterpret_cast<const float4*>(src) + 1);
        o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
        o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = __ldg(src + e);
    }
}

__device__ __forceinline__ void unpack8(uint4 raw, float (&v)[8]) {
    v[0] = bf16lo_to_f32(raw.x);
    v[1] = bf16hi_to_f32(raw.x);
    v[2] = bf16lo_to_f32(raw.y);
    v[3] = bf16hi_to_f32(raw.y);
    v[4] = bf16lo_to_f32(raw.z);
    v[5] = bf16hi_to_f32(raw.z);
    v[6] = bf16lo_to_f32(raw.w);
    v[7] = bf16hi_to_f32(raw.w);
}

// Outputs of one pass (all in the workspace):
//   qa [T, N]: rowwise codes; qa_s: their scales in the GEMM tiled order
//     (rows = tokens up to Tp, G = 128, nkt_n = N / 128 K steps)
//   qb [N, Tp]: columnwise codes (tokens past T are 0); qb_s: tiled order
//     (rows = channels, G = 128, nkt_t = Tp / 128 K steps)
//   dbp [ceil(T/32), N]: float32 sums of each 32-token block
// Every scale byte of both tiled arrays is written (0 where the values are 0).
struct RqArgs {
    const uint16_t* dq;
    int64_t T, Tp;
    int H, Dn;
    const float* cos_tab;
    const float* sin_tab;
    int64_t cs_rows, cs_width;
    int cs_vec;
    const int32_t* pos;
    uint8_t* qa;
    uint8_t* qa_s;
    uint8_t* qb;
    uint8_t* qb_s;
    float* dbp;
    int* status;
};

// Fast path: a CTA takes 128 tokens x 64 channels of dq viewed as [T, N]
// (N % 64 == 0; a 64-channel span is all rope or all pass-through when
// Dn % 64 == 0 and Dr == 64, and holds a whole rope half-pair set when
// Dr == 32). Tiles go channel span fastest.
//  * rows: 8 lanes per token row (16 bytes = 8 channels each), 4 rows per
//    warp at a time, 4 passes for the CTA's 128 rows, all loads issued
//    first. A 32-channel block is a lane quad (amax by two shuffles); a rope
//    pair's partner channels sit Dr/16 lanes away in the same row (one
//    shuffle exchange); the rope arithmetic runs only in rope spans.
//  * the rotated float32 rows go to a shared tile [128][64]; then warp w
//    takes token block w / 2 (32 tokens) and channels 32 (w % 2) + lane:
//    it quantizes that channel's block, stores 32 codes (the CTA writes each
//    channel's 128 tokens, one whole 128-byte line of qb) and the block's
//    float32 sum for db.
// V32: qb 32-byte aligned (its rows are Tp bytes, Tp % 128 == 0): a block's
// 32 codes leave in one 32-byte store (`st.global.v8.b32`, sm_100 and later)
template <int DR, bool V32>
__global__ void __launch_bounds__(kRqThreads) rope_bwd_quant_fast(const RqArgs a) {
    __shared__ __align__(16) float tile[128][64];
    constexpr int HH = DR / 2;
    constexpr int PX = HH / 8;  // lanes between the two channels of a rope pair
    const int D = a.Dn + DR;
    const int N = a.H * D;
    const int nsp = N / 64;     // channel spans
    const int ts = (int)(blockIdx.x / nsp), sp = (int)(blockIdx.x % nsp);
    const int64_t t0 = (int64_t)ts * 128;
    const int n0 = sp * 64;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 3, j = lane & 7;  // row within the warp's 4, 16-byte chunk of the row
    const int n = n0 + 8 * j;
    const int c = n % D;          // channel within the head
    const bool rope = c >= a.Dn;  // (a whole span when Dr == 64)
    const int q0 = c - a.Dn;      // rope index of the lane's first channel
    const bool first = q0 < HH;   // holds i (else i + Dr/2) of its pairs
    const int nkt_n = N / 128;
    uint4 raws[4];
    int pps[4];
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int64_t t = t0 + it * 32 + warp * 4 + g;
        raws[it] = make_uint4(0, 0, 0, 0);
        pps[it] = 0;
        if (t < a.T) {
            raws[it] = __ldg(reinterpret_cast<const uint4*>(a.dq + t * N + n));
            if (rope) pps[it] = a.pos ? __ldg(a.pos + t) : (int)t;
        }
    }
    const bool rope_span = __any_sync(0xffffffffu, rope);  // warp-uniform
#pragma unroll
    for (int it = 0; it < 4; ++it) {
        const int r = it * 32 + warp * 4 + g;
        const int64_t t = t0 + r;
        float v[8];
        unpack8(raws[it], v);
        if (rope_span) {
            uint4 pr;
            pr.x = __shfl_xor_sync(0xffffffffu, raws[it].x, PX);
            pr.y = __shfl_xor_sync(0xffffffffu, raws[it].y, PX);
            pr.z = __shfl_xor_sync(0xffffffffu, raws[it].z, PX);
            pr.w = __shfl_xor_sync(0xffffffffu, raws[it].w, PX);
            if (rope && t < a.T) {
                const int pp = pps[it];
                if (pp < 0 || pp >= a.cs_rows) {
                    record_status(a.status, MLA_ERR_POS_RANGE);
                } else {
                    // out_i = fl(fl(g_i c_i) + fl(g_{i+h} s_{i+h})), out_{i+h} = fl(fl(g_{i+h} c_{i+h}) - fl(g_i s_i));
                    // the second half adds fl(g_i * -s_i) = -fl(g_i s_i) (negation is exact), one formula
                    float o[8], cw[8], sw[8];
                    unpack8(pr, o);
                    const int64_t row0 = (int64_t)pp * a.cs_width;
                    load8_f32(a.cos_tab + row0 + q0, a.cs_vec != 0, cw);
                    load8_f32(a.sin_tab + row0 + (first ? q0 + HH : q0 - HH), a.cs_vec != 0, sw);
                    const uint32_t neg = first ? 0u : 0x80000000u;
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        v[k] = __fadd_rn(__fmul_rn(v[k], cw[k]),
                                         __fmul_rn(o[k], __uint_as_float(__float_as_uint(sw[k]) ^ neg)));
                }
            }
        }
        // rowwise block of 32 channels = this lane quad (NaN-propagating amax)
        float am = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) am = amax_nan(am, v[k]);
        am = amax_nan(am, __shfl_xor_sync(0xffffffffu, am, 1));
        am = amax_nan(am, __shfl_xor_sync(0xffffffffu, am, 2));
        if (a.qa) {
            uint32_t w[2];
            const uint32_t sb = quantize8_block_scale(v, __float_as_uint(am), w);
            if (t < a.T) *reinterpret_cast<uint2*>(a.qa + t * N + n) = make_uint2(w[0], w[1]);
            // the row's two scale bytes (blocks n0/32 and n0/32 + 1) are adjacent in the tiled order
            const uint32_t pair = sb | (__shfl_down_sync(0xffffffffu, sb, 4) << 8);
            if (j == 0)
                *reinterpret_cast<uint16_t*>(a.qa_s + sf_tiled_offset(t, n0 / 32, 128, nkt_n)) = (uint16_t)pair;
        }
        // lanes with bit 2 set store their halves in the other order: no bank conflicts
        float* dst = &tile[r][8 * j];
        const float4 lo = make_float4(v[0], v[1], v[2], v[3]), hi = make_float4(v[4], v[5], v[6], v[7]);
        if (j & 4) {
            *reinterpret_cast<float4*>(dst + 4) = hi;
            *reinterpret_cast<float4*>(dst) = lo;
        } else {
            *reinterpret_cast<float4*>(dst) = lo;
            *reinterpret_cast<float4*>(dst + 4) = hi;
        }
    }
    __syncthreads();
    // token block tb (32 tokens) of channel ch
    const int blk = warp >> 1;
    const int col = 32 * (warp & 1) + lane;
    const int64_t ch = n0 + col;
    const int64_t tb = (int64_t)ts * 4 + blk;
    float v[32];
    float sum = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        v[r] = tile[32 * blk + r][col];
        sum += v[r];  // token order; rows past T are 0
    }
    if (a.qb) {
        // rows past T hold zeros: they leave the amax unchanged and encode as 0
        uint32_t w[8];
        const uint32_t sb = quantize_block32(v, w);
        uint8_t* dst = a.qb + ch * a.Tp + tb * 32;
        if (V32) {
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                         "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                         : "memory");
        } else {
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        a.qb_s[sf_tiled_offset(ch, tb, 128, a.Tp / 128)] = (uint8_t)sb;
    }
    if (a.dbp && tb * 32 < a.T) a.dbp[tb * N + ch] = sum;
}

// General shapes: a CTA takes 32 tokens x one head (D % 32 == 0), staged in
// shared memory as float32 with a row pitch of D + 1 words; same outputs.
template <int DR>
__global__ void __launch_bounds__(kRqThreads) rope_bwd_quant_kernel(const RqArgs a) {
    extern __shared__ float stile[];
    constexpr int HH = DR / 2;
    const int D = a.Dn + DR;
    const int P = D + 1;  // row pitch (words)
    const int64_t N = (int64_t)a.H * D;
    const int64_t ntb = a.Tp / 32;
    const int64_t tb = blockIdx.x % ntb;
    const int h = (int)(blockIdx.x / ntb);
    const int64_t t0 = tb * 32;
    const int tid = threadIdx.x;
    const int vpr = D / 8;
    for (int k = tid; k < 32 * vpr; k += kRqThreads) {
        const int r = k / vpr, v = k % vpr;
        const int64_t t = t0 + r;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (t < a.T) raw = __ldg(reinterpret_cast<const uint4*>(a.dq + t * N + (int64_t)h * D + 8 * v));
        float f[8];
        unpack8(raw, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) stile[r * P + 8 * v + e] = f[e];
    }
    __syncthreads();
    for (int k = tid; k < 32 * HH; k += kRqThreads) {
        const int r = k / HH, i = k % HH;
        const int64_t t = t0 + r;
        if (t >= a.T) continue;
        const int64_t pp = a.pos ? (int64_t)__ldg(a.pos + t) : t;
        if (pp < 0 || pp >= a.cs_rows) {
            record_status(a.status, MLA_ERR_POS_RANGE);
            continue;
        }
        const float* cs = a.cos_tab + pp * a.cs_width;
        const float* sn = a.sin_tab + pp * a.cs_width;
        float* row = stile + r * P + a.Dn;
        const float g0 = row[i], g1 = row[i + HH];
        row[i] = __fadd_rn(__fmul_rn(g0, __ldg(cs + i)), __fmul_rn(g1, __ldg(sn + i + HH)));
        row[i + HH] = __fsub_rn(__fmul_rn(g1, __ldg(cs + i + HH)), __fmul_rn(g0, __ldg(sn + i)));
    }
    __syncthreads();
    const int nb = D / 32;
    const int64_t nkt_n = N / 128;
    for (int k = tid; a.qa && k < 32 * nb; k += kRqThreads) {
        const int b = k / 32, r = k % 32;
        const int64_t t = t0 + r;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = stile[r * P + 32 * b + i];
        uint32_t w[8];
        const uint32_t sb = quantize_block_regs<32>(v, 32, w);
        const int64_t blk = ((int64_t)h * D) / 32 + b;
        if (t < a.T) {
            uint8_t* dst = a.qa + t * N + (int64_t)h * D + 32 * b;
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        a.qa_s[sf_tiled_offset(t, blk, 128, nkt_n)] = (uint8_t)sb;
    }
    const int64_t left = a.T - t0;
    const int nv = left <= 0 ? 0 : (left < 32 ? (int)left : 32);
    for (int c = tid; c < D; c += kRqThreads) {
        float v[32];
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            v[r] = stile[r * P + c];
            sum += v[r];
        }
        const int64_t ch = (int64_t)h * D + c;
        if (a.qb) {
            uint32_t w[8];
            const uint32_t sb = quantize_block_regs<32>(v, nv, w);
            uint8_t* dst = a.qb + ch * a.Tp + t0;
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
            a.qb_s[sf_tiled_offset(ch, tb, 128, a.Tp / 128)] = (uint8_t)sb;
        }
        if (a.dbp && t0 < a.T) a.dbp[tb * N + ch] = sum;
    }
}

// db[n] = bf16(sum over token blocks b = 0, 1, ... of dbp[b, n]), in that
// order (float32); nblk = 0 gives zeros.
__global__ void __launch_bounds__(256) db_reduce_kernel(const float* __restrict__ dbp, int64_t nblk, int64_t N,
                                                        uint16_t* __restrict__ db) {
    for (int64_t n = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; n < N; n += (int64_t)gridDim.x * blockDim.x) {
        float s = 0.f;
        for (int64_t b = 0; b < nblk; ++b) s += dbp[b * N + n];
        db[n] = (uint16_t)(pack_bf16x2(s, 0.f) & 0xFFFFu);
    }
}

// out[0, n) = 0 (16-byte words; n % 16 == 0, out 16-byte aligned)
__global__ void __launch_bounds__(256) zero_fill_kernel(uint4* __restrict__ out, int64_t words) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < words; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = make_uint4(0, 0, 0, 0);
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

unsigned grid_for(int64_t items, int64_t per_block, int64_t cap) {
    int64_t b = (items + per_block - 1) / per_block;
    if (b < 1) b = 1;
    if (b > cap) b = cap;
    return (unsigned)b;
}

}  // namespace

int bwd_mxfp8_layout(int64_t T, int64_t K, int64_t N, Mxfp8BwdLayout* L) {
    if (T < 0 || K <= 0 || N <= 0 || !L) return MLA_ERR_INVALID_ARG;
    const int64_t G = fwd_tile_n(K, (int)K, (int)K, 0, 192, 32);  // the GEMMs' tile width over K
    if (G == 0) return MLA_ERR_UNSUPPORTED;
    const int64_t Tp = (T + 127) / 128 * 128;
    const int64_t nbt = (T + 31) / 32;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L->Tp = Tp;
    L->G = G;
    L->qa = take((size_t)T * N);
    L->qa_s = take((size_t)sf_tiled_bytes(Tp, N / 32, 128));
    L->qb = take((size_t)N * Tp);
    L->qb_s = take((size_t)sf_tiled_bytes(N, Tp / 32, 128));
    L->wt = take((size_t)K * N);
    L->wt_s = take((size_t)sf_tiled_bytes(K, N / 32, G));
    L->xt = take((size_t)K * Tp);
    L->xt_s = take((size_t)sf_tiled_bytes(K, Tp / 32, G));
    L->dbp = take((size_t)nbt * N * sizeof(float));
    L->total = off;
    return MLA_OK;
}

int launch_rope_bwd_quant(const BwdArgs& a, int64_t Tp, uint8_t* qa, uint8_t* qa_s, uint8_t* qb, uint8_t* qb_s,
                          float* dbp, cudaStream_t stream) {
    RqArgs r{};
    r.dq = static_cast<const uint16_t*>(a.dq);
    r.T = a.T;
    r.Tp = Tp;
    r.H = a.H;
    r.Dn = a.Dn;
    r.cos_tab = a.cos_tab;
    r.sin_tab = a.sin_tab;
    r.cs_rows = a.cs_rows;
    r.cs_width = a.cs_width;
    r.cs_vec = (a.cs_width % 4 == 0) && (reinterpret_cast<uintptr_t>(a.cos_tab) % 16 == 0) &&
               (reinterpret_cast<uintptr_t>(a.sin_tab) % 16 == 0);
    r.pos = a.pos;
    r.qa = qa;
    r.qa_s = qa_s;
    r.qb = qb;
    r.qb_s = qb_s;
    r.dbp = dbp;
    r.status = a.status;
    const int D = a.Dn + a.Dr;
    const int64_t N = (int64_t)a.H * D;
    const int64_t ntb = Tp / 32;
    // the fast path needs whole 64-channel spans, each all rope or all pass-through
    // (or a whole 32-channel rope region), and 32-bit tile indices
    const bool fast = N % 64 == 0 && (a.Dr == 32 || (a.Dr == 64 && a.Dn % 64 == 0)) &&
                      (Tp / 128) * (N / 64) <= 0x7fffffffLL;
    if (fast) {
        const unsigned grid = (unsigned)((Tp / 128) * (N / 64));
        const bool v32 = reinterpret_cast<uintptr_t>(qb) % 32 == 0;
        if (a.Dr == 32 && v32) rope_bwd_quant_fast<32, true><<<grid, kRqThreads, 0, stream>>>(r);
        else if (a.Dr == 32) rope_bwd_quant_fast<32, false><<<grid, kRqThreads, 0, stream>>>(r);
        else if (v32) rope_bwd_quant_fast<64, true><<<grid, kRqThreads, 0, stream>>>(r);
        else rope_bwd_quant_fast<64, false><<<grid, kRqThreads, 0, stream>>>(r);
        return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
    }
    const size_t smem = (size_t)32 * (D + 1) * sizeof(float);
    const unsigned grid = (unsigned)(ntb * a.H);
    const void* k = a.Dr == 32 ? (const void*)rope_bwd_quant_kernel<32> : (const void*)rope_bwd_quant_kernel<64>;
    if (a.Dr != 32 && a.Dr != 64) return MLA_ERR_UNSUPPORTED;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MLA_ERR_CUDA;
    if (a.Dr == 32) rope_bwd_quant_kernel<32><<<grid, kRqThreads, smem, stream>>>(r);
    else rope_bwd_quant_kernel<64><<<grid, kRqThreads, smem, stream>>>(r);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int launch_bwd_mxfp8(const BwdArgs& a, cudaStream_t stream) {
    const int D = a.Dn + a.Dr;
    const int64_t N = (int64_t)a.H * D;
    const int64_t T = a.T, K = a.K;
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const int64_t cap = (int64_t)di.num_sms * 8;
    if (T == 0) {  // empty token sum: dW = 0, db = 0
        if (a.dW) {
            zero_fill_kernel<<<grid_for(N * K * 2 / 16, 256, cap), 256, 0, stream>>>(static_cast<uint4*>(a.dW),
                                                                                    N * K * 2 / 16);
            if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
        }
        if (a.db) {
            db_reduce_kernel<<<grid_for(N, 256, cap), 256, 0, stream>>>(nullptr, 0, N, static_cast<uint16_t*>(a.db));
            if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
        }
        return MLA_OK;
    }
    Mxfp8BwdLayout L;
    st = bwd_mxfp8_layout(T, K, N, &L);
    if (st != MLA_OK) return st;
    uint8_t* ws = static_cast<uint8_t*>(a.workspace);
    const bool want_dx = a.dx != nullptr, want_dw = a.dW != nullptr, want_db = a.db != nullptr;
    // 1. rotate dq once: both MXFP8 copies of dq_pre (scales in the GEMM's tiled order) and the db partials
    st = launch_rope_bwd_quant(a, L.Tp, want_dx ? ws + L.qa : nullptr, ws + L.qa_s, want_dw ? ws + L.qb : nullptr,
                               ws + L.qb_s, want_db ? reinterpret_cast<float*>(ws + L.dbp) : nullptr, stream);
    if (st != MLA_OK) return st;
    if (want_dx) {
        // 2. W [N, K] -> wt [K, N], blocks along N (unless the caller prepared it);
        // 3. dx = qa . wt^T (block-scaled GEMM, reduction over N)
        const uint8_t* wt = a.wt ? a.wt : ws + L.wt;
        const uint8_t* wt_s = a.wt ? a.wt_s : ws + L.wt_s;
        if (!a.wt) {
            st = launch_mxfp8_quantize_cols_tiled_sf(N, K, MLA_IN_BF16, a.W, K, ws + L.wt, N, ws + L.wt_s, L.G,
                                                     stream);
            if (st != MLA_OK) return st;
        }
        FwdArgs g{};
        g.T = T;
        g.K = N;
        g.H = 1;
        g.Dn = (int)K;
        g.Dr = 0;
        g.weight_mode = MLA_WEIGHT_MXFP8;
        g.out_mode = MLA_OUT_BF16;
        g.x = ws + L.qa;
        g.x_scales = ws + L.qa_s;
        g.W = wt;
        g.w_scales = wt_s;
        g.sf_tiled = 1;
        g.sf_group = (int)L.G;
        g.q_out = a.dx;
        g.status = a.status;
        st = launch_fwd(g, stream);
        if (st != MLA_OK) return st;
    }
    if (want_dw) {
        // 4. x [T, K] -> xt [K, Tp], blocks along T; 5. dW = qb . xt^T (reduction over T; the
        //    operands' extent is T, so the tensor maps read zeros past it)
        st = launch_mxfp8_quantize_cols_tiled_sf(T, K, MLA_IN_BF16, a.x, K, ws + L.xt, L.Tp, ws + L.xt_s, L.G,
                                                 stream);
        if (st != MLA_OK) return st;
        FwdArgs g{};
        g.T = N;
        g.K = T;
        g.H = 1;
        g.Dn = (int)K;
        g.Dr = 0;
        g.weight_mode = MLA_WEIGHT_MXFP8;
        g.out_mode = MLA_OUT_BF16;
        g.x = ws + L.qb;
        g.x_scales = ws + L.qb_s;
        g.W = ws + L.xt;
        g.w_scales = ws + L.xt_s;
        g.ld_x = L.Tp;
        g.ld_w = L.Tp;
        g.sf_tiled = 1;
        g.sf_group = (int)L.G;
        g.q_out = a.dW;
        g.status = a.status;
        st = launch_fwd(g, stream);
        if (st != MLA_OK) return st;
    }
    if (want_db) {
        db_reduce_kernel<<<grid_for(N, 256, cap), 256, 0, stream>>>(reinterpret_cast<float*>(ws + L.dbp),
                                                                   (T + 31) / 32, N, static_cast<uint16_t*>(a.db));
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

}  // namespace mlaq
