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

// One CTA: 32 tokens [t0, t0 + 32) x one head's D channels (D % 32 == 0),
// staged in shared memory as float32 with a row pitch of D + 1 words, so
// that row-wise and column-wise reads are both free of bank conflicts.
//   qa [T, N] / qa_s [T, N/32]: rowwise copy (nullable: skipped)
//   qb [N, ldq] / qb_s [N, ldq/32]: columnwise copy (nullable: skipped);
//     the CTA of the last token block also zeroes the scale bytes of the
//     token blocks in [ceil(T/32), ldq/32) (the padding the GEMM reads)
//   dbp [ceil(T/32), N]: per-block channel sums (nullable: skipped)
template <int DR>
__global__ void __launch_bounds__(kRqThreads) rope_bwd_quant_kernel(
    const uint16_t* __restrict__ dq, int64_t T, int H, int Dn, const float* __restrict__ cos_tab,
    const float* __restrict__ sin_tab, int64_t cs_rows, int64_t cs_width, const int32_t* __restrict__ pos,
    uint8_t* __restrict__ qa, uint8_t* __restrict__ qa_s, uint8_t* __restrict__ qb, uint8_t* __restrict__ qb_s,
    int64_t ldq, float* __restrict__ dbp, int* status) {
    extern __shared__ float tile[];
    constexpr int HH = DR / 2;
    const int D = Dn + DR;
    const int P = D + 1;  // row pitch (words)
    const int64_t N = (int64_t)H * D;
    const int64_t nbt = (T + 31) / 32;  // token blocks
    const int64_t tb = blockIdx.x % nbt;
    const int h = (int)(blockIdx.x / nbt);
    const int64_t t0 = tb * 32;
    const int tid = threadIdx.x;
    // load: 32 rows x D bf16, 8 per 16-byte vector; rows past T are zeros
    const int vpr = D / 8;
    for (int k = tid; k < 32 * vpr; k += kRqThreads) {
        const int r = k / vpr, v = k % vpr;
        const int64_t t = t0 + r;
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (t < T) raw = __ldg(reinterpret_cast<const uint4*>(dq + t * N + (int64_t)h * D + 8 * v));
        float* dst = tile + r * P + 8 * v;
        dst[0] = bf16lo_to_f32(raw.x);
        dst[1] = bf16hi_to_f32(raw.x);
        dst[2] = bf16lo_to_f32(raw.y);
        dst[3] = bf16hi_to_f32(raw.y);
        dst[4] = bf16lo_to_f32(raw.z);
        dst[5] = bf16hi_to_f32(raw.z);
        dst[6] = bf16lo_to_f32(raw.w);
        dst[7] = bf16hi_to_f32(raw.w);
    }
    __syncthreads();
    // inverse rotation of the rope channels (the transpose of the forward's
    // rotate-half pair), float32, each product and each sum rounded once:
    //   out[i]     = fl(fl(g[i] cos_i) + fl(g[i+h] sin_{i+h}))
    //   out[i + h] = fl(fl(g[i+h] cos_{i+h}) - fl(g[i] sin_i))
    for (int k = tid; k < 32 * HH; k += kRqThreads) {
        const int r = k / HH, i = k % HH;
        const int64_t t = t0 + r;
        if (t >= T) continue;
        const int64_t pp = pos ? (int64_t)__ldg(pos + t) : t;
        if (pp < 0 || pp >= cs_rows) {
            record_status(status, MLA_ERR_POS_RANGE);
            continue;
        }
        const float* cs = cos_tab + pp * cs_width;
        const float* sn = sin_tab + pp * cs_width;
        float* row = tile + r * P + Dn;
        const float a = row[i], c = row[i + HH];
        row[i] = __fadd_rn(__fmul_rn(a, __ldg(cs + i)), __fmul_rn(c, __ldg(sn + i + HH)));
        row[i + HH] = __fsub_rn(__fmul_rn(c, __ldg(cs + i + HH)), __fmul_rn(a, __ldg(sn + i)));
    }
    __syncthreads();
    // rowwise copy: blocks of 32 channels of one token; a thread takes one
    // (block, token) pair, the lanes of a warp 32 consecutive tokens
    if (qa) {
        const int nb = D / 32;
        for (int k = tid; k < 32 * nb; k += kRqThreads) {
            const int b = k / 32, r = k % 32;
            const int64_t t = t0 + r;
            if (t >= T) continue;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = tile[r * P + 32 * b + i];
            uint32_t w[8];
            const uint32_t sb = quantize_block_regs<32>(v, 32, w);
            uint8_t* dst = qa + t * N + (int64_t)h * D + 32 * b;
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
            qa_s[t * (N / 32) + ((int64_t)h * D) / 32 + b] = (uint8_t)sb;
        }
    }
    // columnwise copy (blocks of 32 tokens of one channel) and the db partial sums
    if (qb || dbp) {
        const int n = (T - t0) < 32 ? (int)(T - t0) : 32;
        const int64_t lds = ldq / 32;
        for (int c = tid; c < D; c += kRqThreads) {
            float v[32];
            float sum = 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                v[r] = tile[r * P + c];
                sum += v[r];  // in token order; rows past T are 0
            }
            const int64_t ch = (int64_t)h * D + c;
            if (qb) {
                uint32_t w[8];
                const uint32_t sb = quantize_block_regs<32>(v, n, w);
                uint8_t* dst = qb + ch * ldq + t0;
                if (n == 32) {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)  // unrolled: w stays in registers
                        if (j < n) dst[j] = (uint8_t)(w[j / 4] >> (8 * (j % 4)));
                }
                qb_s[ch * lds + tb] = (uint8_t)sb;
                if (tb == nbt - 1)
                    for (int64_t j = nbt; j < lds; ++j) qb_s[ch * lds + j] = 0;
            }
            if (dbp) dbp[tb * N + ch] = sum;
        }
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
    const int64_t Tp = (T + 127) / 128 * 128;
    const int64_t nbt = (T + 31) / 32;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L->Tp = Tp;
    L->qa = take((size_t)T * N);
    L->qa_s = take((size_t)T * (N / 32));
    L->qb = take((size_t)N * Tp);
    L->qb_s = take((size_t)N * (Tp / 32));
    L->wt = take((size_t)K * N);
    L->wt_s = take((size_t)K * (N / 32));
    L->xt = take((size_t)K * Tp);
    L->xt_s = take((size_t)K * (Tp / 32));
    L->dbp = take((size_t)nbt * N * sizeof(float));
    L->total = off;
    return MLA_OK;
}

int launch_rope_bwd_quant(const BwdArgs& a, uint8_t* qa, uint8_t* qa_s, uint8_t* qb, uint8_t* qb_s, int64_t ldq,
                          float* dbp, cudaStream_t stream) {
    const int D = a.Dn + a.Dr;
    const int64_t nbt = (a.T + 31) / 32;
    const size_t smem = (size_t)32 * (D + 1) * sizeof(float);
    const unsigned grid = (unsigned)(nbt * a.H);
    const uint16_t* dq = static_cast<const uint16_t*>(a.dq);
    const void* k = nullptr;
    switch (a.Dr) {
        case 16: k = (const void*)rope_bwd_quant_kernel<16>; break;
        case 32: k = (const void*)rope_bwd_quant_kernel<32>; break;
        case 64: k = (const void*)rope_bwd_quant_kernel<64>; break;
        default: return MLA_ERR_UNSUPPORTED;
    }
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MLA_ERR_CUDA;
#define MLAQ_RQ_LAUNCH(DRV)                                                                                   \
    rope_bwd_quant_kernel<DRV><<<grid, kRqThreads, smem, stream>>>(dq, a.T, a.H, a.Dn, a.cos_tab, a.sin_tab,   \
                                                                   a.cs_rows, a.cs_width, a.pos, qa, qa_s, qb, \
                                                                   qb_s, ldq, dbp, a.status)
    switch (a.Dr) {
        case 16: MLAQ_RQ_LAUNCH(16); break;
        case 32: MLAQ_RQ_LAUNCH(32); break;
        default: MLAQ_RQ_LAUNCH(64); break;
    }
#undef MLAQ_RQ_LAUNCH
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
    uint8_t* qa = want_dx ? ws + L.qa : nullptr;
    uint8_t* qb = want_dw ? ws + L.qb : nullptr;
    float* dbp = want_db ? reinterpret_cast<float*>(ws + L.dbp) : nullptr;
    // 1. rotate dq once; both MXFP8 copies of dq_pre and the db partials
    st = launch_rope_bwd_quant(a, qa, ws + L.qa_s, qb, ws + L.qb_s, L.Tp, dbp, stream);
    if (st != MLA_OK) return st;
    if (want_dx) {
        // 2. W [N, K] -> wt [K, N], blocks along N; 3. dx = qa . wt^T (reduction over N)
        st = launch_mxfp8_quantize_cols_ld(N, K, MLA_IN_BF16, a.W, K, ws + L.wt, N, ws + L.wt_s, N / 32, stream);
        if (st != MLA_OK) return st;
        FwdArgs g{};
        g.T = T;
        g.K = N;
        g.H = 1;
        g.Dn = (int)K;
        g.Dr = 0;
        g.weight_mode = MLA_WEIGHT_MXFP8;
        g.out_mode = MLA_OUT_BF16;
        g.x = qa;
        g.x_scales = ws + L.qa_s;
        g.W = ws + L.wt;
        g.w_scales = ws + L.wt_s;
        g.q_out = a.dx;
        g.status = a.status;
        st = launch_fwd(g, stream);
        if (st != MLA_OK) return st;
    }
    if (want_dw) {
        // 4. x [T, K] -> xt [K, Tp], blocks along T; 5. dW = qb . xt^T (reduction over T)
        uint8_t* xt_s = ws + L.xt_s;
        st = launch_mxfp8_quantize_cols_ld(T, K, MLA_IN_BF16, a.x, K, ws + L.xt, L.Tp, xt_s, L.Tp / 32, stream);
        if (st != MLA_OK) return st;
        const int64_t nbt = (T + 31) / 32;
        if (L.Tp / 32 > nbt &&
            cudaMemset2DAsync(xt_s + nbt, (size_t)(L.Tp / 32), 0, (size_t)(L.Tp / 32 - nbt), (size_t)K, stream) !=
                cudaSuccess)
            return MLA_ERR_CUDA;
        FwdArgs g{};
        g.T = N;
        g.K = T;
        g.H = 1;
        g.Dn = (int)K;
        g.Dr = 0;
        g.weight_mode = MLA_WEIGHT_MXFP8;
        g.out_mode = MLA_OUT_BF16;
        g.x = qb;
        g.x_scales = ws + L.qb_s;
        g.W = ws + L.xt;
        g.w_scales = xt_s;
        g.ld_x = L.Tp;
        g.ld_w = L.Tp;
        g.ld_scale = L.Tp / 32;
        g.q_out = a.dW;
        g.status = a.status;
        st = launch_fwd(g, stream);
        if (st != MLA_OK) return st;
    }
    if (want_db) {
        db_reduce_kernel<<<grid_for(N, 256, cap), 256, 0, stream>>>(dbp, (T + 31) / 32, N,
                                                                   static_cast<uint16_t*>(a.db));
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    }
    return MLA_OK;
}

}  // namespace mlaq
