// Fused MLA query up-projection forward on sm_103a tensor cores.
//
// TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
// description paragraph and flowchart: q = RoPE(x W^T + b), then MXFP8
// quantization, with a 16-bit or an MXFP8 projection weight. The pages name
// a cuDNN-frontend kernel for SM100; this is an independent design for
// sm_103a:
//
//   * persistent CTAs (one per SM), each walking a static list of
//     128-token x BN-channel output tiles (token index fastest, so the CTAs
//     running together share weight tiles in L2; with resident weight scales
//     each CTA takes one contiguous range of them instead);
//   * warp 0: TMA producer, filling an S-stage shared-memory ring with x and
//     W tiles (128-byte rows, 128-byte swizzle). For MXFP8 weights it also
//     brings the E8M0 scale bytes of both operands into the 32x16-byte
//     layout that tcgen05.cp replicates into TMEM: one 512-byte bulk copy
//     per 128-row chunk when the scales come pre-tiled, else a gather with
//     4-byte cp.async;
//   * warp 1: one thread issues tcgen05.mma (M=128, N=BN, K=16 bf16 or K=32
//     block-scaled E4M3) into a double-buffered fp32 TMEM accumulator and
//     commits each stage back to the producer;
//   * warps 2-9: epilogue, two per TMEM lane quadrant. Each thread owns one
//     token row of the tile (tcgen05.ld 32x32b) for half of its columns,
//     adds the bias, applies the rotate-half RoPE pair (i, i+Dr/2)
//     thread-locally, and converts to bf16 or MXFP8 (per-32-channel amax ->
//     E8M0 scale -> E4M3 codes). The values pass through shared-memory
//     staging slots and leave as TMA tile stores into a fresh output (one
//     store box per 32-channel block, or per 64 channels when the two warps
//     of a quadrant take the tile's two halves). The next tile's main loop
//     runs in the other accumulator buffer meanwhile;
//   * warp 10 (MXFP8 weights, pre-tiled scales): the scale bulk copies. With
//     resident weight scales (the RES variant) W's scale tiles come only on a
//     channel tile's first tile (kept in TMEM while the CTA stays on it) and
//     a tile's x scales in one copy into one of two buffers.
//
// The tile order, the resident scales and the half-tile store layout are
// compile-time variants: run-time checks of them in every role's loops
// measured slower.
//
// Tiles never split a rope region or an MXFP8 block (the host picks BN so).
// With Dr = 0 the kernel is a plain GEMM on 256-token tiles (two M = 128
// MMAs per K step into one accumulator pair), used by the MXFP8 backward.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstring>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kBM = 128;
// warp 0 TMA, warp 1 MMA, warps 2-9 epilogue, warp 10 the tiled-scale copies
// (MXFP8 weights). 11 warps keep three per SM sub-partition at most, so the
// per-thread register cap stays at 168.
constexpr int kThreads = 352;
constexpr int kSfWarp = 10;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;  // TMEM column offset of accumulator buffer 1
constexpr uint32_t kSfCol0 = 448;     // first TMEM column of the per-stage scale factors
constexpr uint32_t kSfColsPerStage = 12;  // 4 (A: 128 rows) + 8 (B: up to 256 rows)
constexpr uint32_t kSfBytesPerStage = 512 + 1024;
// The plain GEMM (DR = 0) takes 256-row x tiles: two M = 128 MMAs per K chunk
// into two accumulators (TMEM columns 0 and 256, not double-buffered), 30%
// fewer operand bytes per FLOP than one 128-row tile. Its stages carry the
// scales of two 128-row x chunks.
constexpr uint32_t kSfColsPerStage2 = 16;
constexpr uint32_t kSfBytesPerStage2 = 1024 + 1024;
constexpr int kEpiWarps = 8;  // two per TMEM lane quadrant, splitting the tile's units
// Output staging slot: one TMA store box of 32 token rows. bf16 output: 16
// channels (32 bytes a row); MXFP8 output: one 32-channel block (32 bytes a
// row), or 16 channels (16 bytes a row) when Dr = 16, whose rope part is a
// 16-channel block. The TMA unit of an SM handles a fixed number of tile
// operations per second whatever their size, so the number of q stores
// matters (hence also the 64-channel boxes of the half-tile split).
template <bool MXOUT, int DR>
__host__ __device__ constexpr int slot_ch() {
    return (MXOUT && DR % 32 == 0) ? 32 : 16;
}

struct FwdParams {
    int T, H, N, D, Dn;
    int BN;
    int num_m_tiles, num_tiles, k_tiles;
    int stages;
    uint32_t a_bytes, stage_bytes, tx_bytes;
    uint32_t idesc;
    int ksb;  // scale bytes per operand row (K / 32)
    uint32_t slot_bytes;  // room for one store box (32 rows x at most 32 bytes)
    int cs_vec;           // cos/sin rows 16-byte aligned: float4 loads
    int nslots;           // staging slots per epilogue warp
    int scales_bhsd;      // MXFP8 scales head-major [H, T, NB] (else [T, H, NB])
    int qs_swz;           // MXFP8 scales per head in the GEMM's tiled order
    int qs_row_tiles;     //   128-row tiles per head: ceil(T / 128)
    int qs_col_tiles;     //   4-column tiles: ceil(NB / 4)
    int sf_tiled;         // MXFP8 scales pre-tiled (sf_tiled_offset order): one 512-byte bulk
                          // copy per 128-row chunk and K step instead of the per-row gather
    int sf_nsub;          // 128-row chunks of a B tile: ceil(BN / 128)
    int num_n_tiles;
    uint32_t sf_stage;    // scale staging bytes per stage (MXFP8 weights)
    uint32_t sf_cols;     // TMEM scale-factor columns per stage
    int sfb_res;          // (tiled MXFP8 scales, 128-row tiles; launches the RES variant, whose
                          // CTAs take contiguous tile ranges) the weight scales of the
                          // current channel tile stay in TMEM: copied in on the CTA's first
                          // tile of that channel tile only, K step kt at column sfb_col(kt)
    int sfb_n1;           //   K steps held in the columns [BN, 256) between the accumulators
    int sfb_col2;         //   first column for the K steps after those (after the x scales)
                          //   With sfb_res the x scales of a tile come in one bulk copy (all
                          //   its K steps, contiguous in the tiled order) into one of two
                          //   shared-memory buffers, so that a stage is two TMA operations.
    int half_store;       // (with split_half, MXFP8 q) 64-channel store boxes, two per half tile
    int split_half;       // the two warps of a lane quadrant take the tile's two halves and
                          // write each row's scale bytes as one 4-byte word (else: units
                          // alternate between them and scales go byte by byte)
    const uint16_t* bias;
    const float* cos_tab;
    const float* sin_tab;
    // the packed table (mla_rope_table_pack): float4 (cos_i, sin_i,
    // cos_{i+Dr/2}, sin_{i+Dr/2}) of position p at tab4[i * cs_rows + p];
    // used instead of cos_tab/sin_tab when not null
    const float4* tab4;
    const int32_t* pos;
    long long cs_rows, cs_width;
    uint8_t* q_out;
    uint8_t* q_scales;
    const uint8_t* x_scales;
    const uint8_t* w_scales;
    int* status;
    // KV side: a tile is one head's [k_nope (Dn) | v (Dv)] columns
    int Dv;
    int tiles_per_cta;
    uint16_t* o_key;        // [T, H, Dn + Dr] bf16
    uint16_t* o_value;      // [T, H, Dv] bf16
    const uint16_t* k_pe;   // [T, Dr] bf16, shared by the heads
};

struct Smem {
    uint32_t base;      // shared address of stage 0 (1024-aligned)
    uint32_t sf;        // scale staging (MXFP8 weights)
    uint32_t sfx;       // (sfb_res) the two x-scale tile buffers, k_tiles * 512 bytes each
    uint32_t out;       // output staging: kEpiWarps x nslots slots
    uint32_t bars;      // mbarriers
    int S;
    __device__ uint32_t a(int s, const FwdParams& p) const { return base + (uint32_t)s * p.stage_bytes; }
    __device__ uint32_t b(int s, const FwdParams& p) const { return a(s, p) + p.a_bytes; }
    uint32_t sf_stage, sfb_off;
    __device__ uint32_t sfa(int s) const { return sf + (uint32_t)s * sf_stage; }
    __device__ uint32_t sfb(int s) const { return sfa(s) + sfb_off; }
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t empty(int s) const { return bars + 8u * (S + s); }
    __device__ uint32_t tfull(int b) const { return bars + 8u * (2 * S + b); }
    __device__ uint32_t tempty(int b) const { return bars + 8u * (2 * S + 2 + b); }
    __device__ uint32_t drain() const { return bars + 8u * (2 * S + 4); }
    __device__ uint32_t xfull(int b) const { return bars + 8u * (2 * S + 5 + b); }
    __device__ uint32_t xempty(int b) const { return bars + 8u * (2 * S + 7 + b); }
};

// ------------------------------------------------------------ epilogue parts
// Each epilogue warp owns 32 token rows of the tile. Its results go through a
// ring of p.nslots shared-memory slots (one store box each) and leave
// as TMA tile stores (one per slot), so global writes are whole, coalesced
// boxes and the LSU queue carries no per-row stores.
struct EpiCtx {
    uint32_t slots;   // this warp's staging ring
    const uint16_t* bias;  // the tile's bias (bf16, 16-byte aligned rows of 8), or null
    int cursor;       // next free slot (counts pieces; taken modulo nslots)
    int prev_pieces;  // pieces of the previous unit (its store may still read)
    int prev2_pieces; // pieces of the unit before it
    int32_t t0;       // first token row of this warp's 32-row slab
    uint32_t sword;   // packed scale bytes of this row's half tile (split_half)
    int64_t sbase;    // first 32-channel block index of that half
    int32_t hcol0;    // (half_store) first channel of this warp's half tile
    const CUtensorMap* tmh;  // (half_store) q as 64-channel x 32-token boxes, 64-byte swizzle
};

__device__ __forceinline__ uint32_t slot_addr(const FwdParams& p, const EpiCtx& c, int k) {
    return c.slots + (uint32_t)(k % p.nslots) * p.slot_bytes;
}

__device__ __forceinline__ void add_bias(float* v, int nv, const uint16_t* bias) {
    for (int k = 0; k < nv / 8; ++k) {
        const uint4 b = __ldg(reinterpret_cast<const uint4*>(bias) + k);  // same address in every lane
        v[8 * k + 0] += bf16lo_to_f32(b.x);
        v[8 * k + 1] += bf16hi_to_f32(b.x);
        v[8 * k + 2] += bf16lo_to_f32(b.y);
        v[8 * k + 3] += bf16hi_to_f32(b.y);
        v[8 * k + 4] += bf16lo_to_f32(b.z);
        v[8 * k + 5] += bf16hi_to_f32(b.z);
        v[8 * k + 6] += bf16lo_to_f32(b.w);
        v[8 * k + 7] += bf16hi_to_f32(b.w);
    }
}

// Quantize/convert this thread's NV values (output channels [n, n + NV) of
// token t, i.e. channels [cin, cin + NV) of head h) into the staging ring and
// store them with TMA, one store per CH channels. NV is a multiple of CH.
// A lane's 32-byte row of a slot is written as two 16-byte halves, lanes
// with bit 2 set upper half first, so each store instruction of the warp
// takes the minimum four shared-memory wavefronts.
// HS: the 64-channel half-tile store boxes (p.half_store), fixed at compile
// time: the kernel variant launched exactly when p.half_store is set.
template <bool MXOUT, int NV, int CH, bool HS = false>
__device__ __forceinline__ void emit_unit(const FwdParams& p, const CUtensorMap* tmC, EpiCtx& c,
                                          const float (&v)[NV], bool valid, int64_t t, int64_t n, int h,
                                          int cin) {
    static_assert(NV % CH == 0 && (CH == 16 || (MXOUT && CH == 32)), "slot width");
    constexpr int PIECES = NV / CH;
    const int lane = threadIdx.x & 31;
    const uint32_t h0 = (lane & 4) ? 16u : 0u, h1 = 16u - h0;  // byte offsets of the two halves, in store order
    if constexpr (MXOUT && CH == 32 && HS) {
        {
            // A warp's half tile (128 channels, in column order) leaves in two
            // 64-channel store boxes: two 2 KB slots, rows 64 bytes apart in
            // the 64-byte swizzled order of the store's tensor map (16-byte
            // chunk k of row r at position k ^ ((r / 2) % 4)), so each store
            // instruction takes the minimum four wavefronts. A slot is reused
            // once the store before the previous one has read it.
#pragma unroll
            for (int blk = 0; blk < NV / 32; ++blk) {
                float b[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) b[i] = v[blk * 32 + i];
                uint32_t codes[8];
                const uint32_t sb = quantize_block_regs<32>(b, 32, codes);
                const int co = (int)n + 32 * blk - c.hcol0;  // 0, 32, 64 or 96
                const uint32_t slot = c.slots + (uint32_t)(co / 64) * 2048u;
                if ((co & 63) == 0) {
                    if (lane == 0) bulk_wait_group_read<1>();
                    __syncwarp();
                }
                const uint32_t k0 = (uint32_t)(co & 63) / 16u, sw = ((uint32_t)lane >> 1) & 3u;
                const uint32_t row = slot + 64u * lane;
                sts_v4(row + ((k0 ^ sw) << 4), codes[0], codes[1], codes[2], codes[3]);
                sts_v4(row + (((k0 + 1u) ^ sw) << 4), codes[4], codes[5], codes[6], codes[7]);
                c.sword |= sb << (8 * (int)((n + 32 * blk) / 32 - c.sbase));
                if ((co & 63) == 32) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d_hint(c.tmh, c.hcol0 + (co & ~63), c.t0, slot, l2_evict_first_policy());
                        bulk_commit_group();
                    }
                }
            }
            return;
        }
    }
    // the slots about to be written were last read by stores older than the previous unit's
    if (lane == 0) {
        // the stores of the last two units may still read their slots when those
        // and this unit's fit in the ring together (ring positions never overlap)
        if (c.prev2_pieces + c.prev_pieces + PIECES <= p.nslots) bulk_wait_group_read<2>();
        else if (c.prev_pieces + PIECES <= p.nslots) bulk_wait_group_read<1>();
        else bulk_wait_group_read<0>();
    }
    __syncwarp();
    const int first = c.cursor;
    if (MXOUT) {
        const int NB = (p.D + 31) / 32;
#pragma unroll
        for (int blk = 0; blk < (NV + 31) / 32; ++blk) {
            float b[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) b[i] = (blk * 32 + i < NV) ? v[blk * 32 + i] : 0.f;
            const int nvalid = (NV - blk * 32) < 32 ? (NV - blk * 32) : 32;
            uint32_t codes[8];
            const uint32_t sb = quantize_block_regs<32>(b, nvalid, codes);
            if (CH == 32) {
                // the block's 32 codes: one 32-byte slot row
                const uint32_t a = slot_addr(p, c, first + blk) + 32u * lane;
                const uint32_t* q0 = (lane & 4) ? codes + 4 : codes;
                const uint32_t* q1 = (lane & 4) ? codes : codes + 4;
                sts_v4(a + h0, q0[0], q0[1], q0[2], q0[3]);
                sts_v4(a + h1, q1[0], q1[1], q1[2], q1[3]);
            } else {
                // 16-channel slots (a 16 x 32 box: rows 16 bytes apart), two per block
                sts_v4(slot_addr(p, c, first + 2 * blk) + 16u * lane, codes[0], codes[1], codes[2], codes[3]);
                if (nvalid > 16)
                    sts_v4(slot_addr(p, c, first + 2 * blk + 1) + 16u * lane, codes[4], codes[5], codes[6],
                           codes[7]);
            }
            if (p.split_half) {
                c.sword |= sb << (8 * (int)((n + 32 * blk) / 32 - c.sbase));
            } else if (p.qs_swz) {
                // head h's [T, NB] scales in the GEMM's tiled order: 128-row x
                // 4-column tiles of 512 bytes. Rows t >= T of the last row tile
                // (these threads exist: token tiles are 128 rows) and the
                // columns past NB are padding, written as 0.
                const int bc = (cin + blk * 32) / 32;
                const int64_t rt = ((int64_t)h * p.qs_row_tiles + t / 128) * p.qs_col_tiles;
                const uint32_t rr = (uint32_t)(t % 32) * 16u + (uint32_t)((t % 128) / 32) * 4u;
                p.q_scales[(rt + bc / 4) * 512 + rr + bc % 4] = valid ? (uint8_t)sb : (uint8_t)0;
                if (bc == NB - 1)
                    for (int pc = NB; pc < 4 * p.qs_col_tiles; ++pc) p.q_scales[(rt + pc / 4) * 512 + rr + pc % 4] = 0;
            } else if (valid)
                p.q_scales[(p.scales_bhsd ? (int64_t)h * p.T + t : t * p.H + h) * NB + (cin + blk * 32) / 32] =
                    (uint8_t)sb;
        }
    } else {
#pragma unroll
        for (int pc = 0; pc < PIECES; ++pc) {
            const uint32_t a = slot_addr(p, c, first + pc) + 32u * lane;
            const float* w = v + 16 * pc;
            const float* w0 = (lane & 4) ? w + 8 : w;
            const float* w1 = (lane & 4) ? w : w + 8;
            sts_v4(a + h0, pack_bf16x2(w0[0], w0[1]), pack_bf16x2(w0[2], w0[3]), pack_bf16x2(w0[4], w0[5]),
                   pack_bf16x2(w0[6], w0[7]));
            sts_v4(a + h1, pack_bf16x2(w1[0], w1[1]), pack_bf16x2(w1[2], w1[3]), pack_bf16x2(w1[4], w1[5]),
                   pack_bf16x2(w1[6], w1[7]));
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        const uint64_t pol = l2_evict_first_policy();  // q is written once: do not let it push x, W out of L2
#pragma unroll
        for (int pc = 0; pc < PIECES; ++pc)
            tma_store_2d_hint(tmC, (int32_t)(n + CH * pc), c.t0, slot_addr(p, c, first + pc), pol);
        bulk_commit_group();
    }
    c.cursor = first + PIECES;
    c.prev2_pieces = c.prev_pieces;
    c.prev_pieces = PIECES;
}

template <bool MXOUT, int CH, bool HS = false>
__device__ __forceinline__ void nope_unit(const FwdParams& p, const CUtensorMap* tmC, EpiCtx& c,
                                          uint32_t taddr, int col, bool valid, int64_t t, int64_t n, int h,
                                          int cin) {
    uint32_t r[32];
    __syncwarp();  // tcgen05.ld is .sync.aligned: the whole warp, converged
    tmem_ld32(taddr, r);
    tmem_ld_wait();
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
    if (c.bias) add_bias(v, 32, c.bias + col);
    emit_unit<MXOUT, 32, CH, HS>(p, tmC, c, v, valid, t, n, h, cin);
}

__device__ __forceinline__ void load_table8(const float* src, bool vec, float (&o)[8]) {
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

// The rotate-half pair (a, b) = (y[i], y[i + Dr/2]) of position p, with one
// rounding order for both table layouts: the second product is rounded,
// then the first is added by one fused multiply-add.
__device__ __forceinline__ void rot_pair_fwd(float& a, float& b, float ci, float si, float cj, float sj) {
    const float a0 = a, b0 = b;
    a = __fmaf_rn(a0, ci, -__fmul_rn(b0, si));  // a cos_i - b sin_i
    b = __fmaf_rn(b0, cj, __fmul_rn(a0, sj));   // b cos_{i+h} + a sin_{i+h}
}

// part < 0: this warp emits the whole rope unit; part 0 / 1 (DR = 64): the
// quadrant's two warps both rotate it and each emits one 32-channel half.
template <bool MXOUT, int DR, bool PACKED, bool HS = false>
__device__ __forceinline__ void rope_unit(const FwdParams& p, const CUtensorMap* tmC, EpiCtx& c,
                                          uint32_t taddr, int col, bool valid, int64_t t, int64_t n, int h,
                                          int prow, int part) {
    constexpr int HH = DR / 2;
    uint32_t r[DR / 16][16];
    __syncwarp();
#pragma unroll
    for (int j = 0; j < DR / 16; ++j) tmem_ld16(taddr + 16 * j, r[j]);
    tmem_ld_wait();
    float y[DR];
#pragma unroll
    for (int i = 0; i < DR; ++i) y[i] = __uint_as_float(r[i / 16][i % 16]);
    if (c.bias) add_bias(y, DR, c.bias + col);
    if constexpr (PACKED) {
        // packed table: one 16-byte load per pair; the lanes of a warp (tokens
        // with consecutive positions) read consecutive 16-byte entries
        const float4* tp = p.tab4 + prow;
        const int64_t stride = p.cs_rows;
#pragma unroll
        for (int q = 0; q < HH; q += 4) {
            float4 tv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                tv[e] = __ldg(tp);
                tp += stride;
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) rot_pair_fwd(y[q + e], y[q + e + HH], tv[e].x, tv[e].y, tv[e].z, tv[e].w);
        }
    } else {
        const float* cs = p.cos_tab + (int64_t)prow * p.cs_width;
        const float* sn = p.sin_tab + (int64_t)prow * p.cs_width;
        const bool vec = p.cs_vec != 0;
        // rotate in place, 8 pairs at a time: (a, c) = (y[i], y[i + HH])
#pragma unroll
        for (int q = 0; q < HH; q += 8) {
            float ci[8], si[8], cj[8], sj[8];
            load_table8(cs + q, vec, ci);
            load_table8(sn + q, vec, si);
            load_table8(cs + q + HH, vec, cj);
            load_table8(sn + q + HH, vec, sj);
#pragma unroll
            for (int e = 0; e < 8; ++e) rot_pair_fwd(y[q + e], y[q + e + HH], ci[e], si[e], cj[e], sj[e]);
        }
    }
    if (DR == 64 && part >= 0) {
        float yb[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) yb[i] = part ? y[(32 + i) % DR] : y[i];
        emit_unit<MXOUT, 32, slot_ch<MXOUT, DR>(), HS>(p, tmC, c, yb, valid, t, n + 32 * part, h, p.Dn + 32 * part);
    } else {
        emit_unit<MXOUT, DR, slot_ch<MXOUT, DR>(), HS>(p, tmC, c, y, valid, t, n, h, p.Dn);
    }
}

// Tile order: tiles are strided over the CTAs, so the CTAs running together
// take consecutive tiles. The query side numbers them token tile fastest,
// the KV side (kv_tile) the same: the tiles of a wave share a few heads'
// rows of W, which stay in L2 while the outputs stream past. With resident
// weight scales (sfb_res) each CTA instead takes one contiguous range of
// tiles, so that it keeps a channel tile for up to num_m_tiles tiles in a
// row (W and x then sit in L2 whole: the range order costs no DRAM reads).
// (CONTIG, a compile-time choice: the ranges come with resident weight scales)
template <bool KV, bool CONTIG>
__device__ __forceinline__ int tile_first(const FwdParams& p) {
    return CONTIG ? (int)((int64_t)blockIdx.x * p.num_tiles / gridDim.x) : (int)blockIdx.x;
}
template <bool KV, bool CONTIG>
__device__ __forceinline__ int tile_end(const FwdParams& p) {
    return CONTIG ? (int)((int64_t)(blockIdx.x + 1) * p.num_tiles / gridDim.x) : p.num_tiles;
}
template <bool KV, bool CONTIG>
__device__ __forceinline__ int tile_next(const FwdParams&, int tile) {
    return tile + (CONTIG ? 1 : (int)gridDim.x);
}
// KV tile -> (token tile, head)
__device__ __forceinline__ void kv_tile(const FwdParams& p, int tile, int& mt, int& h) {
    h = tile / p.num_m_tiles;
    mt = tile - h * p.num_m_tiles;
}
// (token tile, channel tile) of query-side tile index g. The rope forward
// runs the token tile fastest (CTAs running together share W tiles); the
// plain GEMM (DR = 0) the channel tile, so they share the x row-tile (there x
// is the large, streamed operand).
template <int DR>
__device__ __forceinline__ void q_tile(const FwdParams& p, int g, int& mt, int& nt) {
    if (DR == 0) {
        mt = g / p.num_n_tiles;
        nt = g % p.num_n_tiles;
    } else {
        mt = g % p.num_m_tiles;
        nt = g / p.num_m_tiles;
    }
}

// ------------------------------------------------------------------- kernel
template <bool MXW, bool MXOUT, int DR, bool KV = false, bool PACKED = false, bool RES = false,
          bool HALF = false>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
               const FwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    constexpr bool M2 = DR == 0 && !KV;  // 256-row tiles, two accumulators
    // resident weight scales (the host's sfb_res), with contiguous tile ranges
    // and per-tile x scales: a compile-time variant
    constexpr bool RESC = RES && MXW && !KV && !M2;
    // the half-tile split with 64-channel store boxes (p.split_half and
    // p.half_store set): a compile-time variant as well
    constexpr bool HS = HALF && !MXW && MXOUT && !KV && DR == 64;
    constexpr int BM = M2 ? 2 * kBM : kBM;
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.S = p.stages;
    sm.base = (raw + 1023u) & ~1023u;
    sm.sf = sm.base + (uint32_t)p.stages * p.stage_bytes;
    sm.sf_stage = p.sf_stage;
    sm.sfb_off = M2 ? 1024u : (RESC ? 0u : 512u);  // resident mode: stages stage only W's scales
    sm.sfx = sm.sf + (MXW ? (uint32_t)p.stages * p.sf_stage : 0u);
    sm.out = sm.sfx + (RESC ? 2u * 512u * (uint32_t)p.k_tiles : 0u);
    sm.bars = sm.out + (uint32_t)(kEpiWarps * p.nslots) * p.slot_bytes;
    uint8_t* tail = smem_raw + (sm.bars - raw) + 8u * (2 * p.stages + 9);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(tail);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(sm.full(s), (MXW && !p.sf_tiled) ? 1 + 32 : 1);
            mbar_init(sm.empty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.tfull(b), 1);
            mbar_init(sm.tempty(b), kEpiWarps);
        }
        mbar_init(sm.drain(), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.xfull(b), 1);
            mbar_init(sm.xempty(b), 1);
        }
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32((const void*)tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int s = 0;
        uint32_t ph = 0;
        uint32_t issued_mask = 0, issued_par = 0;
        bool ok = true;
        // x's row tiles are re-read for every channel tile (keep them in L2),
        // except in the plain GEMM, whose large A operand streams through once
        const uint64_t a_pol = (DR == 0 && !KV) ? l2_evict_first_policy() : l2_evict_last_policy();
        int prev_nt = -1;
        for (int tile = tile_first<KV, RESC>(p); ok && tile < tile_end<KV, RESC>(p); tile = tile_next<KV, RESC>(p, tile)) {
            int mt, nt;
            if (KV) {
                kv_tile(p, tile, mt, nt);
            } else {
                q_tile<DR>(p, tile, mt, nt);
            }
            const bool a_hi = (int64_t)mt * BM + kBM < p.T;
            // resident weight scales: none to load while the channel tile stays
            const bool sfb_keep = RESC && nt == prev_nt;
            prev_nt = nt;
            const uint32_t tx = p.tx_bytes - ((M2 && MXW && p.sf_tiled && !a_hi) ? 512u : 0u);
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    // resident weight scales: the weight-scale bytes on a channel tile's first
                    // tile only; the x scales come on their own barrier
                    mbar_arrive_expect_tx(
                        sm.full(s), RESC ? p.stage_bytes + (sfb_keep ? 0u : 512u * (uint32_t)p.sf_nsub)
                                                       : tx);
                    // x / W tiles: inner coordinate is the K element index
                    const int kc = kt * (MXW ? 128 : 64);
                    tma_load_2d_hint(sm.a(s, p), &tmA, kc, mt * BM, sm.full(s), a_pol);
                    tma_load_2d(sm.b(s, p), &tmB, kc, nt * p.BN, sm.full(s));
                    // (the tiled scales: warp kSfWarp, on the same stage barrier)
                }
                if (MXW && !p.sf_tiled) {
                    // scale bytes [4 kt, 4 kt + 4) of each row; row r of a 128-row
                    // chunk goes to byte (r % 32) * 16 + (r / 32) * 4.
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int r = lane + 32 * j;
                        const int64_t row = (int64_t)mt * BM + r;
                        if (row < p.T)
                            cp_async_4(sm.sfa(s) + lane * 16 + j * 4,
                                       p.x_scales + row * p.ksb + kt * 4);
                    }
                    for (int j = 0; j < p.BN / 32; ++j) {
                        const int r = lane + 32 * j;
                        const int64_t row = (int64_t)nt * p.BN + r;
                        cp_async_4(sm.sfb(s) + (r / 128) * 512 + lane * 16 + ((r % 128) / 32) * 4,
                                   p.w_scales + row * p.ksb + kt * 4);
                    }
                    cp_async_mbar_arrive_noinc(sm.full(s));
                }
                issued_mask |= 1u << s;
                issued_par = (issued_par & ~(1u << s)) | (ph << s);
                if (++s == p.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok) {
            // unwinding: let every copy this warp started land before the CTA exits
            for (int q = 0; q < p.stages; ++q)
                if (issued_mask & (1u << q))
                    mbar_wait(sm.full(q), (issued_par >> q) & 1u, nullptr, 200000000ull);
        }
    } else if (warp == kSfWarp) {
        // -------------------------------------------- tiled-scale producer
        // The stage's E8M0 scale tiles (one 512-byte bulk copy per 128-row
        // chunk of each operand), issued by a second thread so that warp 0
        // issues only the two operand tiles per stage. The copies complete
        // on the stage's full barrier, whose expected bytes warp 0 posts.
        // With resident weight scales, W's scale tiles come on a channel
        // tile's first tile only, and the x scales of a whole tile in one
        // bulk copy into x-scale buffer (local tile & 1), on its own barrier.
        if (MXW && p.sf_tiled && lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued_mask = 0, issued_par = 0;
            uint32_t x_issued = 0, x_par = 0;
            bool ok = true;
            int prev_nt = -1, local = 0;
            const uint32_t xbytes = 512u * (uint32_t)p.k_tiles;
            for (int tile = tile_first<KV, RESC>(p); ok && tile < tile_end<KV, RESC>(p); tile = tile_next<KV, RESC>(p, tile), ++local) {
                int mt, nt;
                q_tile<DR>(p, tile, mt, nt);
                const bool a_hi = (int64_t)mt * BM + kBM < p.T;
                const bool sfb_keep = RESC && nt == prev_nt;  // (same rule as warp 0)
                prev_nt = nt;
                if (RESC) {
                    const int xb = local & 1;
                    const uint32_t xu = (uint32_t)(local >> 1);
                    if (!mbar_wait(sm.xempty(xb), (xu & 1u) ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(sm.xfull(xb), xbytes);
                    bulk_load(sm.sfx + (uint32_t)xb * xbytes, p.x_scales + (int64_t)mt * p.k_tiles * 512, xbytes,
                              sm.xfull(xb));
                    x_issued |= 1u << xb;
                    x_par = (x_par & ~(1u << xb)) | ((xu & 1u) << xb);
                }
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (!RESC)
                        bulk_load(sm.sfa(s), p.x_scales + ((int64_t)(M2 ? 2 * mt : mt) * p.k_tiles + kt) * 512,
                                  512u, sm.full(s));
                    if (M2 && a_hi)  // the second 128-row chunk, when it holds rows below T
                        bulk_load(sm.sfa(s) + 512u, p.x_scales + ((int64_t)(2 * mt + 1) * p.k_tiles + kt) * 512, 512u,
                                  sm.full(s));
                    for (int c = 0; c < (sfb_keep ? 0 : p.sf_nsub); ++c)
                        bulk_load(sm.sfb(s) + 512u * c,
                                  p.w_scales + (((int64_t)nt * p.sf_nsub + c) * p.k_tiles + kt) * 512, 512u,
                                  sm.full(s));
                    issued_mask |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // unwinding: let every copy this thread started land before the CTA exits
                for (int q = 0; q < p.stages; ++q)
                    if (issued_mask & (1u << q))
                        mbar_wait(sm.full(q), (issued_par >> q) & 1u, nullptr, 200000000ull);
                for (int q = 0; q < 2; ++q)
                    if (x_issued & (1u << q)) mbar_wait(sm.xfull(q), (x_par >> q) & 1u, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        // One thread issues every tcgen05 op of the CTA, and its own instruction
        // count per K step shows in the tensor pipe's idle time (the pipe runs
        // only a few ops ahead of it): the shared-memory descriptors are built
        // once and advanced by adding to their start-address field (address / 16,
        // 14 bits: shared addresses stay below 2^18, so the field never carries).
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            bool ok = true;
            int prev_nt = -1;
            const uint64_t da0 = desc_kmajor_sw128(sm.a(0, p)), db0 = desc_kmajor_sw128(sm.b(0, p));
            const uint64_t ds0 = smem_desc(sm.sfa(0), 0, 128, kLayoutNone);
            const uint64_t dop = p.stage_bytes >> 4, dsf = p.sf_stage >> 4, dsfb = sm.sfb_off >> 4;
            uint64_t da = da0, db = db0, ds = ds0;  // stage s's A, B and scale descriptors
            const uint32_t idesc = p.idesc;
            const int nsub = (p.BN + 127) / 128;
            const uint32_t xbytes = 512u * (uint32_t)p.k_tiles;
            for (int tile = tile_first<KV, RESC>(p); ok && tile < tile_end<KV, RESC>(p); tile = tile_next<KV, RESC>(p, tile), ++local) {
                const int b = M2 ? 0 : (local & 1);
                const uint32_t use = M2 ? (uint32_t)local : (uint32_t)(local >> 1);
                // Resident weight scales: copied into TMEM on the first tile of a
                // channel tile only. A K step's columns are next rewritten k_tiles
                // >= stages steps later, after the full barrier of that step, which
                // follows the empty-barrier commit of every MMA that read them.
                bool sfb_keep = false;
                if (RESC) {
                    int mt_r, nt_r;
                    q_tile<DR>(p, tile, mt_r, nt_r);
                    sfb_keep = nt_r == prev_nt;
                    prev_nt = nt_r;
                }
                if (!mbar_wait(sm.tempty(b), (use & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                // resident weight scales: the tile's x scales, one buffer of K steps
                const int xb = local & 1;
                uint64_t dsx = 0;
                if (RESC) {
                    if (!mbar_wait(sm.xfull(xb), (uint32_t)(local >> 1) & 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    dsx = smem_desc(sm.sfx + (uint32_t)xb * xbytes, 0, 128, kLayoutNone);
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)b * kAccStride;
                uint32_t sfb_res_col = tmem_base + (uint32_t)p.BN;  // K step kt's weight-scale columns
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!mbar_wait(sm.full(s), ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if constexpr (M2) {
                        // 256-row tiles (the plain GEMM): this per-step sequence measured
                        // faster here than the prebuilt-descriptor one below (0.892 against
                        // 0.916 ms for the MXFP8 backward at T = 8192)
                        const uint32_t a0 = sm.a(s, p), b0 = sm.b(s, p);
                        if (MXW) {
                            if (!p.sf_tiled) fence_proxy_async_smem();
                            const uint32_t sfa_col = tmem_base + kSfCol0 + p.sf_cols * s;
                            const uint32_t sfb_col = sfa_col + 8u;
                            tmem_cp_32x128b_warpx4(sfa_col, smem_desc(sm.sfa(s), 0, 128, kLayoutNone));
                            tmem_cp_32x128b_warpx4(sfa_col + 4, smem_desc(sm.sfa(s) + 512, 0, 128, kLayoutNone));
                            for (int c = 0; c < (p.BN + 127) / 128; ++c)
                                tmem_cp_32x128b_warpx4(sfb_col + 4 * c,
                                                       smem_desc(sm.sfb(s) + 512 * c, 0, 128, kLayoutNone));
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint32_t id = p.idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29);
#pragma unroll
                                for (int hm = 0; hm < 2; ++hm)
                                    mma_mxf8(d_tmem + hm * kAccStride, desc_kmajor_sw128(a0 + hm * 16384u + 32 * j),
                                             desc_kmajor_sw128(b0 + 32 * j), id, sfa_col + 4 * hm, sfb_col,
                                             (kt | j) != 0);
                            }
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
#pragma unroll
                                for (int hm = 0; hm < 2; ++hm)
                                    mma_bf16(d_tmem + hm * kAccStride, desc_kmajor_sw128(a0 + hm * 16384u + 32 * j),
                                             desc_kmajor_sw128(b0 + 32 * j), p.idesc, (kt | j) != 0);
                        }
                        mma_commit(sm.empty(s));
                        if (++s == p.stages) {
                            s = 0;
                            ph ^= 1u;
                        }
                        continue;
                    }
                    if (MXW) {
                        if (!p.sf_tiled) fence_proxy_async_smem();  // gathered bytes came through the generic proxy
                        const uint32_t sfa_col = tmem_base + kSfCol0 + p.sf_cols * s;
                        const uint32_t sfb_col = RESC ? sfb_res_col : sfa_col + 4u;
                        tmem_cp_32x128b_warpx4(sfa_col, RESC ? dsx : ds);
                        for (int c = 0; c < (sfb_keep ? 0 : nsub); ++c)
                            tmem_cp_32x128b_warpx4(sfb_col + 4u * c, ds + dsfb + 32u * (uint32_t)c);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t id = idesc | ((uint32_t)j << 4) | ((uint32_t)j << 29);
                            mma_mxf8(d_tmem, da + 2u * j, db + 2u * j, id, sfa_col, sfb_col, (kt | j) != 0);
                        }
                        dsx += 32u;  // the next K step's 512 bytes
                        sfb_res_col = kt + 1 == p.sfb_n1 ? tmem_base + (uint32_t)p.sfb_col2 : sfb_res_col + 8u;
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            mma_bf16(d_tmem, da + 2u * j, db + 2u * j, idesc, (kt | j) != 0);
                    }
                    mma_commit(sm.empty(s));
                    const bool wrap = s + 1 == p.stages;
                    s = wrap ? 0 : s + 1;
                    ph ^= wrap ? 1u : 0u;
                    da = wrap ? da0 : da + dop;
                    db = wrap ? db0 : db + dop;
                    ds = wrap ? ds0 : ds + dsf;
                }
                if (ok) {
                    mma_commit(sm.tfull(b));
                    if (RESC) mma_commit(sm.xempty(xb));  // the x-scale buffer is read
                }
            }
            if (!ok) {
                // unwinding: wait (bounded) for the MMAs already issued
                mma_commit(sm.drain());
                mbar_wait(sm.drain(), 0, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if constexpr (KV) {
        // ------------------------------------------------- KV-side epilogue
        // A tile = 128 tokens x one head's Dn + Dv columns; the quadrant's two
        // warps take alternate 32-column units (k_nope -> o_key, v -> o_value),
        // staged in a 2-slot ring and written by TMA. The shared key's rope
        // part was rotated once per token by kv_rope_pre_kernel into head 0's
        // rope slot; each tile of another head copies it from there (through
        // a shared-memory slab, each warp one half of the channels when
        // DR = 64) into its own.
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int ew = warp - 2;
        const int half = ew >> 2;
        const int Dk = p.Dn + DR;
        const uint32_t ring = sm.out + (uint32_t)(ew * 3) * 2048u;  // slots 0, 1; rope slab 2
        const uint32_t slab = ring + 2u * 2048u;
        int slot = 0, cur_mt = -1;
        int local = 0;
        for (int tile = tile_first<KV, RESC>(p); tile < tile_end<KV, RESC>(p); tile = tile_next<KV, RESC>(p, tile), ++local) {
            const int b = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            int mt, h;
            kv_tile(p, tile, mt, h);
            const int64_t t = (int64_t)mt * kBM + row;
            const bool valid = t < p.T;
            const int t0 = mt * kBM + quad * 32;
            if (h != 0 && mt != cur_mt && (DR == 64 || half == 0)) {
                // this warp's rope channels of the token block: [32 half, +32)
                // when DR = 64, else all of them in warp 0 (DR <= 32)
                if (lane == 0) bulk_wait_group_read<0>();  // stores still reading the slab
                __syncwarp();
                constexpr int NO = DR == 64 ? 32 : DR;  // channels this warp copies
                const int o0 = DR == 64 ? 32 * half : 0;
                const uint32_t ra = slab + (uint32_t)lane * (uint32_t)(NO * 2);
                const uint16_t* src = p.o_key + t * ((int64_t)p.H * Dk) + p.Dn + o0;  // head 0
#pragma unroll
                for (int q = 0; q < NO; q += 8) {
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (valid) v = __ldcg(reinterpret_cast<const uint4*>(src + q));
                    sts_v4(ra + (uint32_t)(2 * q), v.x, v.y, v.z, v.w);
                }
                fence_proxy_async_smem();
                __syncwarp();
                cur_mt = mt;
            }
            if (!mbar_wait(sm.tfull(b), use & 1u, abort_flag)) break;
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)b * kAccStride;
            for (int col = 32 * half; col < p.BN; col += 64) {  // 32-column units, alternating
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(trow + col, r);
                tmem_ld_wait();
                if (lane == 0) bulk_wait_group_read<1>();  // the slot's previous store has read it
                __syncwarp();
                const uint32_t sa = ring + (uint32_t)slot * 2048u + (uint32_t)lane * 64u;
#pragma unroll
                for (int i = 0; i < 32; i += 8)
                    sts_v4(sa + (uint32_t)(2 * i), pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                           pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                           pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                           pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (col < p.Dn) tma_store_2d(&tmC, h * Dk + col, t0, ring + (uint32_t)slot * 2048u);
                    else tma_store_2d(&tmD, h * p.Dv + (col - p.Dn), t0, ring + (uint32_t)slot * 2048u);
                    bulk_commit_group();
                }
                slot ^= 1;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(b));
            // the key's rope part of this head (32-channel slabs by TMA; 16 by plain
            // stores); head 0's holds it already
            if (h != 0 && DR >= 32 && lane == 0 && (DR == 64 || half == 0)) {
                tma_store_2d(&tmC, h * Dk + p.Dn + (DR == 64 ? 32 * half : 0), t0, slab);
                bulk_commit_group();
            }
            if (h != 0 && DR == 16 && half == 0 && valid) {
                const uint4 v0 = lds_v4(slab + (uint32_t)lane * 32u);
                const uint4 v1 = lds_v4(slab + (uint32_t)lane * 32u + 16u);
                uint16_t* dst = p.o_key + (t * p.H + h) * Dk + p.Dn;
                st_global_v4(dst, v0.x, v0.y, v0.z, v0.w);
                st_global_v4(dst + 8, v1.x, v1.y, v1.z, v1.w);
            }
        }
        if (lane == 0) bulk_wait_group_all();  // every output store has landed
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int quad = warp & 3;  // TMEM lane quadrant this warp may access
        const int row = quad * 32 + lane;
        const int ew = warp - 2;    // epilogue warp 0..3
        EpiCtx ec;
        ec.slots = sm.out + (uint32_t)(ew * p.nslots) * p.slot_bytes;
        ec.tmh = &tmD;
        ec.cursor = 0;
        ec.prev_pieces = 0;
        ec.prev2_pieces = 0;
        const int half = ew >> 2;   // which of the tile's units this warp takes (alternating)
        int local = 0;
        for (int tile = tile_first<false, RESC>(p); tile < tile_end<false, RESC>(p); tile = tile_next<false, RESC>(p, tile), ++local) {
            const int b = M2 ? 0 : (local & 1);
            const uint32_t use = M2 ? (uint32_t)local : (uint32_t)(local >> 1);
            if (!mbar_wait(sm.tfull(b), use & 1u, abort_flag)) break;
            tc_fence_after();
            int mt, nt;
            q_tile<DR>(p, tile, mt, nt);
            // 256-row tiles: the warps of half 1 take the second accumulator (rows 128..255)
            const int rbase = M2 ? half * kBM : 0;
            const int64_t t = (int64_t)mt * BM + rbase + row;
            const bool valid = t < p.T;
            int prow = 0;
            if (valid) {
                const int64_t pp = p.pos ? (int64_t)__ldg(p.pos + t) : t;
                if (pp < 0 || pp >= p.cs_rows) record_status(p.status, MLA_ERR_POS_RANGE);
                else prow = (int)pp;
            }
            const uint32_t trow =
                tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(M2 ? half : b) * kAccStride;
            const int64_t n0 = (int64_t)nt * p.BN;
            ec.t0 = mt * BM + rbase + quad * 32;
            ec.bias = p.bias ? p.bias + n0 : nullptr;
            ec.sword = 0;
            const bool split = HS || p.split_half;
            ec.sbase = (n0 + (split ? half * (p.BN / 2) : 0)) / 32;
            ec.hcol0 = (int32_t)n0 + half * (p.BN / 2);
            int col = split ? half * (p.BN / 2) : 0, unit = 0;
            const int col_end = split ? col + p.BN / 2 : p.BN;
            while (col < col_end) {
                const int n32 = (int)n0 + col;  // channel indices fit in 32 bits (N is an int)
                const int h = n32 / p.D;
                const int c = n32 - h * p.D;
                const int64_t n = n32;
                const bool nope = c < p.Dn;
                if (DR == 64 && !nope && !M2 && !split) {
                    // units alternate between the quadrant's two warps: both rotate the
                    // rope unit and each writes one half, which balances their work
                    if constexpr (DR == 64) rope_unit<MXOUT, DR, PACKED, HS>(p, &tmC, ec, trow + col, col, valid, t, n, h, prow, half);
                    ++unit;
                } else if (M2 || split || (unit++ & 1) == half) {
                    if (nope) nope_unit<MXOUT, slot_ch<MXOUT, DR>(), HS>(p, &tmC, ec, trow + col, col, valid, t, n, h, c);
                    else if constexpr (DR > 0) rope_unit<MXOUT, DR, PACKED, HS>(p, &tmC, ec, trow + col, col, valid, t, n, h, prow, -1);
                }
                col += nope ? 32 : DR;
            }
            if (MXOUT && split && valid)
                *reinterpret_cast<uint32_t*>(p.q_scales + t * (p.N / 32) + ec.sbase) = ec.sword;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(b));
        }
        if (lane == 0) bulk_wait_group_all();  // every output store has landed
        __syncwarp();
    }

    // ------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) record_status(p.status, MLA_ERR_TIMEOUT);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool MXW, bool MXOUT, int DR, bool PACKED = false, bool RES = false, bool HALF = false>
int launch_variant(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                   const FwdParams& p, int grid, size_t smem, cudaStream_t stream, const CUtensorMap* td = nullptr) {
    // resident weight scales, and the half-tile stores: their own instantiations
    if constexpr (MXW && !RES && DR != 0) {
        if (p.sfb_res) return launch_variant<MXW, MXOUT, DR, PACKED, true>(ta, tb, tc, p, grid, smem, stream, td);
    }
    if constexpr (!MXW && MXOUT && DR == 64 && !HALF) {
        if (p.half_store) return launch_variant<MXW, MXOUT, DR, PACKED, RES, true>(ta, tb, tc, p, grid, smem, stream, td);
    }
    auto kern = fwd_kernel<MXW, MXOUT, DR, false, PACKED, RES, HALF>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return MLA_ERR_CUDA;
    kern<<<grid, kThreads, smem, stream>>>(ta, tb, tc, td ? *td : tc, p);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

template <bool MXW, bool MXOUT, bool PACKED>
int launch_dr_t(int Dr, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& td,
                const FwdParams& p, int grid, size_t smem, cudaStream_t stream) {
    switch (Dr) {
        case 16: return launch_variant<MXW, MXOUT, 16, PACKED>(ta, tb, tc, p, grid, smem, stream, &td);
        case 32: return launch_variant<MXW, MXOUT, 32, PACKED>(ta, tb, tc, p, grid, smem, stream, &td);
        case 64: return launch_variant<MXW, MXOUT, 64, PACKED>(ta, tb, tc, p, grid, smem, stream, &td);
        default: return MLA_ERR_UNSUPPORTED;
    }
}

// the table layout is a compile-time choice: one table path per kernel
template <bool MXW, bool MXOUT>
int launch_dr(int Dr, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& td,
              const FwdParams& p, int grid, size_t smem, cudaStream_t stream) {
    return p.tab4 ? launch_dr_t<MXW, MXOUT, true>(Dr, ta, tb, tc, td, p, grid, smem, stream)
                  : launch_dr_t<MXW, MXOUT, false>(Dr, ta, tb, tc, td, p, grid, smem, stream);
}

}  // namespace

namespace {
// The shared k_pe rotated once per token (rotate-half pairs (i, i + Dr/2),
// the query's rule, fp32, rounded to bf16 once) into head 0's rope slot of
// o_key; the KV kernel copies it into the other heads. A thread takes 8
// pairs of one token. Positions outside the table: zeros, and the status.
__global__ void __launch_bounds__(256) kv_rope_pre_kernel(const uint16_t* __restrict__ k_pe, int64_t T, int Dr,
                                                          const float* __restrict__ cos_tab,
                                                          const float* __restrict__ sin_tab, long long cs_rows,
                                                          long long cs_width, const int32_t* __restrict__ pos,
                                                          uint16_t* __restrict__ o_key, int64_t key_pitch, int Dn,
                                                          int* status) {
    const int HH = Dr / 2;
    const int groups = (HH + 7) / 8;
    const int64_t items = T * groups;
    for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = it / groups;
        const int i0 = (int)(it - t * groups) * 8;
        const int n = HH - i0 < 8 ? HH - i0 : 8;  // Dr = 16: one group of 8
        const int64_t pp = pos ? (int64_t)__ldg(pos + t) : t;
        const bool ok = pp >= 0 && pp < cs_rows;
        if (!ok) record_status(status, MLA_ERR_POS_RANGE);
        uint32_t oa[4] = {0u, 0u, 0u, 0u}, oc[4] = {0u, 0u, 0u, 0u};
        if (ok) {
            const uint16_t* kp = k_pe + t * Dr;
            const float* cr = cos_tab + pp * cs_width;
            const float* sr = sin_tab + pp * cs_width;
            float ra[8], rc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (e < n) {
                    const float a = __uint_as_float((uint32_t)__ldg(kp + i0 + e) << 16);
                    const float c = __uint_as_float((uint32_t)__ldg(kp + i0 + e + HH) << 16);
                    ra[e] = a;
                    rc[e] = c;
                    rot_pair_fwd(ra[e], rc[e], __ldg(cr + i0 + e), __ldg(sr + i0 + e), __ldg(cr + i0 + e + HH),
                                 __ldg(sr + i0 + e + HH));
                } else {
                    ra[e] = rc[e] = 0.f;
                }
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                oa[w] = pack_bf16x2(ra[2 * w], ra[2 * w + 1]);
                oc[w] = pack_bf16x2(rc[2 * w], rc[2 * w + 1]);
            }
        }
        uint16_t* dst = o_key + t * key_pitch + Dn;
        // 8 channels at i0 and at i0 + HH (16-byte aligned: Dn, HH and i0 are multiples of 8)
        st_global_v4(dst + i0, oa[0], oa[1], oa[2], oa[3]);
        st_global_v4(dst + i0 + HH, oc[0], oc[1], oc[2], oc[3]);
    }
}
}  // namespace

int launch_kv_fwd(const KvArgs& a, cudaStream_t stream) {
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const int BN = a.Dn + a.Dv;
    const int64_t N = (int64_t)a.H * BN;
    FwdParams p{};
    p.T = (int)a.T;
    p.H = a.H;
    p.N = (int)N;
    p.D = BN;
    p.Dn = a.Dn;
    p.Dv = a.Dv;
    p.BN = BN;
    p.num_m_tiles = (int)((a.T + kBM - 1) / kBM);
    p.num_tiles = p.num_m_tiles * a.H;
    p.k_tiles = (int)((a.K + 63) / 64);
    p.a_bytes = kBM * 128;
    p.stage_bytes = p.a_bytes + (uint32_t)BN * 128;
    p.tx_bytes = p.stage_bytes;
    p.idesc = idesc_bf16(kBM, (uint32_t)BN, 0, 0);
    p.cos_tab = a.cos_tab;
    p.sin_tab = a.sin_tab;
    p.pos = a.pos;
    p.cs_rows = a.cs_rows;
    p.cs_width = a.cs_width;
    p.cs_vec = (a.cs_width % 4 == 0) && (reinterpret_cast<uintptr_t>(a.cos_tab) % 16 == 0) &&
               (reinterpret_cast<uintptr_t>(a.sin_tab) % 16 == 0);
    p.o_key = static_cast<uint16_t*>(a.o_key);
    p.o_value = static_cast<uint16_t*>(a.o_value);
    p.k_pe = static_cast<const uint16_t*>(a.k_pe);
    p.status = a.status;
    p.slot_bytes = 2048;  // epilogue warp: 2 ring slots + the rope slab, 32 rows x 32 bf16 each
    p.nslots = 3;
    const size_t fixed = 1024 + 256 + (size_t)kEpiWarps * 3 * 2048;
    int stages = (int)((size_t)(di.max_smem_optin - fixed) / p.stage_bytes);
    if (stages > 8) stages = 8;
    if (stages < 2) return MLA_ERR_UNSUPPORTED;
    p.stages = stages;
    const size_t smem = fixed + (size_t)stages * p.stage_bytes;
    alignas(64) CUtensorMap ta, tb, tc, td;
    st = make_tmap_2d(&ta, a.c_kv, 1, (uint64_t)a.K, (uint64_t)a.T, (uint64_t)a.K * 2, 64, kBM, true);
    if (st != MLA_OK) return st;
    st = make_tmap_2d(&tb, a.W, 1, (uint64_t)a.K, (uint64_t)N, (uint64_t)a.K * 2, 64, (uint32_t)BN, true);
    if (st != MLA_OK) return st;
    // outputs as 2-D [T, H*Dk] and [T, H*Dv]: store boxes of 32 channels x 32 tokens
    const int64_t Dk = a.Dn + a.Dr;
    st = make_tmap_2d(&tc, a.o_key, 1, (uint64_t)(a.H * Dk), (uint64_t)a.T, (uint64_t)(a.H * Dk) * 2, 32, 32, false);
    if (st != MLA_OK) return st;
    st = make_tmap_2d(&td, a.o_value, 1, (uint64_t)a.H * a.Dv, (uint64_t)a.T, (uint64_t)a.H * a.Dv * 2, 32, 32, false);
    if (st != MLA_OK) return st;
    const int grid = p.num_tiles < di.num_sms ? p.num_tiles : di.num_sms;
    // 1. the shared k_pe, rotated once into head 0's rope slot
    {
        const int64_t items = a.T * ((a.Dr / 2 + 7) / 8);
        int64_t blocks = (items + 255) / 256;
        if (blocks > (int64_t)di.num_sms * 8) blocks = (int64_t)di.num_sms * 8;
        if (blocks > 0)
            kv_rope_pre_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
                static_cast<const uint16_t*>(a.k_pe), a.T, a.Dr, a.cos_tab, a.sin_tab, a.cs_rows, a.cs_width, a.pos,
                static_cast<uint16_t*>(a.o_key), (int64_t)a.H * Dk, a.Dn, a.status);
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    }
    // 2. the GEMM, its epilogue copying the rope part into the other heads
    const void* k = nullptr;
    switch (a.Dr) {
        case 16: k = (const void*)fwd_kernel<false, false, 16, true>; break;
        case 32: k = (const void*)fwd_kernel<false, false, 32, true>; break;
        case 64: k = (const void*)fwd_kernel<false, false, 64, true>; break;
        default: return MLA_ERR_UNSUPPORTED;
    }
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MLA_ERR_CUDA;
    switch (a.Dr) {
        case 16: fwd_kernel<false, false, 16, true><<<grid, kThreads, smem, stream>>>(ta, tb, tc, td, p); break;
        case 32: fwd_kernel<false, false, 32, true><<<grid, kThreads, smem, stream>>>(ta, tb, tc, td, p); break;
        default: fwd_kernel<false, false, 64, true><<<grid, kThreads, smem, stream>>>(ta, tb, tc, td, p); break;
    }
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

namespace {
// out[i * rows + p] = (cos[p, i], sin[p, i], cos[p, i + h], sin[p, i + h]):
// a re-layout of the table's first 2h columns, no arithmetic.
__global__ void __launch_bounds__(256) rope_table_pack_kernel(const float* __restrict__ cos_tab,
                                                              const float* __restrict__ sin_tab, long long rows,
                                                              long long width, int h, float4* __restrict__ out) {
    const long long n = rows * h;
    for (long long k = (long long)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += (long long)gridDim.x * blockDim.x) {
        const long long i = k / rows, pr = k - i * rows;
        const long long o = pr * width + i;
        out[k] = make_float4(__ldg(cos_tab + o), __ldg(sin_tab + o), __ldg(cos_tab + o + h), __ldg(sin_tab + o + h));
    }
}
}  // namespace

int launch_rope_table_pack(int64_t rows, int64_t width, int Dr, const float* cos_tab, const float* sin_tab,
                           void* packed, cudaStream_t stream) {
    const long long n = rows * (Dr / 2);
    if (n == 0) return MLA_OK;
    long long blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    rope_table_pack_kernel<<<(unsigned)blocks, 256, 0, stream>>>(cos_tab, sin_tab, rows, width, Dr / 2,
                                                                 static_cast<float4*>(packed));
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int fwd_tile_n(int64_t N, int D, int Dn, int Dr, int max_bn, int step) {
    for (int bn = max_bn / step * step; bn >= step; bn -= step) {
        if (N % bn) continue;
        bool ok = true;
        const int64_t heads = N / D;
        for (int64_t h = 0; ok && h < heads; ++h) {
            const int64_t rs = h * D + Dn, re = h * D + D - 1;  // rope region (none when Dr == 0)
            if (Dr > 0 && rs / bn != re / bn) ok = false;
            for (int c = 0; ok && c < Dn; c += 32)  // pass-through blocks
                if ((h * D + c) / bn != (h * D + c + 31) / bn) ok = false;
        }
        if (ok) return bn;
    }
    return 0;
}

int launch_fwd(const FwdArgs& a, cudaStream_t stream) {
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const bool mxw = a.weight_mode == MLA_WEIGHT_MXFP8;
    const int D = a.Dn + a.Dr;
    const int64_t N = (int64_t)a.H * D;
    // TMEM: two accumulators at columns 0 and 256; MXFP8 scale factors from column 448.
    const int BN = fwd_tile_n(N, D, a.Dn, a.Dr, mxw ? 192 : 256, mxw ? 32 : 16);
    if (BN == 0) return MLA_ERR_UNSUPPORTED;

    FwdParams p{};
    p.T = (int)a.T;
    p.H = a.H;
    p.N = (int)N;
    p.D = D;
    p.Dn = a.Dn;
    p.BN = BN;
    const int bm = a.Dr == 0 ? 2 * kBM : kBM;  // the plain GEMM's 256-row tiles
    p.num_m_tiles = (int)((a.T + bm - 1) / bm);
    p.num_n_tiles = (int)(N / BN);
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    const int bk = mxw ? 128 : 64;  // K elements per 128-byte row
    p.k_tiles = (int)((a.K + bk - 1) / bk);
    p.a_bytes = (uint32_t)bm * 128;
    p.stage_bytes = p.a_bytes + (uint32_t)BN * 128;
    p.sf_stage = bm == kBM ? kSfBytesPerStage : kSfBytesPerStage2;
    p.sf_cols = bm == kBM ? kSfColsPerStage : kSfColsPerStage2;
    p.sf_tiled = a.sf_tiled;
    p.sf_nsub = (BN + 127) / 128;
    if (a.sf_tiled && (!mxw || BN != a.sf_group)) return MLA_ERR_UNSUPPORTED;
    if (a.Dr == 0 && mxw && !a.sf_tiled) return MLA_ERR_UNSUPPORTED;  // 256-row tiles load tiled scales only
    p.tx_bytes = p.stage_bytes + (a.sf_tiled ? 512u * ((uint32_t)(bm / kBM) + (uint32_t)p.sf_nsub) : 0u);
    p.idesc = mxw ? idesc_mxf8(kBM, BN, 0) : idesc_bf16(kBM, BN, 0, 0);
    p.ksb = (int)(a.ld_scale ? a.ld_scale : a.K / 32);
    p.bias = static_cast<const uint16_t*>(a.bias);
    p.cos_tab = a.cos_tab;
    p.sin_tab = a.sin_tab;
    p.tab4 = static_cast<const float4*>(a.rope_packed);
    p.pos = a.pos;
    p.cs_rows = a.Dr == 0 ? (long long)INT64_MAX : a.cs_rows;  // plain GEMM: no table rows read
    p.cs_width = a.cs_width;
    p.q_out = static_cast<uint8_t*>(a.q_out);
    p.q_scales = a.q_scales;
    p.x_scales = a.x_scales;
    p.w_scales = a.w_scales;
    p.status = a.status;
    p.cs_vec = (a.cs_width % 4 == 0) && (reinterpret_cast<uintptr_t>(a.cos_tab) % 16 == 0) &&
               (reinterpret_cast<uintptr_t>(a.sin_tab) % 16 == 0);
    const bool mxo = a.out_mode != MLA_OUT_BF16;
    p.scales_bhsd = a.out_mode == MLA_OUT_MXFP8_BHSD;
    p.qs_swz = a.out_mode == MLA_OUT_MXFP8_BHSD_SWIZZLED;
    p.qs_row_tiles = (int)((a.T + 127) / 128);
    p.qs_col_tiles = (D / 32 + (D % 32 ? 1 : 0) + 3) / 4;
    // 32 rows x 32 bytes per slot; a unit takes at most 4 slots (64 bf16 rope
    // channels, or 16-channel MXFP8 slots), 2 with 32-channel MXFP8 slots
    const int slot_c = mxo && a.Dr % 32 == 0 ? 32 : 16;
    p.slot_bytes = 1024;
    p.nslots = 4;
    // The half split packs a row's scale bytes for half a tile into one aligned
    // 4-byte word: only when half a tile is exactly 4 blocks (BN = 256, so the
    // word starts at a multiple of 4 blocks) and rows of scales keep 4-byte
    // alignment (N % 128 == 0).
    p.split_half = mxo && !p.scales_bhsd && !p.qs_swz && D % 32 == 0 && BN == 256 && N % 128 == 0 &&
                   reinterpret_cast<uintptr_t>(a.q_scales) % 4 == 0 &&
                   fwd_tile_n(N, D, a.Dn, a.Dr, BN / 2, BN / 2) == BN / 2;
    // Two 64-channel store boxes per half tile: the warp's 4 KB of staging
    // slots hold them, 512-byte aligned (the stages before them are multiples
    // of 1 KB with bf16 weights); rope regions start on 64-channel boundaries.
    p.half_store = p.split_half && !mxw && a.Dr % 32 == 0 && BN / 2 == 128 && a.Dn % 64 == 0 && D % 64 == 0 &&
                   p.nslots * p.slot_bytes == 4096;

    const size_t fixed = 1024 /* alignment slack */ + 256 /* barriers + slots */ +
                         (size_t)kEpiWarps * p.nslots * p.slot_bytes;
    const size_t per_stage = p.stage_bytes + (mxw ? p.sf_stage : 0);
    int stages = (int)((size_t)(di.max_smem_optin - fixed) / per_stage);
    if (stages > 8) stages = 8;
    if (stages < 2) return MLA_ERR_UNSUPPORTED;
    if (mxw && kSfCol0 + p.sf_cols * (uint32_t)stages > kTmemCols) stages = (kTmemCols - kSfCol0) / p.sf_cols;
    p.stages = stages;
    // Resident weight scales (MXFP8 weights, tiled scales, 128-row tiles): 8
    // TMEM columns per K step, first in the columns between the accumulators
    // ([BN, 256); accumulator 1 ends at 256 + BN <= kSfCol0), then after the
    // x scales (4 columns per stage from kSfCol0). Each CTA then takes one
    // range of tiles, token tile fastest, so it keeps a channel tile for up
    // to num_m_tiles tiles. A tile's x scales come in one bulk copy into one
    // of two buffers (k_tiles x 512 bytes each), so a stage carries only the
    // two operand tiles: the SM's TMA unit completes operations at a fixed
    // rate whatever their size, and that rate paces this main loop.
    size_t stage_sf = mxw ? p.sf_stage : 0, xbuf = 0;
    if (mxw && a.sf_tiled && bm == kBM && BN <= 192 && p.k_tiles >= stages) {
        const int n1 = (256 - BN) / 8;
        const int col2 = (int)kSfCol0 + 4 * stages;
        const uint32_t sfs = 512u * (uint32_t)p.sf_nsub;
        const size_t xb = 2u * 512u * (size_t)p.k_tiles;
        if (p.k_tiles <= n1 + ((int)kTmemCols - col2) / 8 &&
            fixed + (size_t)stages * (p.stage_bytes + sfs) + xb <= (size_t)di.max_smem_optin) {
            p.sfb_res = 1;
            p.sf_cols = 4;
            p.sfb_n1 = n1;
            p.sfb_col2 = col2;
            p.sf_stage = sfs;
            stage_sf = sfs;
            xbuf = xb;
        }
    }
    const size_t smem = fixed + (size_t)stages * (p.stage_bytes + stage_sf) + xbuf;

    alignas(64) CUtensorMap ta, tb;
    const uint64_t esz = mxw ? 1 : 2;
    st = make_tmap_2d(&ta, a.x, mxw ? 0 : 1, (uint64_t)a.K, (uint64_t)a.T,
                      (uint64_t)(a.ld_x ? a.ld_x : a.K) * esz, 128 / (uint32_t)esz, (uint32_t)bm, true);
    if (st != MLA_OK) return st;
    st = make_tmap_2d(&tb, a.W, mxw ? 0 : 1, (uint64_t)a.K, (uint64_t)N, (uint64_t)(a.ld_w ? a.ld_w : a.K) * esz,
                      128 / (uint32_t)esz, (uint32_t)BN, true);
    if (st != MLA_OK) return st;
    // output q [T, N] (bf16 or E4M3 bytes): TMA store boxes of slot_c channels x 32 tokens
    alignas(64) CUtensorMap tc;
    st = make_tmap_2d(&tc, a.q_out, mxo ? 0 : 1, (uint64_t)N, (uint64_t)a.T, (uint64_t)N * (mxo ? 1 : 2),
                      (uint32_t)slot_c, 32, false);
    if (st != MLA_OK) return st;

    int grid = p.num_tiles < di.num_sms ? p.num_tiles : di.num_sms;
    if (a.Dr == 0)  // plain GEMM: every unit is a pass-through unit
        return mxw ? launch_variant<true, false, 0>(ta, tb, tc, p, grid, smem, stream)
                   : launch_variant<false, false, 0>(ta, tb, tc, p, grid, smem, stream);
    // the half-tile stores: 64 channels x 32 tokens, 64-byte swizzle
    alignas(64) CUtensorMap td = tc;
    if (p.half_store) {
        st = make_tmap_2d(&td, a.q_out, 0, (uint64_t)N, (uint64_t)a.T, (uint64_t)N, 64, 32, false, true);
        if (st != MLA_OK) return st;
    }
    if (mxw)
        return mxo ? launch_dr<true, true>(a.Dr, ta, tb, tc, td, p, grid, smem, stream)
                   : launch_dr<true, false>(a.Dr, ta, tb, tc, td, p, grid, smem, stream);
    return mxo ? launch_dr<false, true>(a.Dr, ta, tb, tc, td, p, grid, smem, stream)
               : launch_dr<false, false>(a.Dr, ta, tb, tc, td, p, grid, smem, stream);
}

}  // namespace mlaq
