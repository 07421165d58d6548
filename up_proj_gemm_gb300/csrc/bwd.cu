// Backward of the fused MLA query up-projection on sm_103a tensor cores.
//
// TransformerEngine PR "Add a backwards linear function to be used with the
// fused mla q up-proj": the query gradient first goes through the RoPE
// backward (dq_pre = J^T dq), then the linear backward gives
//   dgrad  dx[T, K] = dq_pre[T, N] W[N, K]
//   wgrad  dW[N, K] = dq_pre[T, N]^T x[T, K]       (the saved input x)
//   bgrad  db[N]    = sum_t dq_pre[t, N]          (review: "BF16 bias gradient
//                                                   remains missing")
// The pages run the RoPE backward as its own Triton kernel and hand dq_pre
// to a library GEMM. Here only the rope third of dq_pre is ever stored, and
// on some shapes not even that. Persistent kernels (one CTA per SM), each
// with a single-thread tcgen05.mma issuer and 128-byte-swizzled TMA stages:
//
//   rope_pre_kernel (Dr = 64, Dn % 64 == 0): rotates every head's rope
//     channels once into dq_pre_rope [T, H, 64] bf16 (the caller's buffer or
//     dgrad's workspace); a thread takes 8 pairs of eight heads of a token,
//     loading the token's table entries once.
//   dgrad_pre_kernel: dx as a plain GEMM over [dq pass-through | rotated rope]:
//     every 64-channel K chunk comes whole from one of the two. 256-token
//     tiles are two M = 128 MMAs per stage into TMEM columns 0 and 256. The
//     reduction is split by wave efficiency into fp32 partials that
//     dgrad_reduce_kernel adds in a fixed order.
//   dgrad_kernel (other shapes, or less workspace): A = dq [T x N] K-major,
//     B = W [N x K] MN-major, reduction over channels, 64 per stage, with
//     separate rings and producers for A and B (warps 0 and 14). Warps 2-5
//     are the epilogue (bf16 dx, or fp32 partials when split); warps 6-13
//     are "transform" warps. Each thread of those owns half of one token row
//     for a whole work unit, keeps that row's cos/sin in registers, and
//     rotates the rope channels of each dq tile in shared memory (fp32 math,
//     rounded to bf16, the MMA operand type). They fence the tile into the
//     async proxy and release the stage. They can also store the rotated
//     channels to dq_pre_rope.
//   wgrad_pre_kernel (paired heads: Dr = 64, Dn % 128 == 0, even H,
//     K % 64 == 0, dq_pre_rope given): 256-channel tiles of two 128-channel
//     sub-tiles in head-pair order, A = dq_pre^T MN-major from dq or the
//     rotated buffer, B = x [T x K] MN-major, 64-token stages, two
//     accumulators. Warps 10-17 sum db over the tokens of the first column
//     tile, in a fixed order.
//   wgrad_kernel (other shapes, or no hand-off): 128-channel tiles,
//     32-token stages (each stage needs fresh table rows), three transform
//     groups of 4 warps rotating the rope stages and summing db.
//
// In the transform kernels a shared-memory "row" is 128 bytes = 64
// consecutive channels of one token, which is what the transform rewrites.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstring>

#include "internal.h"
#include "mx.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

constexpr int kBM = 128;
constexpr int kXformWarp0 = 6;

// Reduction rows per stage: 64 channels (dgrad); 32 tokens for a wgrad that
// rotates (its stages each need fresh cos/sin rows: a deeper ring of smaller
// stages), 64 for a wgrad whose rope tiles come rotated.
constexpr int kBKD = 64, kBKW = 32, kBKWPre = 64;
// wgrad: transform groups taking turns on stages, threads per group, block size
constexpr int kWgGroups = 3;
constexpr int kWgGroupThreads = 128;
constexpr int kWgThreads = 32 * kXformWarp0 + kWgGroupThreads * kWgGroups;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccStride = 256;

struct BwdParams {
    int T, K, N, D, Dn;
    int BN;
    int num_m_tiles, num_n_tiles, num_tiles, k_tiles;
    int stages;
    uint32_t a_bytes, stage_bytes, tx_bytes;
    uint32_t idesc;
    const int32_t* pos;
    const float* cos_tab;
    const float* sin_tab;
    long long cs_rows, cs_width;
    int cs_vec;  // cos/sin rows 16-byte aligned: float4 loads
    int a3d, b3d;  // operand maps are 3-D chunk views (one TMA op per operand and stage)
    // wgrad channel tiles by head pair (see tile_chunks); tiles per pair
    int paired, tiles_per_pair;
    // wgrad: the rope tiles come rotated from dq_pre_rope (wgrad_pre_kernel)
    int pre;
    // dgrad: rotated rope channels out, [T, H, Dr] bf16 (nullable; each head's
    // channels written by the units of column tile head mod num_n_tiles)
    uint16_t* rope_out;
    int H, Dr;
    // dgrad: slots of the A ring and of the B ring, bytes of one B slot
    int sa_slots, sb_slots;
    uint32_t b_bytes;
    uint16_t* out;
    int out_rows, out_cols;
    // work units: each tile's reduction split in ksplit parts of kts stages
    // (dgrad only; the parts write fp32 partials to ws, summed afterwards)
    int ksplit, kts, num_units;
    float* ws;
    // dgrad_pre_kernel's stream-K schedule: (token tile, K step) iterations,
    // one fp32 partial slot [BN/4][256] float4 and one flag per CTA (null
    // when no tile is split), and this launch's flag value
    long long sk_total;
    float* sk_slots;
    unsigned* sk_flags;
    unsigned sk_epoch;
    uint16_t* db;
    int* status;
};

struct Smem {
    uint32_t base, bars;
    int S;
    __device__ uint32_t a(int s, const BwdParams& p) const { return base + (uint32_t)s * p.stage_bytes; }
    __device__ uint32_t b(int s, const BwdParams& p) const { return a(s, p) + p.a_bytes; }
    // full: TMA landed (stages the transform does not touch; awaited by the MMA)
    // xfull: TMA landed (transform stages; one set per transform group, awaited
    //        only by that group, so every barrier sees its uses in order)
    // ready: transform done (awaited by the MMA); empty: MMA done (producer)
    __device__ uint32_t full(int s) const { return bars + 8u * s; }
    __device__ uint32_t ready(int s) const { return bars + 8u * (S + s); }
    __device__ uint32_t empty(int s) const { return bars + 8u * (2 * S + s); }
    __device__ uint32_t tfull(int b) const { return bars + 8u * (3 * S + b); }
    __device__ uint32_t tempty(int b) const { return bars + 8u * (3 * S + 2 + b); }
    __device__ uint32_t drain() const { return bars + 8u * (3 * S + 4); }
    __device__ uint32_t xfull(int g, int s) const { return bars + 8u * (3 * S + 5 + g * S + s); }
};

__device__ __forceinline__ void lds_v4(uint32_t addr, uint32_t (&v)[4]) {
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
                 : "r"(addr));
}
__device__ __forceinline__ void sts_v4(uint32_t addr, const uint32_t (&v)[4]) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]),
                 "r"(v[3])
                 : "memory");
}

__device__ __forceinline__ void load8(const float* p, bool vec, float* v) {
    if (vec) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(p));
        const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = __ldg(p + e);
    }
}

// Start channels of the rope regions inside [n0, n0 + width). Rope regions
// are Dr-aligned and Dr <= 64 divides 64, so none straddles a 64-channel row
// or a 128-channel tile. (N < 2^31: 32-bit arithmetic.)
__device__ __forceinline__ int rope_regions(const BwdParams& p, int n0, int width, int (&st)[8]) {
    int cnt = 0;
    for (int rs = (n0 / p.D) * p.D + p.Dn; cnt < 8 && rs < n0 + width && rs < p.N; rs += p.D)
        if (rs >= n0) st[cnt++] = rs;
    return cnt;
}

__device__ __forceinline__ bool has_rope(const BwdParams& p, int n0, int width) {
    int rs = (n0 / p.D) * p.D + p.Dn;
    if (rs < n0) rs += p.D;
    return rs < n0 + width && rs < p.N;
}

// Work unit u -> its tile and split. Units run split-major: the CTAs of a
// wave share one slice of the reduction, so each slice of the reused operand
// (W for dgrad) is read from DRAM about once instead of once per wave.
__device__ __forceinline__ void unit_split(const BwdParams& p, int u, int& tile, int& sp) {
    sp = u / p.num_tiles;
    tile = u - sp * p.num_tiles;
}

// Work unit u -> its tile and stage range [k0, k1).
__device__ __forceinline__ void unit_range(const BwdParams& p, int u, int& tile, int& k0, int& k1) {
    int sp;
    unit_split(p, u, tile, sp);
    k0 = sp * p.kts;
    k1 = min(p.k_tiles, k0 + p.kts);
}

// wgrad: channel starts of the two 64-channel chunks of channel tile mt
// (a start >= N means that half is empty) and whether it is a rope pair.
// Contiguous tiles [128 mt, 128 mt + 128) in general. With heads paired
// (rope dim 64, pass-through dim a multiple of 128, even H), each head pair
// has its pass-through chunks in tiles of 128 contiguous channels, then one
// tile holding both heads' 64 rope channels: only a third of the tiles need
// the inverse rotation, and each cos/sin row serves two heads.
__device__ __forceinline__ void tile_chunks(const BwdParams& p, int mt, int& c0, int& c1, bool& rope_pair) {
    rope_pair = false;
    if (!p.paired) {
        c0 = mt * kBM;
        c1 = c0 + 64;
        return;
    }
    const int g = mt / p.tiles_per_pair, k = mt - g * p.tiles_per_pair;
    const int nh = p.Dn / 128;  // pass-through tiles per head
    if (k < 2 * nh) {
        c0 = (2 * g + k / nh) * p.D + (k % nh) * 128;
        c1 = c0 + 64;
    } else {
        c0 = 2 * g * p.D + p.Dn;
        c1 = c0 + p.D;
        rope_pair = true;
    }
}

// Walks a CTA's stages (its tiles, each k-tile of each) and says which go
// through the transform warps (else TMA -> MMA directly): dgrad stages whose
// 64 channels hold rope channels; every stage of a wgrad tile that holds
// rope channels or sums the bias gradient. Incremental: no division per
// stage, since the producer's loop paces the whole pipeline.
template <bool WG>
struct StageWalk {
    int mt = 0, nt = 0;
    bool tile_x = false;  // wgrad: the tile's stages are transform stages
    int c0 = 0;           // dgrad: channel phase (kt * 64) mod D of the current stage
    // wgrad: the tile's two chunk starts, and the A operand's TMA source:
    // rope view (head pair) or chunk view / 2-D map; az = its 3rd coordinate
    int w0 = 0, w1 = 0, az = 0;
    bool rope_pair = false;
    __device__ void begin_tile(const BwdParams& p, int tile, int k0) {
        mt = tile / p.num_n_tiles;
        nt = tile % p.num_n_tiles;
        c0 = WG ? 0 : (k0 * kBKD) % p.D;
        if (WG) {
            tile_chunks(p, mt, w0, w1, rope_pair);
            const bool rot = rope_pair || has_rope(p, w0, 64) || has_rope(p, w1, 64);
            tile_x = rot || (p.db != nullptr && nt == 0);
            az = rope_pair ? (w0 - p.Dn) / p.D : w0 / 64;
        }
    }
    __device__ bool needs(const BwdParams& p, int kt) const {
        if (WG) return tile_x;
        const int off = (c0 <= p.Dn) ? (p.Dn - c0) : (p.D + p.Dn - c0);  // next rope region start
        return off < kBKD && kt * kBKD + off < p.N;
    }
    __device__ void next(const BwdParams& p) {
        if (!WG) {
            c0 += kBKD;
            while (c0 >= p.D) c0 -= p.D;
        }
    }
};

// Inverse RoPE of one pair in float32, one fma each with the other product
// rounded first, so every path that rotates dq (the fused dgrad and wgrad
// transforms, the standalone pass) produces the same bf16 bits:
//   out[i]     = fma(g[i],   cos[i],   fl(g[i+h] sin[i+h]))
//   out[i + h] = fma(g[i+h], cos[i+h], -fl(g[i] sin[i]))
// 8 pairs: g1 holds g[i .. i+8) and g2 g[i+h .. i+h+8) as bf16 pairs; ci/si at
// i, cj/sj at i + h; o1/o2 the rotated values as bf16 pairs.
__device__ __forceinline__ void rope_inv8(const uint32_t (&g1)[4], const uint32_t (&g2)[4], const float* ci,
                                          const float* si, const float* cj, const float* sj, uint32_t (&o1)[4],
                                          uint32_t (&o2)[4]) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float gi0 = bf16lo_to_f32(g1[w]), gi1 = bf16hi_to_f32(g1[w]);
        const float gj0 = bf16lo_to_f32(g2[w]), gj1 = bf16hi_to_f32(g2[w]);
        const int e0 = 2 * w, e1 = 2 * w + 1;
        o1[w] = pack_bf16x2(__fmaf_rn(gi0, ci[e0], __fmul_rn(gj0, sj[e0])),
                            __fmaf_rn(gi1, ci[e1], __fmul_rn(gj1, sj[e1])));
        o2[w] = pack_bf16x2(__fmaf_rn(gj0, cj[e0], -__fmul_rn(gi0, si[e0])),
                            __fmaf_rn(gj1, cj[e1], -__fmul_rn(gi1, si[e1])));
    }
}

// Inverse RoPE on 8 pairs of one token, in place in a 128-byte swizzled
// shared-memory row (row index r inside its 1024-byte swizzle group gives
// the XOR). Chunk q1 holds g[i], chunk q2 = q1 + Dr/16 holds g[i + Dr/2]:
//   out[i]        =  g[i] cos[p, i] + g[i+h] sin[p, i+h]
//   out[i + h]    = -g[i] sin[p, i] + g[i+h] cos[p, i+h]     (h = Dr / 2)
// ci/si: cos, sin at i; cj/sj: cos, sin at i + h (8 consecutive pairs).
// o (nullable): the rotated values as written (bf16 pairs: 4 words at i, 4 at i + h).
__device__ __forceinline__ void rot8(uint32_t row_addr, int r, int q1, int q2, const float* ci,
                                     const float* si, const float* cj, const float* sj,
                                     uint32_t* o = nullptr) {
    const uint32_t a1 = row_addr + (uint32_t)((q1 ^ (r & 7)) * 16);
    const uint32_t a2 = row_addr + (uint32_t)((q2 ^ (r & 7)) * 16);
    uint32_t g1[4], g2[4];
    lds_v4(a1, g1);
    lds_v4(a2, g2);
    uint32_t o1[4], o2[4];
    rope_inv8(g1, g2, ci, si, cj, sj, o1, o2);
    sts_v4(a1, o1);
    sts_v4(a2, o2);
    if (o != nullptr) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            o[w] = o1[w];
            o[4 + w] = o2[w];
        }
    }
}

// Position row of token t, or -1 (recorded) when outside the table.
__device__ __forceinline__ int pos_row(const BwdParams& p, int64_t t) {
    const int64_t pp = p.pos ? (int64_t)__ldg(p.pos + t) : t;
    if (pp < 0 || pp >= p.cs_rows) {
        record_status(p.status, MLA_ERR_POS_RANGE);
        return -1;
    }
    return (int)pp;
}

template <int DR, int BK>
__global__ void __launch_bounds__(kWgThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmR,
               const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.S = p.stages;
    sm.base = (raw + 1023u) & ~1023u;
    sm.bars = sm.base + (uint32_t)p.stages * p.stage_bytes;
    uint8_t* tail = smem_raw + (sm.bars - raw) + 8u * ((3 + kWgGroups) * p.stages + 5);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(tail);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 4);
    float* db_part = reinterpret_cast<float*>(tail + 16);  // 2 x groups x 128 floats (wgrad bias sums)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.ready(s), kWgGroupThreads / 32);
            mbar_init(sm.empty(s), 1);
            for (int g = 0; g < kWgGroups; ++g) mbar_init(sm.xfull(g, s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.tfull(b), 1);
            mbar_init(sm.tempty(b), 4);
        }
        mbar_init(sm.drain(), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32((const void*)tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nb_chunks = p.BN / 64;
    constexpr uint32_t CH = (uint32_t)BK * 128u;  // bytes of one 64-wide MN-major chunk

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        int s = 0;
        uint32_t ph = 0;
        int gnext = 0;  // group owning the next transform stage
        // per-slot parity of each barrier's next use (full, and xfull of groups 0..2),
        // and which barrier each slot's last use went to (2 bits: 0 full, g+1 xfull g)
        uint32_t fpar = 0, xp0 = 0, xp1 = 0, xp2 = 0, last_kind = 0, issued_mask = 0;
        StageWalk<true> walk;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
            int tile, k0, k1;
            unit_range(p, u, tile, k0, k1);
            walk.begin_tile(p, tile, k0);
            const int nt = walk.nt;
            for (int kt = k0; kt < k1; ++kt, walk.next(p)) {
                if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                uint32_t fb;
                uint32_t kind = 0;
                if (walk.needs(p, kt)) {
                    const int g = gnext;
                    gnext = (gnext + 1 == kWgGroups) ? 0 : gnext + 1;
                    fb = sm.xfull(g, s);
                    if (g == 0) xp0 ^= 1u << s;
                    else if (g == 1) xp1 ^= 1u << s;
                    else xp2 ^= 1u << s;
                    kind = (uint32_t)g + 1;
                } else {
                    fb = sm.full(s);
                    fpar ^= 1u << s;
                }
                last_kind = (last_kind & ~(3u << (2 * s))) | (kind << (2 * s));
                if (lane == 0) {
                    mbar_arrive_expect_tx(fb, p.tx_bytes);
                    // A: dq^T, the tile's two 64-channel chunks, tokens [kt*BK, +BK)
                    // (rope pair: the rope view, heads 2g and 2g+1, head stride D)
                    if (walk.rope_pair || p.a3d)
                        tma_load_3d(sm.a(s, p), walk.rope_pair ? &tmR : &tmA, 0, kt * BK, walk.az, fb);
                    else {
                        tma_load_2d(sm.a(s, p), &tmA, walk.w0, kt * BK, fb);
                        tma_load_2d(sm.a(s, p) + CH, &tmA, walk.w1, kt * BK, fb);
                    }
                    // B: 64-column chunks of x (rows = tokens)
                    if (p.b3d) {
                        tma_load_3d(sm.b(s, p), &tmB, 0, kt * BK, nt * nb_chunks, fb);
                    } else {
                        for (int c = 0; c < nb_chunks; ++c)
                            tma_load_2d(sm.b(s, p) + (uint32_t)c * CH, &tmB, nt * p.BN + 64 * c, kt * BK, fb);
                    }
                }
                issued_mask |= 1u << s;
                if (++s == p.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok) {
            // unwinding: let every copy this warp started land before the CTA
            // exits (bounded; the last use of each slot's barrier)
            for (int q = 0; q < p.stages; ++q) {
                if (!(issued_mask & (1u << q))) continue;
                const uint32_t k = (last_kind >> (2 * q)) & 3u;
                const uint32_t bits = k == 0 ? fpar : (k == 1 ? xp0 : (k == 2 ? xp1 : xp2));
                // the last use toggled its bit: its phase has the other parity
                mbar_wait(k == 0 ? sm.full(q) : sm.xfull((int)k - 1, q), ((bits >> q) & 1u) ^ 1u, nullptr,
                          200000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            uint32_t rpar = 0, fpar = 0;  // per-slot parities of the ready / full barriers
            StageWalk<true> walk;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++local) {
                int tile, k0, k1;
                unit_range(p, u, tile, k0, k1);
                const int b = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!mbar_wait(sm.tempty(b), (use & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)b * kAccStride;
                walk.begin_tile(p, tile, k0);
                for (int kt = k0; kt < k1; ++kt, walk.next(p)) {
                    const bool xf = walk.needs(p, kt);
                    // transform stages: wait for the transform's release; others: the TMA
                    const uint32_t bar = xf ? sm.ready(s) : sm.full(s);
                    const uint32_t par = ((xf ? rpar : fpar) >> s) & 1u;
                    if (!mbar_wait(bar, par, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (xf) rpar ^= 1u << s;
                    else fpar ^= 1u << s;
                    tc_fence_after();
                    const uint32_t a0 = sm.a(s, p), b0 = sm.b(s, p);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j) {
                        // 16 reduction rows (tokens) per MMA: 16 rows of 128 bytes
                        // in each MN-major chunk
                        const uint64_t ad = desc_mnmajor_sw128(a0 + 2048u * j, CH);
                        const uint64_t bd = desc_mnmajor_sw128(b0 + 2048u * j, CH);
                        mma_bf16(d_tmem, ad, bd, p.idesc, (kt != k0 || j != 0));
                    }
                    mma_commit(sm.empty(s));
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) mma_commit(sm.tfull(b));
            }
            if (!ok) {
                mma_commit(sm.drain());
                mbar_wait(sm.drain(), 0, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp < kXformWarp0) {
        // ---------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        int local = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++local) {
            const int tile = u;  // wgrad does not split its reduction
            const int b = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!mbar_wait(sm.tfull(b), use & 1u, abort_flag)) break;
            tc_fence_after();
            const int mt = tile / p.num_n_tiles;
            const int nt = tile % p.num_n_tiles;
            int c0, c1;
            bool rp;
            tile_chunks(p, mt, c0, c1, rp);
            const int64_t orow = (row < 64 ? c0 : c1) + (row & 63);  // output channel
            const bool valid = orow < p.out_rows;
            const uint32_t trow = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)b * kAccStride;
            for (int col = 0; col < p.BN; col += 32) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(trow + col, r);
                tmem_ld_wait();
                const int64_t kc = (int64_t)nt * p.BN + col;
                if (valid) {
                    uint16_t* dst = p.out + orow * p.out_cols + kc;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        if (kc + i + 8 <= p.out_cols)
                            st_global_v4(dst + i,
                                         pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                         pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                         pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                                         pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(b));
        }
    } else {
        // --------------------------------------------------------- transform
        constexpr int G = kWgGroups;
        constexpr int GT = kWgGroupThreads;
        constexpr int HH = DR / 2;
        // Work split of one stage: TPR threads per token row; each thread owns
        // the pairs [k PPI, (k + 1) PPI) of the rope regions it takes (region j
        // goes to the threads with (j * IPR + k) % TPR == sub).
        constexpr int TPR = 4;
        constexpr int PPI = (HH / TPR >= 8) ? HH / TPR : 8;  // pairs per item: 8 or 16
        constexpr int IPR = HH / PPI;                        // items per region: 1, 2 or 4
        const int xt = threadIdx.x - kXformWarp0 * 32;
        const int grp = xt / GT;  // this thread's group
        const int gt = xt % GT;   // thread within the group
        const int r = gt / TPR, sub = gt % TPR;
        const int kpart = sub % IPR;
        const int pb = kpart * PPI;  // first pair of this thread's items
        const bool vec = p.cs_vec != 0;
        int s = 0;
        uint32_t xpar = 0;  // per-slot parity of this group's next barrier use
        int gnext = 0;      // group owning the next transform stage
        StageWalk<true> walk;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            int tile, k0, k1;
            unit_range(p, u, tile, k0, k1);
            const int mt = tile / p.num_n_tiles;
            const int nt = tile % p.num_n_tiles;
            const bool do_db = p.db != nullptr && nt == 0;
            walk.begin_tile(p, tile, k0);
            float acc0 = 0.f, acc1 = 0.f;
            // cos/sin of this thread's pairs for the token of the current stage
            float ci[PPI], si[PPI], cj[PPI], sj[PPI];
            int reg[8];
            int nreg = 0;
            {
                // rope regions of the tile, as offsets in its 128 rows
                int c0, c1;
                bool rp;
                tile_chunks(p, mt, c0, c1, rp);
                // (32-token stages, 4 threads per token row)
                {
                    int r0[8], r1[8];
                    const int n0r = rope_regions(p, c0, 64, r0), n1r = rope_regions(p, c1, 64, r1);
                    for (int j = 0; j < n0r && nreg < 8; ++j) reg[nreg++] = r0[j] - c0;
                    for (int j = 0; j < n1r && nreg < 8; ++j) reg[nreg++] = 64 + r1[j] - c1;
                }
            }
            for (int kt = k0; kt < k1; ++kt) {
                const bool nx = walk.needs(p, kt);
                walk.next(p);
                bool skip = !nx;
                if (nx) {
                    skip = gnext != grp;
                    gnext = (gnext + 1 == G) ? 0 : gnext + 1;
                }
                if (skip) {
                    if (++s == p.stages) s = 0;
                    continue;
                }
                const uint32_t xbar = sm.xfull(grp, s);
                const uint32_t xp = (xpar >> s) & 1u;
                xpar ^= 1u << s;
                bool wrote = false;
                {
                    const int64_t t = (int64_t)kt * BK + r;
                    bool mine = false;
                    for (int j = 0; j < nreg; ++j) mine |= ((j * IPR + kpart) % TPR == sub);
                    int prow = -1;
                    if (mine && t < p.T) {
                        prow = pos_row(p, t);
                        if (prow >= 0) {  // issued before the stage's data is awaited
                            const float* cr = p.cos_tab + (int64_t)prow * p.cs_width + pb;
                            const float* sr = p.sin_tab + (int64_t)prow * p.cs_width + pb;
#pragma unroll
                            for (int q = 0; q < PPI; q += 8) {
                                load8(cr + q, vec, ci + q);
                                load8(sr + q, vec, si + q);
                                load8(cr + HH + q, vec, cj + q);
                                load8(sr + HH + q, vec, sj + q);
                            }
                        }
                    }
                    const bool ok = mbar_wait(xbar, xp, abort_flag);
                    if (ok && prow >= 0) {
                        const uint32_t a0 = sm.a(s, p);
                        for (int j = 0; j < nreg; ++j) {
                            if ((j * IPR + kpart) % TPR != sub) continue;
                            const int o = reg[j];  // channel offset in the tile
                            const uint32_t row = a0 + (uint32_t)(o / 64) * CH + (uint32_t)r * 128;
                            const int q0 = (o % 64 + pb) / 8;
#pragma unroll
                            for (int g = 0; g < PPI / 8; ++g)
                                rot8(row, r, q0 + g, q0 + g + HH / 8, ci + 8 * g, si + 8 * g, cj + 8 * g,
                                     sj + 8 * g);
                            wrote = true;
                        }
                    }
                }
                if (wrote) fence_proxy_async_smem();
                if (do_db) {
                    // per-channel sums of the (rotated) tile: thread = channel pair
                    // pp of the 128, rows [BK/2 rh, BK/2 (rh + 1)) of the stage
                    named_bar_sync(1 + grp, GT);
                    const uint32_t a0 = sm.a(s, p);
                    const int pp = gt & 63, rh = (gt >> 6) & 1;
                    const uint32_t cbase = a0 + (uint32_t)(pp >> 5) * CH + (uint32_t)(pp & 3) * 4;
                    const int q16 = (pp & 31) >> 2;
#pragma unroll 8
                    for (int rr = 0; rr < BK / 2; ++rr) {
                        const int row = rh * (BK / 2) + rr;
                        const uint32_t v =
                            lds_b32(cbase + (uint32_t)row * 128 + (uint32_t)((q16 ^ (row & 7)) * 16));
                        acc0 += bf16lo_to_f32(v);
                        acc1 += bf16hi_to_f32(v);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.ready(s));
                if (++s == p.stages) s = 0;
            }
            if (do_db) {
                // combine the 2G partial sums of each channel, write bf16 db
                const int pp = gt & 63, rh = (gt >> 6) & 1;
                const int part = grp * 2 + rh;
                db_part[part * 128 + 2 * pp] = acc0;
                db_part[part * 128 + 2 * pp + 1] = acc1;
                named_bar_sync(1 + G, G * GT);
                if (part == 0) {
                    float s0 = 0.f, s1v = 0.f;
                    for (int q = 0; q < 2 * G; ++q) {
                        s0 += db_part[q * 128 + 2 * pp];
                        s1v += db_part[q * 128 + 2 * pp + 1];
                    }
                    int c0, c1;
                    bool rp;
                    tile_chunks(p, mt, c0, c1, rp);
                    const int64_t n = (int64_t)(pp < 32 ? c0 : c1) + 2 * (pp & 31);
                    const uint32_t packed = pack_bf16x2(s0, s1v);
                    if (n + 1 < p.N)
                        *reinterpret_cast<uint32_t*>(p.db + n) = packed;
                    else if (n < p.N)
                        p.db[n] = (uint16_t)(packed & 0xFFFFu);
                }
                named_bar_sync(1 + G, G * GT);
            }
        }
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

// ----------------------------------------------------------------- dgrad
// dgrad with separate rings for its two operands. A (dq tiles, 16 KB, the
// ones the transform rotates) has SA slots and its own producer; B (W
// chunks, BN/64 x 8 KB) has SB slots and another producer. With SA > SB a
// rope tile lands and is rotated up to SA stages before the MMA needs it,
// which hides the load + rotation latency that a shared ring of 48 KB stages
// (4 deep) exposed at every rope stage.
//
// Warps: 0 A producer, 1 MMA issuer, 2-5 epilogue, 6-13 transform (one
// group, two threads per token row), 14 B producer.
constexpr int kDgThreads = 480;
constexpr int kDgBWarp = 14;
constexpr uint32_t kDgABytes = (uint32_t)kBM * 128u;  // 128 token rows x 64 channels (bf16)

struct DgSmem {
    uint32_t abase, bbase, bars;
    int SA, SB;
    uint32_t bbytes;
    __device__ uint32_t a(int s) const { return abase + (uint32_t)s * kDgABytes; }
    __device__ uint32_t b(int s) const { return bbase + (uint32_t)s * bbytes; }
    // afull: A landed; aready: A rotated (transform stages); aempty: A consumed
    __device__ uint32_t afull(int s) const { return bars + 8u * s; }
    __device__ uint32_t aready(int s) const { return bars + 8u * (SA + s); }
    __device__ uint32_t aempty(int s) const { return bars + 8u * (2 * SA + s); }
    __device__ uint32_t bfull(int s) const { return bars + 8u * (3 * SA + s); }
    __device__ uint32_t bempty(int s) const { return bars + 8u * (3 * SA + SB + s); }
    __device__ uint32_t tfull(int b) const { return bars + 8u * (3 * SA + 2 * SB + b); }
    __device__ uint32_t tempty(int b) const { return bars + 8u * (3 * SA + 2 * SB + 2 + b); }
    __device__ uint32_t drain() const { return bars + 8u * (3 * SA + 2 * SB + 4); }
};
__host__ __device__ constexpr int dg_bar_count(int SA, int SB) { return 3 * SA + 2 * SB + 5; }

template <int DR>
__global__ void __launch_bounds__(kDgThreads, 1)
    dgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    DgSmem sm;
    sm.SA = p.sa_slots;
    sm.SB = p.sb_slots;
    sm.bbytes = p.b_bytes;
    sm.abase = (raw + 1023u) & ~1023u;
    sm.bbase = sm.abase + (uint32_t)sm.SA * kDgABytes;
    sm.bars = sm.bbase + (uint32_t)sm.SB * sm.bbytes;
    uint8_t* tail = smem_raw + (sm.bars - raw) + 8u * dg_bar_count(sm.SA, sm.SB);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(tail);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int BK = kBKD;
    constexpr uint32_t CHB = (uint32_t)BK * 128u;  // one 64-column chunk of B (BK rows)

    if (threadIdx.x == 0) {
        for (int s = 0; s < sm.SA; ++s) {
            mbar_init(sm.afull(s), 1);
            mbar_init(sm.aready(s), 8);  // the transform's 8 warps
            mbar_init(sm.aempty(s), 1);
        }
        for (int s = 0; s < sm.SB; ++s) {
            mbar_init(sm.bfull(s), 1);
            mbar_init(sm.bempty(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(sm.tfull(b), 1);
            mbar_init(sm.tempty(b), 4);
        }
        mbar_init(sm.drain(), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32((const void*)tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nb_chunks = p.BN / 64;

    if (warp == 0 || warp == kDgBWarp) {
        // ------------------------------------------- TMA producers (A / B)
        if (lane == 0) {
            const bool is_a = warp == 0;
            const int S = is_a ? sm.SA : sm.SB;
            int s = 0;
            uint32_t ph = 0, issued_mask = 0, issued_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x) {
                int tile, k0, k1;
                unit_range(p, u, tile, k0, k1);
                const int mt = tile / p.num_n_tiles, nt = tile % p.num_n_tiles;
                for (int kt = k0; kt < k1; ++kt) {
                    if (!mbar_wait(is_a ? sm.aempty(s) : sm.bempty(s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    if (is_a) {
                        // dq rows [mt*128, +128) x channels [kt*64, +64)
                        mbar_arrive_expect_tx(sm.afull(s), kDgABytes);
                        tma_load_2d(sm.a(s), &tmA, kt * BK, mt * kBM, sm.afull(s));
                    } else {
                        // W rows (channels) [kt*64, +64), columns in BN/64 chunks
                        mbar_arrive_expect_tx(sm.bfull(s), sm.bbytes);
                        if (p.b3d) {
                            tma_load_3d(sm.b(s), &tmB, 0, kt * BK, nt * nb_chunks, sm.bfull(s));
                        } else {
                            for (int c = 0; c < nb_chunks; ++c)
                                tma_load_2d(sm.b(s) + (uint32_t)c * CHB, &tmB, nt * p.BN + 64 * c, kt * BK,
                                            sm.bfull(s));
                        }
                    }
                    issued_mask |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                // unwinding: let every copy this thread started land before the CTA exits
                for (int q = 0; q < S; ++q)
                    if (issued_mask & (1u << q))
                        mbar_wait(is_a ? sm.afull(q) : sm.bfull(q), (issued_par >> q) & 1u, nullptr,
                                  200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int sa = 0, sb = 0;
            uint32_t pha = 0, phb = 0, rpar = 0;  // rpar: per-slot parity of aready
            int local = 0;
            StageWalk<false> walk;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < p.num_units; u += gridDim.x, ++local) {
                int tile, k0, k1;
                unit_range(p, u, tile, k0, k1);
                const int b = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!mbar_wait(sm.tempty(b), (use & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)b * kAccStride;
                walk.begin_tile(p, tile, k0);
                for (int kt = k0; kt < k1; ++kt, walk.next(p)) {
                    const bool xf = walk.needs(p, kt);
                    bool w = xf ? mbar_wait(sm.aready(sa), (rpar >> sa) & 1u, abort_flag)
                                : mbar_wait(sm.afull(sa), pha, abort_flag);
                    w = w && mbar_wait(sm.bfull(sb), phb, abort_flag);
                    if (!w) {
                        ok = false;
                        break;
                    }
                    if (xf) rpar ^= 1u << sa;
                    tc_fence_after();
                    const uint32_t a0 = sm.a(sa), b0 = sm.b(sb);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)
                        mma_bf16(d_tmem, desc_kmajor_sw128(a0 + 32u * j), desc_mnmajor_sw128(b0 + 2048u * j, CHB),
                                 p.idesc, (kt != k0 || j != 0));
                    mma_commit(sm.aempty(sa));
                    mma_commit(sm.bempty(sb));
                    if (++sa == sm.SA) {
                        sa = 0;
                        pha ^= 1u;
                    }
                    if (++sb == sm.SB) {
                        sb = 0;
                        phb ^= 1u;
                    }
                }
                if (ok) mma_commit(sm.tfull(b));
            }
            if (!ok) {
                mma_commit(sm.drain());
                mbar_wait(sm.drain(), 0, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp < kXformWarp0) {
        // ---------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        int local = 0;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x, ++local) {
            int tile, sp;
            unit_split(p, u, tile, sp);
            const int b = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            if (!mbar_wait(sm.tfull(b), use & 1u, abort_flag)) break;
            tc_fence_after();
            const int mt = tile / p.num_n_tiles;
            const int nt = tile % p.num_n_tiles;
            const int64_t orow = (int64_t)mt * kBM + row;  // token
            const bool valid = orow < p.out_rows;
            const uint32_t trow = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)b * kAccStride;
            for (int col = 0; col < p.BN; col += 32) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(trow + col, r);
                tmem_ld_wait();
                const int64_t c0 = (int64_t)nt * p.BN + col;
                if (valid && p.ws) {
                    // partial sum of split sp, fp32
                    float* dst = p.ws + ((int64_t)sp * p.out_rows + orow) * p.out_cols + c0;
#pragma unroll
                    for (int i = 0; i < 32; i += 4)
                        if (c0 + i + 4 <= p.out_cols) st_global_v4(dst + i, r[i], r[i + 1], r[i + 2], r[i + 3]);
                } else if (valid) {
                    uint16_t* dst = p.out + orow * p.out_cols + c0;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        if (c0 + i + 8 <= p.out_cols)
                            st_global_v4(dst + i,
                                         pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                         pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                         pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                                         pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(b));
        }
    } else {
        // --------------------------------------------------------- transform
        // inverse RoPE on the rope channels of each transform stage's A tile,
        // in place; thread = (token row r, sub) with TPR = 2 threads per row,
        // each taking PPI pairs of the regions assigned to it
        constexpr int HH = DR / 2;
        constexpr int TPR = 2;
        constexpr int PPI = (HH / TPR >= 8) ? HH / TPR : 8;
        constexpr int IPR = HH / PPI;
        constexpr int E = PPI / 8;  // groups of 8 pairs per item
        // A warp takes 16 token rows; lanes l and l + 16 share row l. The 8 lanes
        // of each 16-byte shared-memory access phase then sit on 8 different
        // rows, whose swizzled chunks fall in 8 different bank groups.
        const int xw = warp - kXformWarp0;  // 0..7
        const int r = xw * 16 + (lane & 15), sub = lane >> 4;
        const int kpart = sub % IPR;
        const int pb = kpart * PPI;
        const bool vec = p.cs_vec != 0;
        int sa = 0;
        uint32_t pha = 0;
        StageWalk<false> walk;
        for (int u = blockIdx.x; u < p.num_units; u += gridDim.x) {
            int tile, k0, k1;
            unit_range(p, u, tile, k0, k1);
            const int mt = tile / p.num_n_tiles;
            const int nt = tile % p.num_n_tiles;
            walk.begin_tile(p, tile, k0);
            // cos/sin of this thread's pairs for its token, kept for the whole unit
            float ci[PPI], si[PPI], cj[PPI], sj[PPI];
            int drow = -1;
            const int64_t tok = (int64_t)mt * kBM + r;
            if (tok < p.T) drow = pos_row(p, tok);
            if (drow >= 0) {
                const float* cr = p.cos_tab + (int64_t)drow * p.cs_width + pb;
                const float* sr = p.sin_tab + (int64_t)drow * p.cs_width + pb;
#pragma unroll
                for (int q = 0; q < PPI; q += 8) {
                    load8(cr + q, vec, ci + q);
                    load8(sr + q, vec, si + q);
                    load8(cr + HH + q, vec, cj + q);
                    load8(sr + HH + q, vec, sj + q);
                }
            }
            for (int kt = k0; kt < k1; ++kt) {
                const bool nx = walk.needs(p, kt);
                // first rope region of the stage, as an offset in its 64 channels; the
                // others follow every D channels (no array: local memory lives in L2 here)
                const int off0 = (walk.c0 <= p.Dn) ? (p.Dn - walk.c0) : (p.D + p.Dn - walk.c0);
                walk.next(p);
                if (nx) {
                    const bool ok = mbar_wait(sm.afull(sa), pha, abort_flag);
                    const uint32_t a0 = sm.a(sa);
                    // rotated values still to be stored to rope_out once the stage is
                    // released: at most two groups of 8 pairs per thread and stage
                    uint32_t v[2][8];
                    uint16_t* ga = nullptr;
                    uint16_t* gb = nullptr;
                    bool wrote = false;
                    int taken = 0;
                    int j = 0;
                    for (int off = off0; ok && drow >= 0 && off < BK && kt * BK + off < p.N; off += p.D, ++j) {
                        if ((j * IPR + kpart) % TPR != sub) continue;
                        const int q0 = (off + pb) / 8;
                        // rope_out[t, head, pb ...]: stored once per token, by the column
                        // tile nt = head mod (column tiles)
                        const int head = (kt * BK + off) / p.D;
                        uint16_t* g = (p.rope_out != nullptr && head % p.num_n_tiles == nt)
                                          ? p.rope_out + (tok * p.H + head) * DR + pb
                                          : nullptr;
                        if (E == 2 || taken == 0) {
#pragma unroll
                            for (int e = 0; e < E; ++e)
                                rot8(a0 + (uint32_t)r * 128, r, q0 + e, q0 + e + HH / 8, ci + 8 * e, si + 8 * e,
                                     cj + 8 * e, sj + 8 * e, v[e]);
                            ga = g;
                        } else {
                            rot8(a0 + (uint32_t)r * 128, r, q0, q0 + HH / 8, ci, si, cj, sj, v[1]);
                            gb = g;
                        }
                        ++taken;
                        wrote = true;
                    }
                    if (wrote) fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sm.aready(sa));
                    if (ga != nullptr) {  // after the release: off the MMA's path
#pragma unroll
                        for (int e = 0; e < E; ++e) {
                            st_global_v4(ga + 8 * e, v[e][0], v[e][1], v[e][2], v[e][3]);
                            st_global_v4(ga + 8 * e + HH, v[e][4], v[e][5], v[e][6], v[e][7]);
                        }
                    }
                    if (E == 1 && gb != nullptr) {
                        st_global_v4(gb, v[1][0], v[1][1], v[1][2], v[1][3]);
                        st_global_v4(gb + HH, v[1][4], v[1][5], v[1][6], v[1][7]);
                    }
                }
                if (++sa == sm.SA) {
                    sa = 0;
                    pha ^= 1u;
                }
            }
        }
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

// --------------------------------------------- dgrad with pre-rotated rope
// Rope pass: rope_out[t, h, :] = the inverse rotation of dq's last Dr = 64
// channels of head h (rope_inv8: the bits the fused transforms produce). A
// thread takes 8 pairs of one (token, head): 4 threads per pair set, a warp 8
// heads of one token (reads of 128 contiguous bytes per head, 1 KB written).
constexpr int kRopeHeads = 8;  // heads per thread in rope_pre_kernel (2, 4, 16 measured slower)

__global__ void __launch_bounds__(256) rope_pre_kernel(const uint16_t* __restrict__ dq, int64_t T, int H, int Dn,
                                                       const float* __restrict__ cos_tab,
                                                       const float* __restrict__ sin_tab, long long cs_rows,
                                                       long long cs_width, int cs_vec,
                                                       const int32_t* __restrict__ pos,
                                                       uint16_t* __restrict__ rope_out, int* status) {
    // A thread takes one quarter q of the 32 pairs (8 pairs) of kRopeHeads
    // heads of one token: the token's table entries are loaded once and used
    // for every head (the rows depend on the position only).
    constexpr int DR = 64, HH = 32;
    const int D = Dn + DR;
    const int nhg = (H + kRopeHeads - 1) / kRopeHeads;
    const int64_t items = T * nhg * 4;
    for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
         it += (int64_t)gridDim.x * blockDim.x) {
        const int q = (int)(it & 3);
        const int64_t tg = it >> 2;
        const int64_t t = tg / nhg;
        const int h0 = (int)(tg - t * nhg) * kRopeHeads;
        const int64_t pp = pos ? (int64_t)__ldg(pos + t) : t;
        if (pp < 0 || pp >= cs_rows) {
            record_status(status, MLA_ERR_POS_RANGE);
            continue;
        }
        uint4 ra[kRopeHeads], rc[kRopeHeads];
#pragma unroll
        for (int k = 0; k < kRopeHeads; ++k) {
            if (h0 + k < H) {
                const uint16_t* g = dq + (t * H + h0 + k) * D + Dn + 8 * q;
                ra[k] = __ldg(reinterpret_cast<const uint4*>(g));
                rc[k] = __ldg(reinterpret_cast<const uint4*>(g + HH));
            }
        }
        float ci[8], si[8], cj[8], sj[8];
        const float* cr = cos_tab + pp * cs_width + 8 * q;
        const float* sr = sin_tab + pp * cs_width + 8 * q;
        load8(cr, cs_vec != 0, ci);
        load8(sr, cs_vec != 0, si);
        load8(cr + HH, cs_vec != 0, cj);
        load8(sr + HH, cs_vec != 0, sj);
#pragma unroll
        for (int k = 0; k < kRopeHeads; ++k) {
            if (h0 + k < H) {
                const uint32_t g1[4] = {ra[k].x, ra[k].y, ra[k].z, ra[k].w};
                const uint32_t g2[4] = {rc[k].x, rc[k].y, rc[k].z, rc[k].w};
                uint32_t o1[4], o2[4];
                rope_inv8(g1, g2, ci, si, cj, sj, o1, o2);
                uint16_t* o = rope_out + (t * H + h0 + k) * DR + 8 * q;
                st_global_v4(o, o1[0], o1[1], o1[2], o1[3]);
                st_global_v4(o + HH, o2[0], o2[1], o2[2], o2[3]);
            }
        }
    }
}

// dgrad as a plain GEMM over [dq pass-through | rotated rope]: Dr = 64 and
// Dn % 64 == 0, so each 64-channel K chunk is all pass-through (A from dq) or
// all rope (A from rope_out, a {64, T, H} view). 256-token x BN tiles: two
// M = 128 MMAs per K step into TMEM columns 0 and 256 (one accumulator pair,
// not double-buffered; the segments are long), one ring of A + B stages.
// Warps: 0 producer, 1 MMA issuer, 2-5 epilogue of rows 0-127, 6-9 of rows
// 128-255 (warp w reads TMEM lanes 32 (w % 4) ...).
//
// Schedule (stream-K over groups): the CTAs form groups of num_n_tiles, CTA
// j of a group computing column tile j, so the CTAs of a group read the same
// dq rows at the same time and share them in L2. The groups split the
// (token tile, K step) iterations evenly: group g takes the contiguous range
// [sk_begin(g), sk_begin(g + 1)), in token-tile-major order. A range starts
// and ends anywhere inside a token tile, so a tile may be split between
// consecutive groups: the CTA holding the tile's first K step (its owner)
// finishes it. A CTA whose range starts inside a tile (its first segment;
// only that one can) writes that segment's fp32 partial sums to its own
// workspace slot and raises its flag; the owner, which reaches the tile at
// the end of its range, waits for the flags of the later CTAs of the same
// column (bounded), adds their partials in group order (deterministic) and
// writes dx. Partials are stored column-group-major: float4 (row, 4c..4c+3)
// at [c][row], so a warp's 32 rows of one float4 column are 512 contiguous
// bytes.
constexpr int kDpThreads = 320;
constexpr int kDpBM = 256;
constexpr uint32_t kDpABytes = (uint32_t)kDpBM * 128u;

// First (token tile, K step) iteration of group g (of `groups`), iterations
// token-tile major: sk_total = token tiles x K steps.
__device__ __forceinline__ long long sk_begin(const BwdParams& p, int g, int groups) {
    return p.sk_total * (long long)g / groups;
}

// The next segment [k0, k1) of token tile mt in a range that continues at
// iteration it (< end); advances it.
__device__ __forceinline__ void sk_segment(const BwdParams& p, long long& it, long long end, int& mt, int& k0,
                                           int& k1) {
    mt = (int)(it / p.k_tiles);
    k0 = (int)(it - (long long)mt * p.k_tiles);
    const long long left = end - it;
    k1 = left < (long long)(p.k_tiles - k0) ? k0 + (int)left : p.k_tiles;
    it += k1 - k0;
}

__global__ void __launch_bounds__(kDpThreads, 1)
    dgrad_pre_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmR, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.S = p.stages;
    sm.base = (raw + 1023u) & ~1023u;
    sm.bars = sm.base + (uint32_t)p.stages * p.stage_bytes;
    uint8_t* tail = smem_raw + (sm.bars - raw) + 8u * (3 * p.stages + 5);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(tail);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 4);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int BK = kBKD;
    constexpr uint32_t CHB = (uint32_t)BK * 128u;
    const int NT = p.num_n_tiles;
    const int groups = (int)gridDim.x / NT;
    const int grp = (int)blockIdx.x / NT;
    const int nt = (int)blockIdx.x - grp * NT;  // this CTA's column tile
    const long long beg = sk_begin(p, grp, groups), end = sk_begin(p, grp + 1, groups);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), 1);
        }
        mbar_init(sm.tfull(0), 1);
        mbar_init(sm.tempty(0), 8);
        mbar_init(sm.drain(), 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmR);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32((const void*)tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nb_chunks = p.BN / 64;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued_mask = 0, issued_par = 0;
            bool ok = true;
            // dq (and its rotated rope channels) stream through L2 once per
            // group; W is re-read by every group: keep W, let dq go first
            const uint64_t stream_pol = l2_evict_first_policy(), keep_pol = l2_evict_last_policy();
            for (long long it = beg; ok && it < end;) {
                int mt, k0, k1;
                sk_segment(p, it, end, mt, k0, k1);
                int c0 = (k0 * BK) % p.D, head = (k0 * BK) / p.D;  // chunk position, no division per stage
                for (int kt = k0; kt < k1; ++kt) {
                    if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(sm.full(s), p.tx_bytes);
                    if (c0 < p.Dn) tma_load_2d_hint(sm.a(s, p), &tmA, kt * BK, mt * kDpBM, sm.full(s), stream_pol);
                    else tma_load_3d_hint(sm.a(s, p), &tmR, 0, mt * kDpBM, head, sm.full(s), stream_pol);
                    tma_load_3d_hint(sm.b(s, p), &tmB, 0, kt * BK, nt * nb_chunks, sm.full(s), keep_pol);
                    issued_mask |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                    c0 += BK;
                    if (c0 >= p.D) {
                        c0 -= p.D;
                        ++head;
                    }
                }
            }
            if (!ok) {
                for (int q = 0; q < p.stages; ++q)
                    if (issued_mask & (1u << q))
                        mbar_wait(sm.full(q), (issued_par >> q) & 1u, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            bool ok = true;
            for (long long it = beg; ok && it < end; ++local) {
                int mt, k0, k1;
                sk_segment(p, it, end, mt, k0, k1);
                if (!mbar_wait(sm.tempty(0), ((uint32_t)local & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = k0; kt < k1; ++kt) {
                    if (!mbar_wait(sm.full(s), ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sm.a(s, p), b0 = sm.b(s, p);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j)
#pragma unroll
                        for (int hm = 0; hm < 2; ++hm)
                            mma_bf16(tmem_base + hm * kAccStride, desc_kmajor_sw128(a0 + hm * 16384u + 32u * j),
                                     desc_mnmajor_sw128(b0 + 2048u * j, CHB), p.idesc, (kt != k0 || j != 0));
                    mma_commit(sm.empty(s));
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) mma_commit(sm.tfull(0));
            }
            if (!ok) {
                mma_commit(sm.drain());
                mbar_wait(sm.drain(), 0, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        // The 8 warps agree through named barrier 1 (256 threads) on every
        // step that one of them may fail, so none waits at a barrier for a
        // warp that has left.
        const int quad = warp & 3;
        const int hm = (warp - 2) >> 2;  // which accumulator: token rows 0-127 or 128-255
        const int row = hm * 128 + quad * 32 + lane;
        const bool leader = threadIdx.x == 64;  // warp 2, lane 0: flag waits and writes
        const long long slot_floats = (long long)kDpBM * p.BN;
        float* my_slot = p.sk_slots ? p.sk_slots + (long long)blockIdx.x * slot_floats : nullptr;
        int local = 0;
        for (long long it = beg; it < end; ++local) {
            int mt, k0, k1;
            sk_segment(p, it, end, mt, k0, k1);
            bool ok = mbar_wait(sm.tfull(0), (uint32_t)local & 1u, abort_flag);
            if (!named_bar_and(1, 256, ok)) break;
            tc_fence_after();
            const bool contrib = k0 > 0;               // a later part of a split tile
            const bool owner = !contrib && k1 < p.k_tiles;  // a split tile's first part
            int g_last = grp;                          // the last group holding part of this tile
            if (owner) {
                const long long s_last = (long long)(mt + 1) * p.k_tiles - 1;
                g_last = (int)(((s_last + 1) * groups - 1) / p.sk_total);
                bool got = true;
                if (leader)
                    for (int g2 = grp + 1; got && g2 <= g_last; ++g2)
                        got = wait_flag_gpu(p.sk_flags + g2 * NT + nt, p.sk_epoch, abort_flag);
                if (!named_bar_and(1, 256, got)) g_last = grp;  // timed out: the status says so
            }
            const int64_t orow = (int64_t)mt * kDpBM + row;  // token
            const bool valid = orow < p.out_rows;
            const uint32_t trow = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)hm * kAccStride;
            for (int col = 0; col < p.BN; col += 32) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(trow + col, r);
                tmem_ld_wait();
                if (contrib) {
                    float4* dst = reinterpret_cast<float4*>(my_slot) + (int64_t)(col / 4) * kDpBM + row;
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[(int64_t)i * kDpBM] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                                              __uint_as_float(r[4 * i + 2]),
                                                              __uint_as_float(r[4 * i + 3]));
                    continue;
                }
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                for (int g2 = grp + 1; g2 <= g_last; ++g2) {
                    const float4* src = reinterpret_cast<const float4*>(p.sk_slots + (long long)(g2 * NT + nt) * slot_floats) +
                                        (int64_t)(col / 4) * kDpBM + row;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float4 a = __ldcg(src + (int64_t)i * kDpBM);
                        v[4 * i] += a.x;
                        v[4 * i + 1] += a.y;
                        v[4 * i + 2] += a.z;
                        v[4 * i + 3] += a.w;
                    }
                }
                const int64_t c0 = (int64_t)nt * p.BN + col;
                if (valid) {
                    uint16_t* dst = p.out + orow * p.out_cols + c0;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        if (c0 + i + 8 <= p.out_cols)
                            st_global_v4(dst + i, pack_bf16x2(v[i], v[i + 1]), pack_bf16x2(v[i + 2], v[i + 3]),
                                         pack_bf16x2(v[i + 4], v[i + 5]), pack_bf16x2(v[i + 6], v[i + 7]));
                    }
                }
            }
            tc_fence_before();
            if (contrib) {
                __threadfence();  // this thread's partials, before the flag
                named_bar_sync(1, 256);
                if (leader) st_release_gpu(p.sk_flags + blockIdx.x, p.sk_epoch);
            } else if (g_last > grp) {
                named_bar_sync(1, 256);  // every thread has read the partials
                if (leader)
                    for (int g2 = grp + 1; g2 <= g_last; ++g2) p.sk_flags[g2 * NT + nt] = 0u;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(0));
        }
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

// ------------------------------------- wgrad reading the rotated rope tiles
// The hand-off case (Dr = 64, Dn % 128 == 0, H even, dq_pre_rope given): dW
// as a plain GEMM over 256-channel tiles made of two 128-channel sub-tiles
// of the head-pair order (tile_chunks): each sub-tile is one 3-D TMA op,
// two pass-through chunks of dq or one head pair's rotated rope channels.
// Two M = 128 MMAs per K step (tokens) into TMEM columns 0 and 256; 64-token
// stages of A (4 MN-major chunks, 32 KB) and B (x, BN/64 chunks).
// Warps: 0 producer, 1 MMA, 2-9 epilogue (accumulator (w - 2) / 4, lanes
// 32 (w % 4)), 10-17 bias gradient: on the first column tile every stage's
// 256 channels are summed over its tokens (thread: 8 channels x 8 of the
// 64 token rows; the 8 row groups are added in order at the tile's end), and
// these warps release each stage together with the MMA.
constexpr int kWpThreads = 576;
constexpr int kWpDbWarp0 = 10;
constexpr int kWpBK = 64;

__global__ void __launch_bounds__(kWpThreads, 1)
    wgrad_pre_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmR, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    Smem sm;
    sm.S = p.stages;
    sm.base = (raw + 1023u) & ~1023u;
    sm.bars = sm.base + (uint32_t)p.stages * p.stage_bytes;
    uint8_t* tail = smem_raw + (sm.bars - raw) + 8u * (3 * p.stages + 5);
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(tail);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tail + 4);
    // bias partials: written by the 8 bias warps (dba), read by them (dbb)
    const uint32_t dba = smem_u32(tail + 16), dbb = smem_u32(tail + 24);
    float* db_part = reinterpret_cast<float*>(tail + 32);  // [8 row groups][256 channels]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int BK = kWpBK;
    constexpr uint32_t CH = (uint32_t)BK * 128u;  // one 64-channel MN-major chunk of BK rows
    const int n_sub = p.num_m_tiles;              // 128-channel sub-tiles
    const int num_m2 = (n_sub + 1) / 2;
    const int num_units = num_m2 * p.num_n_tiles;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(sm.full(s), 1);
            mbar_init(sm.empty(s), 1 + 8);  // the MMA's commit and the 8 bias warps
        }
        mbar_init(sm.tfull(0), 1);
        mbar_init(sm.tempty(0), 8);
        mbar_init(sm.drain(), 1);
        mbar_init(dba, 8);
        mbar_init(dbb, 8);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmR);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32((const void*)tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int nb_chunks = p.BN / 64;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0, issued_mask = 0, issued_par = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x) {
                const int m2 = u / p.num_n_tiles, nt = u % p.num_n_tiles;
                int az[2];
                bool rp[2], has[2];
                for (int hm = 0; hm < 2; ++hm) {
                    const int ms = 2 * m2 + hm;
                    has[hm] = ms < n_sub;
                    int c0 = 0, c1 = 0;
                    rp[hm] = false;
                    if (has[hm]) tile_chunks(p, ms, c0, c1, rp[hm]);
                    az[hm] = rp[hm] ? (c0 - p.Dn) / p.D : c0 / 64;
                }
                const uint32_t tx = p.tx_bytes - (has[1] ? 0u : 2u * CH);
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!mbar_wait(sm.empty(s), ph ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(sm.full(s), tx);
                    for (int hm = 0; hm < 2; ++hm)
                        if (has[hm])
                            tma_load_3d(sm.a(s, p) + (uint32_t)hm * 2u * CH, rp[hm] ? &tmR : &tmA, 0, kt * BK,
                                        az[hm], sm.full(s));
                    tma_load_3d(sm.b(s, p), &tmB, 0, kt * BK, nt * nb_chunks, sm.full(s));
                    issued_mask |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int q = 0; q < p.stages; ++q)
                    if (issued_mask & (1u << q))
                        mbar_wait(sm.full(q), (issued_par >> q) & 1u, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int local = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < num_units; u += gridDim.x, ++local) {
                if (!mbar_wait(sm.tempty(0), ((uint32_t)local & 1u) ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kt = 0; kt < p.k_tiles; ++kt) {
                    if (!mbar_wait(sm.full(s), ph, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sm.a(s, p), b0 = sm.b(s, p);
#pragma unroll
                    for (int j = 0; j < BK / 16; ++j) {
                        const uint64_t bd = desc_mnmajor_sw128(b0 + 2048u * j, CH);
#pragma unroll
                        for (int hm = 0; hm < 2; ++hm)
                            mma_bf16(tmem_base + hm * kAccStride,
                                     desc_mnmajor_sw128(a0 + (uint32_t)hm * 2u * CH + 2048u * j, CH), bd, p.idesc,
                                     (kt != 0 || j != 0));
                    }
                    mma_commit(sm.empty(s));
                    if (++s == p.stages) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (ok) mma_commit(sm.tfull(0));
            }
            if (!ok) {
                mma_commit(sm.drain());
                mbar_wait(sm.drain(), 0, nullptr, 200000000ull);
            }
        }
        __syncwarp();
    } else if (warp < kWpDbWarp0) {
        // ---------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int hm = (warp - 2) >> 2;
        const int row = quad * 32 + lane;
        int local = 0;
        for (int u = blockIdx.x; u < num_units; u += gridDim.x, ++local) {
            if (!mbar_wait(sm.tfull(0), (uint32_t)local & 1u, abort_flag)) break;
            tc_fence_after();
            const int m2 = u / p.num_n_tiles, nt = u % p.num_n_tiles;
            const int ms = 2 * m2 + hm;
            bool valid = ms < n_sub;
            int64_t orow = 0;
            if (valid) {
                int c0, c1;
                bool rp;
                tile_chunks(p, ms, c0, c1, rp);
                orow = (row < 64 ? c0 : c1) + (row & 63);  // output channel
                valid = orow < p.out_rows;
            }
            const uint32_t trow = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)hm * kAccStride;
            for (int col = 0; col < p.BN; col += 32) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(trow + col, r);
                tmem_ld_wait();
                const int64_t kc = (int64_t)nt * p.BN + col;
                if (valid) {
                    uint16_t* dst = p.out + orow * p.out_cols + kc;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        if (kc + i + 8 <= p.out_cols)
                            st_global_v4(dst + i,
                                         pack_bf16x2(__uint_as_float(r[i]), __uint_as_float(r[i + 1])),
                                         pack_bf16x2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])),
                                         pack_bf16x2(__uint_as_float(r[i + 4]), __uint_as_float(r[i + 5])),
                                         pack_bf16x2(__uint_as_float(r[i + 6]), __uint_as_float(r[i + 7])));
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.tempty(0));
        }
    } else {
        // ------------------------------------------------------ bias gradient
        const int dt = threadIdx.x - 32 * kWpDbWarp0;  // 0..255
        const int cg = dt & 31;                        // channels [8 cg, 8 cg + 8) of the tile's 256
        const int rg = dt >> 5;                        // token rows rg, rg + 8, ... of each stage
        const int chunk = cg >> 3, q = cg & 7;         // MN-major chunk, 16-byte group in its rows
        int s = 0;
        uint32_t ph = 0;
        uint32_t nsum = 0;  // tiles summed so far (the phase of dba / dbb)
        for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
            const int m2 = u / p.num_n_tiles, nt = u % p.num_n_tiles;
            const bool sum = p.db != nullptr && nt == 0;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            bool ok = true;
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!mbar_wait(sm.full(s), ph, abort_flag)) {
                    ok = false;
                    break;
                }
                if (sum) {
                    const uint32_t base = sm.a(s, p) + (uint32_t)chunk * CH;
#pragma unroll
                    for (int i = 0; i < BK / 8; ++i) {
                        const int r = rg + 8 * i;
                        uint32_t v[4];
                        lds_v4(base + (uint32_t)r * 128u + (uint32_t)((q ^ (r & 7)) * 16), v);
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            acc[2 * w] += bf16lo_to_f32(v[w]);
                            acc[2 * w + 1] += bf16hi_to_f32(v[w]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(sm.empty(s));
                if (++s == p.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            if (sum) {
                // the 8 row groups' partial sums added in order, one channel per thread; the
                // previous tile's readers are done with db_part first (dbb). Bounded waits.
                if (nsum > 0 && !mbar_wait(dbb, (nsum - 1) & 1u, abort_flag)) break;
#pragma unroll
                for (int e = 0; e < 8; ++e) db_part[rg * 256 + 8 * cg + e] = acc[e];
                __syncwarp();
                if (lane == 0) mbar_arrive(dba);
                if (!mbar_wait(dba, nsum & 1u, abort_flag)) break;
                const int c = dt;  // channel of the tile
                float tot = 0.f;
#pragma unroll
                for (int g = 0; g < 8; ++g) tot += db_part[g * 256 + c];
                const int ms = 2 * m2 + c / 128;
                if (ms < n_sub) {
                    int c0, c1;
                    bool rp;
                    tile_chunks(p, ms, c0, c1, rp);
                    const int cc = c & 127;
                    const int64_t ch = (cc < 64 ? c0 : c1) + (cc & 63);
                    if (ch < p.out_rows) p.db[ch] = (uint16_t)(pack_bf16x2(tot, 0.f) & 0xFFFFu);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(dbb);
                ++nsum;
            }
        }
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

// wgrad rotating dq itself (32-token stages)
int launch_wgrad_self(int Dr, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tr,
                      const BwdParams& p, int grid, size_t smem, cudaStream_t stream) {
    const void* k = nullptr;
    switch (Dr) {
        case 16: k = (const void*)wgrad_kernel<16, kBKW>; break;
        case 32: k = (const void*)wgrad_kernel<32, kBKW>; break;
        case 64: k = (const void*)wgrad_kernel<64, kBKW>; break;
        default: return MLA_ERR_UNSUPPORTED;
    }
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MLA_ERR_CUDA;
    switch (Dr) {
        case 16: wgrad_kernel<16, kBKW><<<grid, kWgThreads, smem, stream>>>(ta, tb, tr, p); break;
        case 32: wgrad_kernel<32, kBKW><<<grid, kWgThreads, smem, stream>>>(ta, tb, tr, p); break;
        default: wgrad_kernel<64, kBKW><<<grid, kWgThreads, smem, stream>>>(ta, tb, tr, p); break;
    }
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// wgrad with pre-rotated rope tiles: head pairs only, so Dr = 64
int launch_wgrad_pre(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tr, BwdParams p,
                     const DeviceInfo& di, cudaStream_t stream) {
    constexpr uint32_t CH = (uint32_t)kWpBK * 128u;
    p.a_bytes = 4u * CH;
    p.stage_bytes = p.a_bytes + (uint32_t)(p.BN / 64) * CH;
    p.tx_bytes = p.stage_bytes;
    const size_t fixed = 1024 + 256 + 8 * 256 * sizeof(float);  // alignment, barriers, bias partials
    int stages = (int)((size_t)(di.max_smem_optin - fixed) / p.stage_bytes);
    if (stages > 6) stages = 6;
    if (stages < 2) return MLA_ERR_UNSUPPORTED;
    p.stages = stages;
    const size_t smem = fixed + (size_t)stages * p.stage_bytes;
    const int units = ((p.num_m_tiles + 1) / 2) * p.num_n_tiles;
    const int grid = units < di.num_sms ? units : di.num_sms;
    if (cudaFuncSetAttribute(wgrad_pre_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MLA_ERR_CUDA;
    wgrad_pre_kernel<<<grid, kWpThreads, smem, stream>>>(ta, tb, tr, p);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

// dx = bf16(sum over splits of the fp32 partials), in split order (the
// result does not depend on which split finished first). 8 elements per
// thread: ksplit x two 16-byte loads, one 16-byte store.
__global__ void __launch_bounds__(256) dgrad_reduce_kernel(const float* __restrict__ ws, int ksplit,
                                                           int64_t n, uint16_t* __restrict__ dx) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; i < n; i += stride) {
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int sp = 0; sp < ksplit; ++sp) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(ws + sp * n + i));
            const float4 b = __ldg(reinterpret_cast<const float4*>(ws + sp * n + i) + 1);
            v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
            v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
        }
        st_global_v4(dx + i, pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                     pack_bf16x2(v[6], v[7]));
    }
}

// ------------------------------------------------ dgrad: which path, and its launch
// The pre-rotated path: Dr = 64 with Dn % 64 == 0 (64-channel K chunks are
// all pass-through or all rope), K % 64 == 0 (W's chunk view), and a
// workspace that holds its split partials plus, without dq_pre_rope, the
// rotated rope channels.
bool dgrad_pre_shape(int64_t K, int Dn, int Dr) { return Dr == 64 && Dn % 64 == 0 && K % 64 == 0; }

// The pre-rotated path's stream-K schedule for this shape: groups of
// num_n_tiles CTAs (at most the SM count, each group with at least
// kSkMinIters iterations), and whether a group boundary falls inside a token
// tile (then the workspace holds one flag and one fp32 partial tile per CTA).
constexpr long long kSkMinIters = 32;
struct SkLayout {
    int groups = 1, grid = 1;
    long long total = 0;
    bool split = false;
    size_t slots_off = 0, bytes = 0;  // flags at 0, slots at slots_off
};

SkLayout sk_layout(int64_t T, int64_t K, int64_t N, int num_sms) {
    SkLayout L;
    const int64_t bn = (K + 63) / 64 * 64;
    const int64_t BN = bn > 256 ? 256 : bn;
    const int NT = (int)((K + BN - 1) / BN);
    const int64_t KT = (N + kBKD - 1) / kBKD;
    L.total = ((T + kDpBM - 1) / kDpBM) * KT;
    long long groups = num_sms / NT;
    const long long by_work = L.total / kSkMinIters;
    if (groups > by_work) groups = by_work;
    if (groups < 1) groups = 1;
    L.groups = (int)groups;
    L.grid = (int)groups * NT;
    for (long long g = 1; g < groups && !L.split; ++g) L.split = (L.total * g / groups) % KT != 0;
    if (L.split) {
        L.slots_off = ((size_t)L.grid * 4 + 255) / 256 * 256;
        L.bytes = L.slots_off + (size_t)L.grid * kDpBM * (size_t)BN * sizeof(float);
    }
    return L;
}

size_t dgrad_pre_bytes(int64_t T, int64_t K, int64_t N, int H, int Dr, int num_sms, bool rope_buffer, size_t* rope_off) {
    const SkLayout L = sk_layout(T, K, N, num_sms);
    const size_t off = (L.bytes + 255) / 256 * 256;
    if (rope_off) *rope_off = off;
    return rope_buffer ? off + (size_t)T * H * Dr * 2 : L.bytes;
}

bool dgrad_pre_path(const BwdArgs& a, int num_sms) {
    if (a.T == 0 || !dgrad_pre_shape(a.K, a.Dn, a.Dr)) return false;
    const int64_t N = (int64_t)a.H * (a.Dn + a.Dr);
    const size_t need = dgrad_pre_bytes(a.T, a.K, N, a.H, a.Dr, num_sms, a.rope_out == nullptr, nullptr);
    return need == 0 || (a.workspace != nullptr && a.ws_bytes >= need);
}

// Flag value of a stream-K launch: new for every launch (never 0, the value
// the owners leave behind), so a flag left by an earlier launch is never
// taken for this one's.
unsigned next_sk_epoch() {
    static std::atomic<unsigned> counter{0x9E3779B9u};
    unsigned e;
    do {
        e = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
    } while (e == 0u);
    return e;
}

int launch_dgrad_pre(const BwdArgs& a, BwdParams& p, const DeviceInfo& di, cudaStream_t stream) {
    const int64_t N = p.N;
    size_t rope_off = 0;
    dgrad_pre_bytes(a.T, a.K, N, a.H, a.Dr, di.num_sms, true, &rope_off);
    uint16_t* rope = a.rope_out ? static_cast<uint16_t*>(a.rope_out)
                                : reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(a.workspace) + rope_off);
    // 1. the rope channels, rotated once
    {
        const int64_t items = a.T * ((a.H + kRopeHeads - 1) / kRopeHeads) * 4;
        int64_t blocks = (items + 255) / 256;
        if (blocks > (int64_t)di.num_sms * 8) blocks = (int64_t)di.num_sms * 8;
        rope_pre_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const uint16_t*>(a.dq), a.T, a.H, a.Dn,
                                                              a.cos_tab, a.sin_tab, a.cs_rows, a.cs_width, p.cs_vec,
                                                              a.pos, rope, a.status);
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
    }
    // 2. the GEMM over [pass-through | rotated rope], 256-token tiles, stream-K over groups
    p.num_m_tiles = (int)((a.T + kDpBM - 1) / kDpBM);
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    const SkLayout L = sk_layout(a.T, a.K, N, di.num_sms);
    p.sk_total = L.total;
    p.sk_flags = L.split ? static_cast<unsigned*>(a.workspace) : nullptr;
    p.sk_slots = L.split ? reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + L.slots_off) : nullptr;
    p.sk_epoch = next_sk_epoch();
    p.a_bytes = kDpABytes;
    p.stage_bytes = p.a_bytes + (uint32_t)(p.BN / 64) * (uint32_t)kBKD * 128u;
    p.tx_bytes = p.stage_bytes;
    const size_t fixed = 1024 + 256;
    int stages = (int)((size_t)(di.max_smem_optin - fixed) / p.stage_bytes);
    if (stages > 6) stages = 6;
    if (stages < 2) return MLA_ERR_UNSUPPORTED;
    p.stages = stages;
    const size_t smem = fixed + (size_t)stages * p.stage_bytes;
    alignas(64) CUtensorMap ta, tb, tr;
    int st = make_tmap_2d(&ta, a.dq, 1, (uint64_t)N, (uint64_t)a.T, (uint64_t)N * 2, 64, kDpBM, true);
    if (st != MLA_OK) return st;
    st = make_tmap_chunks(&tb, a.W, (uint64_t)N, (uint64_t)a.K, kBKD, (uint32_t)(p.BN / 64));
    if (st != MLA_OK) return st;
    st = make_tmap_3d(&tr, rope, 64, (uint64_t)a.T, (uint64_t)a.H, (uint64_t)a.H * 128, 128, 64, kDpBM, 1);
    if (st != MLA_OK) return st;
    if (cudaFuncSetAttribute(dgrad_pre_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return MLA_ERR_CUDA;
    // The owners of split tiles wait for other CTAs of the grid: launched
    // cooperatively, so all CTAs are resident together.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)L.grid);
    cfg.blockDim = dim3(kDpThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.split ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, dgrad_pre_kernel, ta, tb, tr, p) != cudaSuccess) return MLA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int launch_common(const BwdArgs& a, bool wg, cudaStream_t stream) {
    DeviceInfo di;
    int st = current_device_info(&di);
    if (st != MLA_OK) return st;
    const int D = a.Dn + a.Dr;
    const int64_t N = (int64_t)a.H * D;
    BwdParams p{};
    p.T = (int)a.T;
    p.K = (int)a.K;
    p.N = (int)N;
    p.D = D;
    p.Dn = a.Dn;
    int bn = (int)((a.K + 63) / 64) * 64;
    p.BN = bn > 256 ? 256 : bn;
    p.num_m_tiles = (int)(((wg ? N : a.T) + kBM - 1) / kBM);
    // wgrad: tiles by head pair when the rope part is one 64-channel chunk
    p.paired = wg && a.Dr == 64 && a.Dn % 128 == 0 && a.H % 2 == 0 && N % 64 == 0;
    if (p.paired) {
        p.tiles_per_pair = a.Dn / 64 + 1;
        p.num_m_tiles = (a.H / 2) * p.tiles_per_pair;
    }
    p.pre = p.paired && a.rope_in != nullptr && a.K % 64 == 0;  // its B loads use x's chunk view
    p.rope_out = wg ? nullptr : static_cast<uint16_t*>(a.rope_out);
    p.H = a.H;
    p.Dr = a.Dr;
    p.num_n_tiles = (int)((a.K + p.BN - 1) / p.BN);
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    const int BK = wg ? (p.pre ? kBKWPre : kBKW) : kBKD;
    const uint32_t CH = (uint32_t)BK * 128u;
    p.k_tiles = (int)(((wg ? a.T : N) + BK - 1) / BK);
    // A: 128 token rows of 64 channels (dgrad) or two 64-channel chunks of BK
    // token rows (wgrad); B: BN/64 chunks of BK rows
    p.a_bytes = wg ? 2u * CH : (uint32_t)kBM * 128u;
    p.stage_bytes = p.a_bytes + (uint32_t)(p.BN / 64) * CH;
    p.tx_bytes = p.stage_bytes;
    p.idesc = idesc_bf16(kBM, (uint32_t)p.BN, wg ? 1u : 0u, 1u);
    p.pos = a.pos;
    p.cos_tab = a.cos_tab;
    p.sin_tab = a.sin_tab;
    p.cs_rows = a.cs_rows;
    p.cs_width = a.cs_width;
    p.cs_vec = (a.cs_width % 4 == 0) && (reinterpret_cast<uintptr_t>(a.cos_tab) % 16 == 0) &&
               (reinterpret_cast<uintptr_t>(a.sin_tab) % 16 == 0);
    p.out = static_cast<uint16_t*>(wg ? a.dW : a.dx);
    p.out_rows = (int)(wg ? N : a.T);
    p.out_cols = (int)a.K;
    p.db = wg ? static_cast<uint16_t*>(a.db) : nullptr;
    p.status = a.status;
    if (!wg && dgrad_pre_path(a, di.num_sms)) return launch_dgrad_pre(a, p, di, stream);
    p.ksplit = wg ? 1 : dgrad_ksplit(a.T, a.K, N, di.num_sms);
    p.kts = (p.k_tiles + p.ksplit - 1) / p.ksplit;
    p.num_units = p.num_tiles * p.ksplit;
    p.ws = p.ksplit > 1 ? static_cast<float*>(a.workspace) : nullptr;
    if (p.ksplit > 1 && (!a.workspace || a.ws_bytes < dgrad_workspace_bytes_fused(a.T, a.K, N, di.num_sms)))
        return MLA_ERR_WORKSPACE;

    if (wg && a.T == 0) {  // empty reduction: the gradients are zero
        if (cudaMemsetAsync(a.dW, 0, (size_t)N * a.K * 2, stream) != cudaSuccess) return MLA_ERR_CUDA;
        if (a.db && cudaMemsetAsync(a.db, 0, (size_t)N * 2, stream) != cudaSuccess) return MLA_ERR_CUDA;
        return MLA_OK;
    }

    if (!wg) {
        // separate rings: 4 B slots, as many 16 KB A slots as fit (at most 12)
        const size_t fixed = 1024 + 512;  // alignment slack + barriers, TMEM slot, abort flag
        p.b_bytes = (uint32_t)(p.BN / 64) * CH;
        p.sb_slots = 4;
        const size_t room = (size_t)di.max_smem_optin - fixed - (size_t)p.sb_slots * p.b_bytes;
        int sa = (int)(room / (size_t)kBM / 128u);
        if (sa > 12) sa = 12;
        if (sa < p.sb_slots) return MLA_ERR_UNSUPPORTED;
        p.sa_slots = sa;
        const size_t smem = fixed + (size_t)sa * kBM * 128u + (size_t)p.sb_slots * p.b_bytes;
        alignas(64) CUtensorMap ta, tb;
        st = make_tmap_2d(&ta, a.dq, 1, (uint64_t)N, (uint64_t)a.T, (uint64_t)N * 2, 64, kBM, true);
        p.b3d = (a.K % 64 == 0) &&
                make_tmap_chunks(&tb, a.W, (uint64_t)N, (uint64_t)a.K, BK, (uint32_t)(p.BN / 64)) == MLA_OK;
        if (st == MLA_OK && !p.b3d)
            st = make_tmap_2d(&tb, a.W, 1, (uint64_t)a.K, (uint64_t)N, (uint64_t)a.K * 2, 64, BK, true);
        if (st != MLA_OK) return st;
        const int grid = p.num_units < di.num_sms ? p.num_units : di.num_sms;
        const void* k = nullptr;
        switch (a.Dr) {
            case 16: k = (const void*)dgrad_kernel<16>; break;
            case 32: k = (const void*)dgrad_kernel<32>; break;
            case 64: k = (const void*)dgrad_kernel<64>; break;
            default: return MLA_ERR_UNSUPPORTED;
        }
        if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return MLA_ERR_CUDA;
        switch (a.Dr) {
            case 16: dgrad_kernel<16><<<grid, kDgThreads, smem, stream>>>(ta, tb, p); break;
            case 32: dgrad_kernel<32><<<grid, kDgThreads, smem, stream>>>(ta, tb, p); break;
            default: dgrad_kernel<64><<<grid, kDgThreads, smem, stream>>>(ta, tb, p); break;
        }
        if (cudaGetLastError() != cudaSuccess) return MLA_ERR_CUDA;
        if (p.ksplit == 1) return MLA_OK;
        const int64_t n = a.T * a.K;
        int64_t blocks = (n / 8 + 255) / 256;
        if (blocks > (int64_t)di.num_sms * 8) blocks = (int64_t)di.num_sms * 8;
        dgrad_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p.ws, p.ksplit, n, static_cast<uint16_t*>(a.dx));
        return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
    }

    const size_t fixed = 1024 + 4096;  // alignment slack + barriers, slots, bias partials
    int stages = (int)((size_t)(di.max_smem_optin - fixed) / p.stage_bytes);
    if (stages > 12) stages = 12;
    if (stages < 2) return MLA_ERR_UNSUPPORTED;
    p.stages = stages;
    const size_t smem = fixed + (size_t)stages * p.stage_bytes;

    alignas(64) CUtensorMap ta, tb, tr;
    memset(&tr, 0, sizeof(tr));
    // one TMA operation per MN-major operand and stage when its columns come
    // in whole 64-element chunks; else one per chunk
    if (!wg) {
        st = make_tmap_2d(&ta, a.dq, 1, (uint64_t)N, (uint64_t)a.T, (uint64_t)N * 2, 64, kBM, true);
        p.b3d = (a.K % 64 == 0) &&
                make_tmap_chunks(&tb, a.W, (uint64_t)N, (uint64_t)a.K, BK, (uint32_t)(p.BN / 64)) == MLA_OK;
        if (st == MLA_OK && !p.b3d)
            st = make_tmap_2d(&tb, a.W, 1, (uint64_t)a.K, (uint64_t)N, (uint64_t)a.K * 2, 64, BK, true);
    } else {
        p.a3d = (N % 128 == 0) && make_tmap_chunks(&ta, a.dq, (uint64_t)a.T, (uint64_t)N, BK, 2) == MLA_OK;
        if (p.paired) {
            // rope tiles: {64 rope channels, T tokens, H heads} views of the
            // rotated buffer [T, H, 64] or of dq (head stride D channels)
            const int r = p.pre ? make_tmap_3d(&tr, a.rope_in, 64, (uint64_t)a.T, (uint64_t)a.H,
                                               (uint64_t)a.H * 128, 128, 64, BK, 2)
                                : make_tmap_3d(&tr, static_cast<const uint16_t*>(a.dq) + a.Dn, 64, (uint64_t)a.T,
                                               (uint64_t)a.H, (uint64_t)N * 2, (uint64_t)D * 2, 64, BK, 2);
            if (r != MLA_OK) return MLA_ERR_CUDA;
            if (!p.a3d) return MLA_ERR_CUDA;  // paired tiles load pass-through chunks with the chunk view
        }
        if (!p.a3d) st = make_tmap_2d(&ta, a.dq, 1, (uint64_t)N, (uint64_t)a.T, (uint64_t)N * 2, 64, BK, true);
        p.b3d = (a.K % 64 == 0) &&
                make_tmap_chunks(&tb, a.x, (uint64_t)a.T, (uint64_t)a.K, BK, (uint32_t)(p.BN / 64)) == MLA_OK;
        if (st == MLA_OK && !p.b3d)
            st = make_tmap_2d(&tb, a.x, 1, (uint64_t)a.K, (uint64_t)a.T, (uint64_t)a.K * 2, 64, BK, true);
    }
    if (st != MLA_OK) return st;
    const int grid = p.num_units < di.num_sms ? p.num_units : di.num_sms;
    st = p.pre ? launch_wgrad_pre(ta, tb, tr, p, di, stream)
               : launch_wgrad_self(a.Dr, ta, tb, tr, p, grid, smem, stream);
    if (st != MLA_OK || p.ksplit == 1) return st;
    const int64_t n = a.T * a.K;
    int64_t blocks = (n / 8 + 255) / 256;
    if (blocks > (int64_t)di.num_sms * 8) blocks = (int64_t)di.num_sms * 8;
    dgrad_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p.ws, p.ksplit, n, static_cast<uint16_t*>(a.dx));
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

// Splits of each dgrad tile's channel reduction: the count in 1..4 (keeping
// >= 32 stages per split) whose units fill the SMs' waves best; ties go to
// fewer splits. 1 means no split (and no workspace).
int best_ksplit(int64_t tiles, int64_t k_tiles, int num_sms) {
    if (num_sms <= 0) return 1;
    int best = 1;
    double best_eff = 0.0;
    for (int sp = 1; sp <= 4; ++sp) {
        if (sp > 1 && k_tiles / sp < 32) break;
        const int64_t units = tiles * sp;
        const int64_t waves = (units + num_sms - 1) / num_sms;
        const double eff = (double)units / (double)(waves * num_sms);
        if (eff > best_eff + 1e-9) {
            best_eff = eff;
            best = sp;
        }
    }
    return best;
}

int dgrad_ksplit(int64_t T, int64_t K, int64_t N, int num_sms) {
    return best_ksplit(((T + kBM - 1) / kBM) * ((K + 255) / 256), (N + kBKD - 1) / kBKD, num_sms);
}

size_t dgrad_workspace_bytes_fused(int64_t T, int64_t K, int64_t N, int num_sms) {
    const int sp = dgrad_ksplit(T, K, N, num_sms);
    return sp > 1 ? (size_t)sp * (size_t)T * (size_t)K * sizeof(float) : 0;
}

size_t dgrad_workspace_bytes(int64_t T, int64_t K, int H, int Dn, int Dr, int num_sms) {
    const int64_t N = (int64_t)H * (Dn + Dr);
    if (T > 0 && dgrad_pre_shape(K, Dn, Dr)) return dgrad_pre_bytes(T, K, N, H, Dr, num_sms, true, nullptr);
    return dgrad_workspace_bytes_fused(T, K, N, num_sms);
}

size_t dgrad_pre_shape_bytes(int64_t T, int64_t K, int H, int Dn, int Dr, int num_sms, bool have_rope_out) {
    if (T == 0 || !dgrad_pre_shape(K, Dn, Dr)) return (size_t)-1;  // no such path
    const int64_t N = (int64_t)H * (Dn + Dr);
    return dgrad_pre_bytes(T, K, N, H, Dr, num_sms, !have_rope_out, nullptr);
}

size_t dgrad_min_workspace_bytes(int64_t T, int64_t K, int H, int Dn, int Dr, int num_sms, bool have_rope_out) {
    const int64_t N = (int64_t)H * (Dn + Dr);
    const size_t fused = dgrad_workspace_bytes_fused(T, K, N, num_sms);
    if (T > 0 && dgrad_pre_shape(K, Dn, Dr)) {
        const size_t pre = dgrad_pre_bytes(T, K, N, H, Dr, num_sms, !have_rope_out, nullptr);
        return pre < fused ? pre : fused;
    }
    return fused;
}

int launch_dgrad(const BwdArgs& a, cudaStream_t stream) { return launch_common(a, false, stream); }
int launch_wgrad(const BwdArgs& a, cudaStream_t stream) { return launch_common(a, true, stream); }

}  // namespace mlaq
