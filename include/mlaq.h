/*
 * mlaq.h: C ABI of libmlaq.so, the GB300 (sm_103a) fused MLA query
 * up-projection.
 *
 * The operation (TransformerEngine PR "Add support for fused Q Up-Proj
 * GEMM/RoPE/Quant", description paragraph): the Q up-projection GEMM of
 * DeepSeek-V3-style Multi-Latent Attention, fused with the RoPE that follows
 * it and with MXFP8 quantization of the result, with either a 16-bit or an
 * MXFP8 projection weight. Its backward (TransformerEngine PR "Add a
 * backwards linear function to be used with the fused mla q up-proj",
 * sequence diagram): the query gradient goes through the RoPE backward, then
 * the linear backward yields the input, weight and bias gradients.
 *
 * Notation: T tokens, K = q_lora_rank, H heads, each of D = Dn + Dr channels
 * (Dn pass-through, Dr rotated), N = H * D.
 *   forward   y[t, n] = sum_k x[t, k] W[n, k] + b[n]
 *             q[t, h, c] = y[t, hD + c]                           for c < Dn
 *             q[t, h, Dn+i]      = a cos[p, i]      - c sin[p, i]
 *             q[t, h, Dn+i+Dr/2] = c cos[p, i+Dr/2] + a sin[p, i+Dr/2]
 *             with a = y[t, hD+Dn+i], c = y[t, hD+Dn+i+Dr/2], i < Dr/2,
 *             p = pos[t] (or t), optionally MXFP8-quantized per 32 channels
 *             of each head (E4M3 codes + one E8M0 scale per block).
 *   backward  dq_pre = J^T dq (J the Jacobian of the rotation above)
 *             dx = dq_pre W,  dW = dq_pre^T x,  db = sum_t dq_pre.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     allocates nothing and keeps no state between calls.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without synchronizing.
 *   - The return value is a synchronous mla_status. Nothing is launched when
 *     it is not MLA_OK. Conditions only the GPU can see (a position outside
 *     the cos/sin table, a pipeline wait that timed out) are written to
 *     *dev_status (a device int the caller zeroes before the call; NULL = not
 *     reported); the first one recorded wins.
 *   - Inputs are never written. Outputs must not overlap any input
 *     (MLA_ERR_ALIAS); the Megatron-LM PR "Fix fused MLA YaRN RoPE query
 *     kernel corrupting upstream tensor in-place" is about exactly this
 *     in-place hazard.
 *   - bf16 means IEEE-754 binary16 with 8 exponent bits (bfloat16), stored as
 *     uint16 bit patterns; all row-major, innermost dimension contiguous.
 */
#ifndef MLAQ_H
#define MLAQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLAQ_API __attribute__((visibility("default")))
#else
#define MLAQ_API
#endif

/* Status codes. */
enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1, /* null required pointer, bad mode, non-positive dims, odd Dr, ... */
    MLA_ERR_ROPE_WIDTH = 2,  /* cos/sin table narrower than Dr: rejected, never read past a row */
    MLA_ERR_ALIGNMENT = 3,   /* pointer or row pitch not aligned as the kernel's loads need */
    MLA_ERR_ALIAS = 4,       /* an output byte range overlaps an input byte range */
    MLA_ERR_UNSUPPORTED = 5, /* a valid problem the kernels do not tile (see each call) */
    MLA_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed (no device, launch error) */
    MLA_ERR_TIMEOUT = 7,     /* device only: a pipeline wait gave up; outputs are unspecified */
    MLA_ERR_POS_RANGE = 8,   /* a position outside [0, cs_rows); device-side for pos arrays */
    MLA_ERR_WORKSPACE = 9    /* workspace pointer/size smaller than the size query returned */
};

/* weight_mode */
enum { MLA_WEIGHT_BF16 = 0, MLA_WEIGHT_MXFP8 = 1, MLA_WEIGHT_MXFP8_TILED = 2 };
/* out_mode */
enum { MLA_OUT_BF16 = 0, MLA_OUT_MXFP8 = 1, MLA_OUT_MXFP8_BHSD = 2, MLA_OUT_MXFP8_BHSD_SWIZZLED = 3 };
/* in_dtype of mxfp8_quantize_rows */
enum { MLA_IN_F32 = 0, MLA_IN_BF16 = 1 };

/* Problem shape.
 *   T        tokens (rows of x and q), >= 0
 *   K        q_lora_rank (columns of x and W), > 0
 *   H        heads, > 0
 *   Dn       pass-through channels per head, >= 0
 *   Dr       rotated channels per head, even, > 0
 *   cs_rows  rows of the cos and sin tables (positions)
 *   cs_width columns of the tables = their row pitch in floats; must be >= Dr
 *   T, K, H * (Dn + Dr), cs_rows and cs_width are at most INT32_MAX, else
 *   MLA_ERR_INVALID_ARG
 *            (the width guard of the Megatron-LM PR above: a narrow table
 *            gives MLA_ERR_ROPE_WIDTH, never an out-of-bounds read). Rope
 *            channel j of a head reads column j. */
typedef struct {
    int64_t T;
    int64_t K;
    int32_t H;
    int32_t Dn;
    int32_t Dr;
    int32_t reserved; /* set to 0 */
    int64_t cs_rows;
    int64_t cs_width;
} mla_q_shape;

/*
 * Forward: q = RoPE(x W^T + b), optionally MXFP8-quantized.
 * TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
 * description paragraph and flowchart (input activation, BF16 or MXFP8
 * weight and RoPE cos/sin into the fused up-projection, MXFP8 query out).
 *
 *   weight_mode MLA_WEIGHT_BF16:  x [T, K] bf16, W [N, K] bf16; x_scales and
 *               w_scales must be NULL.
 *   weight_mode MLA_WEIGHT_MXFP8: x [T, K] E4M3 codes (uint8) with x_scales
 *               [T, K/32] E8M0 bytes, W [N, K] E4M3 codes with w_scales
 *               [N, K/32]: value = e4m3(code) * 2^(scale - 127), blocks of 32
 *               along K (the layout mxfp8_quantize_rows writes).
 *               Requires K % 128 == 0.
 *   weight_mode MLA_WEIGHT_MXFP8_TILED: the same codes, with both scale
 *               tensors already in the tiled order the block-scaled GEMM reads,
 *               so they arrive by bulk copies instead of a per-row gather (the
 *               same outputs, bit for bit, in less time):
 *               x_scales = mxfp8_swizzle_scales of the [T, K/32] scales
 *               (mxfp8_swizzled_scale_bytes(T, K/32) bytes; or written so
 *               directly by mxfp8_quantize_rows_tiled, group 128); w_scales =
 *               mxfp8_swizzle_scales_grouped of the [N, K/32] scales with
 *               group = mla_q_uproj_w_scale_group(shape) (the kernel's
 *               channel tile; mxfp8_grouped_scale_bytes(N, K/32, group)
 *               bytes). W is a weight: its tiled scales are prepared once.
 *               Both 16-byte aligned.
 *   bias        [N] bf16 or NULL (added before the rotation).
 *   cos_tab, sin_tab [cs_rows, cs_width] fp32.
 *   pos         [T] int32 positions, or NULL for pos[t] = t (then
 *               T <= cs_rows is checked here, else MLA_ERR_POS_RANGE).
 *   out_mode MLA_OUT_BF16:  q_out [T, H, D] bf16 (round to nearest even);
 *               q_scales_out must be NULL.
 *   out_mode MLA_OUT_MXFP8: q_out [T, H, D] E4M3 codes (uint8) and
 *               q_scales_out [T, H, ceil(D/32)] E8M0 bytes; blocks of 32
 *               consecutive channels of one head (the last may be partial);
 *               scale exponent = the smallest e with amax <= 448 * 2^e,
 *               clamped to [-127, 127]; codes = RNE E4M3 of v * 2^-e with
 *               saturation; a block holding NaN/Inf gets scale 0xFF and NaN
 *               codes.
 *   out_mode MLA_OUT_MXFP8_BHSD: the same codes, with the scales written
 *               head-major, q_scales_out [H, T, ceil(D/32)] (the BHSD scale
 *               order an attention kernel reading one head at a time wants;
 *               TransformerEngine PR "Add support for fused Q Up-Proj
 *               GEMM/RoPE/Quant", review thread: the BHSD scale transpose).
 *   out_mode MLA_OUT_MXFP8_BHSD_SWIZZLED: the same codes; each head's
 *               scales [T, ceil(D/32)] leave the epilogue already in the
 *               tiled order a block-scaled GEMM reads, i.e. the layout
 *               mxfp8_swizzle_scales gives that head's matrix. Head h takes
 *               bytes [h * S, (h + 1) * S), S = mxfp8_swizzled_scale_bytes(T,
 *               ceil(D/32)); the padding of the last row tile (rows T ..)
 *               and of the last column tile is written as 0. This fuses
 *               into the forward the step that the same PR's flowchart puts
 *               between the quantized query and the fused attention: scales
 *               moved to head-major order and tiled for the GEMM.
 * Tiling limits (else MLA_ERR_UNSUPPORTED): Dr in {16, 32, 64}, Dn % 32 == 0,
 * and some channel tile width must divide N while keeping every head's rope
 * region and every 32-channel block whole: a multiple of 16 up to 256 with
 * bf16 weights, a multiple of 32 up to 192 with MXFP8 weights (one head
 * always qualifies when D fits; mla_q_uproj_w_scale_group reports the MXFP8
 * one, 0 when none). bf16 weights need K % 8 == 0 (16-byte rows). Pointers
 * must be 16-byte aligned (scales: 4-byte, tiled scales 16-byte; bias:
 * 16-byte), else MLA_ERR_ALIGNMENT.
 */
MLAQ_API int mla_q_uproj_fwd(const mla_q_shape *shape, int weight_mode, int out_mode,
                             const void *x, const uint8_t *x_scales, const void *W,
                             const uint8_t *w_scales, const void *bias, const float *cos_tab,
                             const float *sin_tab, const int32_t *pos, void *q_out,
                             uint8_t *q_scales_out, int *dev_status, void *stream);

/*
 * The per-position rotary table in the layout the forward's epilogue reads
 * fastest (an addition of this library; the pages only name the cos/sin
 * cache, Megatron-LM PR "Fix fused MLA YaRN RoPE query kernel corrupting
 * upstream tensor in-place", Problem section). For i < Dr/2 and p < cs_rows,
 * packed[i][p] is the float4 (cos[p][i], sin[p][i], cos[p][i + Dr/2],
 * sin[p][i + Dr/2]): the four values that rotate pair i of a token at
 * position p, with the entries of consecutive positions adjacent. It holds
 * the table's first Dr columns, copied bit for bit (no arithmetic).
 *   cos_tab/sin_tab [cs_rows, cs_width] fp32 (row pitch cs_width >= Dr, else
 *   MLA_ERR_ROPE_WIDTH), packed: mla_rope_table_packed_bytes(cs_rows, Dr)
 *   bytes, 16-byte aligned, overlapping neither table (MLA_ERR_ALIAS).
 *   Enqueued on `stream`; cs_rows = 0 is a no-op. Dr must be even and > 0.
 * A table is a model constant: pack it once and pass it to every
 * mla_q_uproj_fwd_packed call.
 */
MLAQ_API size_t mla_rope_table_packed_bytes(int64_t cs_rows, int Dr);
MLAQ_API int mla_rope_table_pack(int64_t cs_rows, int64_t cs_width, int Dr, const float *cos_tab,
                                 const float *sin_tab, float *packed, void *stream);

/*
 * mla_q_uproj_fwd with the rotary table packed by mla_rope_table_pack
 * (rope_packed, 16-byte aligned, shape->cs_rows positions; shape->cs_width
 * is the width of the table it was packed from and must be >= Dr). Same
 * arguments otherwise, same checks, same results bit for bit: only the
 * table's memory layout differs, so a warp's table reads for 32 tokens at
 * consecutive positions are 512 contiguous bytes instead of 32 rows.
 */
MLAQ_API int mla_q_uproj_fwd_packed(const mla_q_shape *shape, int weight_mode, int out_mode,
                                    const void *x, const uint8_t *x_scales, const void *W,
                                    const uint8_t *w_scales, const void *bias, const float *rope_packed,
                                    const int32_t *pos, void *q_out, uint8_t *q_scales_out,
                                    int *dev_status, void *stream);

/*
 * Backward, input gradient: dx = (J^T dq) W.
 * TransformerEngine PR "Add a backwards linear function to be used with the
 * fused mla q up-proj", summary and sequence diagram (RoPE backward, then the
 * linear backward with the weight). Only the rope channels of dq change under
 * the inverse rotation; the pass-through channels go to the tensor cores as
 * they are, and at most the rotated rope channels are ever stored.
 *   dq [T, H, D] bf16, W [N, K] bf16 (the bf16 master weight), dx [T, K] bf16
 *   (fp32 accumulation). cos_tab/sin_tab/pos as in the forward.
 *   dq_pre_rope: NULL, or [T, H, Dr] bf16 (16-byte aligned, not overlapping
 *   anything else) that receives the rope channels of dq_pre = J^T dq, the
 *   last Dr channels of every head after the inverse rotation, rounded to
 *   bf16: exactly the values the tensor cores consume. Pass it on to
 *   mla_q_uproj_bwd_wgrad, which then skips its own rotation. Rows whose
 *   position is out of range are left unwritten and their dx is unspecified
 *   (dev_status reports it).
 *   workspace/ws_bytes: device scratch, 16-byte aligned, not overlapping any
 *   input or output (NULL/0 when the size query returns 0). Two paths:
 *   - with at least mla_q_uproj_workspace_size(shape, 1) bytes, and when
 *     Dr == 64, Dn % 64 == 0, K % 64 == 0: a pass of its own rotates the
 *     rope channels into dq_pre_rope (or, when that is NULL, into the
 *     workspace), then a plain GEMM over [pass-through | rotated] channels
 *     runs on 256-token tiles (fewer operand bytes per FLOP);
 *   - otherwise (at least mla_q_uproj_workspace_size(shape, 4) bytes) the
 *     rotation happens in shared memory between the operand load and the
 *     tensor cores.
 *   Both round the rotated values to bf16 by the same formula. When the
 *   tiles of dx are too few to fill the GPU's SMs evenly, each tile's
 *   reduction over channels is split into parts that write fp32 partial
 *   sums in the workspace; a second kernel on the same stream adds them in
 *   a fixed order (results do not depend on scheduling) and rounds to bf16.
 *   The contents need no initialization and are garbage afterwards; calls
 *   that share a workspace must not overlap on the GPU.
 * Requires K % 8 == 0, Dr in {16, 32, 64}, Dn % Dr == 0, and 16-byte aligned
 * pointers.
 */
MLAQ_API int mla_q_uproj_bwd_dgrad(const mla_q_shape *shape, const void *dq, const void *W,
                                   const float *cos_tab, const float *sin_tab, const int32_t *pos,
                                   void *dx, void *dq_pre_rope, void *workspace, size_t ws_bytes,
                                   int *dev_status, void *stream);

/*
 * Backward, weight and bias gradients: dW = (J^T dq)^T x, db = sum_t J^T dq.
 * Same pull request (input and weight gradients from the saved input), its
 * review comment "BF16 bias gradient remains missing" (db belongs here), and
 * the Megatron-LM PR above (wgrad dw = dy^T x uses the linear's saved INPUT;
 * it may run later, as a separate call, for delayed weight-gradient
 * schedules).
 *   dq [T, H, D] bf16, x [T, K] bf16, dW [N, K] bf16, db [N] bf16 or NULL
 *   (skipped). fp32 accumulation over all T.
 *   dq_pre_rope: NULL (the rope channels of dq are rotated here, on their way
 *   into the tensor cores), or the buffer mla_q_uproj_bwd_dgrad filled from
 *   the same dq, positions and tables (an input here). When Dr == 64,
 *   Dn % 128 == 0, H is even and K % 64 == 0, the rope tiles are then read
 *   from it instead of rotated again (and dW runs on 256-channel tiles);
 *   other shapes rotate dq as with NULL. Either way the operands, and so
 *   dW, are the same bits; db's fp32 sums are grouped differently.
 *   workspace/ws_bytes: unused (NULL/0; mla_q_uproj_workspace_size(shape, 2)
 *   is 0).
 * Requirements as for mla_q_uproj_bwd_dgrad.
 */
MLAQ_API int mla_q_uproj_bwd_wgrad(const mla_q_shape *shape, const void *dq, const void *dq_pre_rope,
                                   const void *x, const float *cos_tab, const float *sin_tab,
                                   const int32_t *pos, void *dW, void *db, void *workspace,
                                   size_t ws_bytes, int *dev_status, void *stream);

/*
 * Backward with MXFP8 tensor-core GEMMs: dx, dW and db from dq in one call.
 * TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
 * Greptile summary: the MXFP8 quantization helpers (rowwise, the transpose
 * copy) that feed block-scaled GEMMs; the pages give no formula for the
 * backward, so this follows the plain reading (each GEMM operand quantized
 * along its reduction dimension):
 *   dq_pre = J^T dq in float32: the Dn pass-through channels of each head as
 *            they are; rope channel pairs (i, i + Dr/2) of head h, token t,
 *            position p = pos[t] (or t), with c_j = cos_tab[p][j] and
 *            s_j = sin_tab[p][j]:
 *              out_i        = fl(fl(g_i c_i) + fl(g_{i+Dr/2} s_{i+Dr/2}))
 *              out_{i+Dr/2} = fl(fl(g_{i+Dr/2} c_{i+Dr/2}) - fl(g_i s_i))
 *            (each product and sum rounded once to float32, in that order)
 *   dx [T, K]  = Q_rows(dq_pre) [T, N] . Q_cols(W)^T, reduced over N
 *   dW [N, K]  = Q_cols(dq_pre) [N, T] . Q_cols(x)^T, reduced over T
 *   db [N]     = sum over t of dq_pre (float32 sums of 32-token blocks,
 *                added in token-block order, rounded to bf16)
 * Q_rows is mxfp8_quantize_rows' rule on rows, Q_cols its rule on columns
 * (mxfp8_quantize_cols); the GEMMs accumulate exact products of the decoded
 * operands in fp32 and round once to bf16.
 *   dq [T, H, D] bf16, W [N, K] bf16, x [T, K] bf16; dx [T, K], dW [N, K],
 *   db [N] bf16. dx, dW and db are each optional (NULL: not computed; at
 *   least one is required); W may be NULL without dx, x without dW.
 *   workspace: at least mla_q_uproj_workspace_size(shape, 3) bytes,
 *   16-byte aligned, overlapping nothing else. After the call it holds the
 *   quantized operands at the offsets mla_q_uproj_bwd_mxfp8_layout gives
 *   (only those of the requested gradients), e.g. for reuse or inspection;
 *   nothing in it needs initialization.
 * Requires Dr in {32, 64} with (Dn + Dr) % 32 == 0 (a rowwise block never
 * spans two heads), N % 128 == 0, K % 32 == 0 (else MLA_ERR_UNSUPPORTED);
 * 16-byte aligned dq, W, x, dx, dW. T may be any size >= 0: the token axis
 * of the wgrad operands is padded to a multiple of 128 with zero codes and
 * zero scale bytes. T == 0 writes dW = 0 and db = 0.
 */
/*
 * The scale arrays of mla_mxfp8_bwd_layout are in the tiled order the
 * block-scaled GEMMs load (one bulk copy per 128 rows and K step): for an
 * operand with `rows` rows and `cols` scale columns (cols = its K / 32),
 * rows go in groups of G (G = 128 for operand A, b_group for operand B);
 * each group is padded to whole 128-row chunks; chunk i of group g, K step
 * kt (scale columns 4kt .. 4kt+3) is the 512-byte tile
 * ((g * ceil(G/128) + i) * ceil(cols/4) + kt), and inside it row rr of the
 * chunk, column c sits at byte (rr % 32) * 16 + (rr / 32) * 4 + c % 4. With
 * G = 128 this is exactly mxfp8_swizzle_scales' layout of the [rows, cols]
 * matrix. Padding bytes of the A arrays (rows T..t_pad-1 of qa_scales,
 * token blocks ceil(T/32)..t_pad/32-1 of qb_scales) are written as 0; the
 * B arrays' columns past ceil(T/32) too; rows that pad a B group to whole
 * chunks are unspecified.
 */
typedef struct {
    int64_t t_pad;       /* T rounded up to a multiple of 128: row pitch of qb and xt */
    int64_t b_group;     /* G of the B operands: the GEMMs' tile width over K */
    size_t qa;           /* E4M3 [T, N], blocks of 32 channels (dgrad operand A) */
    size_t qa_scales;    /* E8M0, tiled: rows t_pad (tokens), cols N/32, G = 128 */
    size_t qb;           /* E4M3 [N, t_pad], blocks of 32 tokens (wgrad operand A); 0 past T */
    size_t qb_scales;    /* E8M0, tiled: rows N, cols t_pad/32, G = 128 */
    size_t wt;           /* E4M3 [K, N]: Q_cols(W) (dgrad operand B) */
    size_t wt_scales;    /* E8M0, tiled: rows K, cols N/32, G = b_group */
    size_t xt;           /* E4M3 [K, t_pad]: Q_cols(x) (wgrad operand B) */
    size_t xt_scales;    /* E8M0, tiled: rows K, cols t_pad/32, G = b_group */
    size_t db_partials;  /* float32 [ceil(T/32), N] */
    size_t total;        /* == mla_q_uproj_workspace_size(shape, 3) */
} mla_mxfp8_bwd_layout;

MLAQ_API int mla_q_uproj_bwd_mxfp8_layout(const mla_q_shape *shape, mla_mxfp8_bwd_layout *out);
MLAQ_API int mla_q_uproj_bwd_mxfp8(const mla_q_shape *shape, const void *dq, const void *W,
                                   const void *x, const float *cos_tab, const float *sin_tab,
                                   const int32_t *pos, void *dx, void *dW, void *db, void *workspace,
                                   size_t ws_bytes, int *dev_status, void *stream);

/*
 * mla_q_uproj_bwd_mxfp8 with W's columnwise MXFP8 copy prepared by the
 * caller instead of W. W stays fixed across the micro-batches of a step, so
 * it is quantized once instead of on every call. The results are bit for
 * bit those of mla_q_uproj_bwd_mxfp8 given W.
 *   wt [K, N] E4M3 codes (row pitch N): the columnwise quantization of W
 *   [N, K], i.e. mxfp8_quantize_cols_tiled(N, K, MLA_IN_BF16, W, K, wt,
 *   wt_scales, group, ...) with group = the b_group that
 *   mla_q_uproj_bwd_mxfp8_layout reports for this shape. wt_scales then
 *   holds mxfp8_grouped_scale_bytes(K, N/32, group) bytes. Both 16-byte
 *   aligned, both required when dx is requested (else unused).
 * Everything else as mla_q_uproj_bwd_mxfp8; the workspace's wt regions stay
 * unused.
 */
MLAQ_API int mla_q_uproj_bwd_mxfp8_prepared(const mla_q_shape *shape, const void *dq, const uint8_t *wt,
                                            const uint8_t *wt_scales, const void *x, const float *cos_tab,
                                            const float *sin_tab, const int32_t *pos, void *dx, void *dW,
                                            void *db, void *workspace, size_t ws_bytes, int *dev_status,
                                            void *stream);

/* KV side of the attention block: see mla_kv_uproj_fwd. */
typedef struct {
    int64_t T;        /* tokens */
    int64_t K;        /* kv_lora_rank (columns of c_kv and of W) */
    int32_t H;        /* heads */
    int32_t Dn;       /* key channels from the up-projection, per head */
    int32_t Dv;       /* value channels, per head */
    int32_t Dr;       /* rope channels of the key (the shared k_pe) */
    int64_t cs_rows;  /* cos/sin table rows */
    int64_t cs_width; /* cos/sin table row pitch (elements), >= Dr */
} mla_kv_shape;

/*
 * KV up-projection with the key's rope part, into fresh buffers: kv = c_kv W^T
 * split per head into k_nope (Dn) and v (Dv); the shared k_pe [T, Dr] is
 * rotated by the same rotate-half rule as the query (column j of the table
 * for rope channel j, positions pos or t) and written after every head's
 * k_nope. Megatron-LM PR "Fix fused MLA YaRN RoPE query kernel corrupting
 * upstream tensor in-place", Solution section: the KV path (rotary kernel
 * for the key) writes fresh o_key and o_value buffers; the split and the
 * broadcast follow the MLA attention block (the pages give no formula).
 *   c_kv [T, K] bf16, W [H*(Dn+Dv), K] bf16 (head h's rows: Dn key rows, then
 *   Dv value rows), k_pe [T, Dr] bf16, cos/sin/pos as in the forward.
 *   o_key [T, H, Dn + Dr] bf16, o_value [T, H, Dv] bf16 (fp32 accumulation,
 *   the rotation in fp32, each rounded to bf16 once).
 * Requires Dn % 32 == 0, Dv % 32 == 0, 32 <= Dn + Dv <= 256, Dr in
 * {16, 32, 64}, K % 8 == 0 and 16-byte aligned c_kv, W, k_pe, o_key,
 * o_value; outputs may overlap nothing. Status words as in the forward.
 */
MLAQ_API int mla_kv_uproj_fwd(const mla_kv_shape *shape, const void *c_kv, const void *W,
                              const void *k_pe, const float *cos_tab, const float *sin_tab,
                              const int32_t *pos, void *o_key, void *o_value, int *dev_status,
                              void *stream);

/* Size of the device scratch array mla_q_uproj_bwd_dgrad_noalloc uses. */
#define MLA_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * dgrad without any workspace argument, for callers that cannot allocate
 * device memory. (The pages have no counterpart: this is an addition of this
 * library.) Some callers of a library like this one cannot allocate: a host
 * framework that lends a plugin only the tensors of one call and owns all
 * other device memory, or a latency-critical path that cannot pay for
 * cudaMalloc's implicit synchronization. This entry point computes exactly
 * what mla_q_uproj_bwd_dgrad computes, with the same arguments minus the
 * workspace, and takes its workspace (the partial sums of split tiles and,
 * without dq_pre_rope, the rotated rope channels) from a scratch array of
 * MLA_NOALLOC_SCRATCH_BYTES that the library keeps in device global memory
 * (every GPU that loads the library holds it until the process exits).
 *   - Arguments are checked first, exactly as mla_q_uproj_bwd_dgrad checks
 *     them, and return the same codes.
 *   - The first call in a CUDA context (per device; a context created after
 *     a device reset counts as new) looks up the scratch address there (a
 *     CUDA runtime query, no allocation); make that first call before any
 *     stream capture. It allocates nothing, ever.
 *   - A shape whose least workspace (mla_q_uproj_workspace_size(shape, 4),
 *     or less with dq_pre_rope) exceeds MLA_NOALLOC_SCRATCH_BYTES is rejected
 *     with MLA_ERR_WORKSPACE. Otherwise the whole scratch is handed to dgrad,
 *     which takes the fastest path whose workspace fits in it (with the same
 *     path, the result is bit-identical to mla_q_uproj_bwd_dgrad's).
 *   - All calls share the one array. Nothing in it has to start at zero
 *     (every partial dgrad reads is written earlier in the same call, and
 *     its flags carry a value new to each launch), but calls that overlap on
 *     the GPU (other streams, other threads) race on it: serialize them.
 */
MLAQ_API int mla_q_uproj_bwd_dgrad_noalloc(const mla_q_shape *shape, const void *dq, const void *W,
                                           const float *cos_tab, const float *sin_tab,
                                           const int32_t *pos, void *dx, void *dq_pre_rope,
                                           int *dev_status, void *stream);

/*
 * Standalone rowwise MXFP8 quantization of in[R, C] (row pitch ld_in
 * elements, ld_in >= C): codes [R, C] uint8 (dense, pitch C) and scales
 * [R, ceil(C/32)] uint8 (dense). Same rule as the forward's MXFP8 output,
 * blocks of 32 consecutive elements of a row (the last may be partial).
 * TransformerEngine PR "Add support for fused Q Up-Proj GEMM/RoPE/Quant",
 * Greptile summary ("two-phase MXFP8 quantization" helpers) and review
 * thread (mxfp8_quantize_only). Bit-exact: codes and scales depend only on
 * the input values. in_dtype is MLA_IN_F32 or MLA_IN_BF16. R = 0 or C = 0 is
 * a no-op. Pointers must be 4-byte aligned (16-byte for the fast path).
 */
MLAQ_API int mxfp8_quantize_rows(int64_t R, int64_t C, int in_dtype, const void *in,
                                 int64_t ld_in, uint8_t *codes, uint8_t *scales, void *stream);

/*
 * mxfp8_quantize_rows with the scales written in the tiled order block-scaled
 * GEMMs read: the layout mxfp8_swizzle_scales_grouped(R, ceil(C/32), group)
 * gives the row-major scales, padding bytes 0 (scales: that many bytes,
 * mxfp8_grouped_scale_bytes). Codes as mxfp8_quantize_rows. For
 * MLA_WEIGHT_MXFP8_TILED: x with group 128, W with
 * mla_q_uproj_w_scale_group(shape). Same errors as mxfp8_quantize_rows, and
 * MLA_ERR_INVALID_ARG for group <= 0.
 */
MLAQ_API int mxfp8_quantize_rows_tiled(int64_t R, int64_t C, int in_dtype, const void *in, int64_t ld_in,
                                       uint8_t *codes, uint8_t *scales, int64_t group, void *stream);

/*
 * Columnwise MXFP8 copy of in[R, C] (row pitch ld_in elements): the rowwise
 * quantization of its transpose, for GEMM operands that are reduced over
 * their rows. codes_t [C, R] uint8 (dense, pitch R) and scales_t
 * [C, ceil(R/32)] uint8 (dense): blocks of 32 consecutive rows of one column
 * (the last may be partial), same scale and element rule as
 * mxfp8_quantize_rows. TransformerEngine PR "Add support for fused Q Up-Proj
 * GEMM/RoPE/Quant", Greptile summary (the transpose among the MXFP8
 * quantization helpers). Bit-exact; R = 0 or C = 0 is a no-op. Outputs may
 * not overlap the input; pointers must be element-aligned.
 */
MLAQ_API int mxfp8_quantize_cols(int64_t R, int64_t C, int in_dtype, const void *in,
                                 int64_t ld_in, uint8_t *codes_t, uint8_t *scales_t, void *stream);

/*
 * mxfp8_quantize_cols with the scales of the transposed copy written in the
 * block-scaled GEMM's tiled order: scales_t = mxfp8_swizzle_scales_grouped
 * of the [C, ceil(R/32)] scales with row groups of `group`, padding 0
 * (mxfp8_grouped_scale_bytes(C, ceil(R/32), group) bytes). codes_t [C, R]
 * as mxfp8_quantize_cols. Needs a 16-byte aligned input with a 16-byte row
 * pitch and C a multiple of the vector width (else MLA_ERR_UNSUPPORTED); for
 * the prepared weight of mla_q_uproj_bwd_mxfp8_prepared.
 */
MLAQ_API int mxfp8_quantize_cols_tiled(int64_t R, int64_t C, int in_dtype, const void *in, int64_t ld_in,
                                       uint8_t *codes_t, uint8_t *scales_t, int64_t group, void *stream);

/*
 * E8M0 scales in the tiled order block-scaled GEMMs read (TransformerEngine PR
 * "Add support for fused Q Up-Proj GEMM/RoPE/Quant": the GEMM scale swizzle
 * among its MXFP8 helpers). in [rows, cols] row-major (pitch ld_in bytes),
 * e.g. the scales of mxfp8_quantize_rows or of the forward's q (rows = T*H,
 * cols = ceil(D/32)); out: mxfp8_swizzled_scale_bytes(rows, cols) bytes,
 * 16-byte aligned: tiles of 128 rows x 4 columns (512 bytes), tile (i, j) at
 * (i * ceil(cols/4) + j) * 512; row r, column c of a tile at byte
 * (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4); bytes past rows or cols
 * are 0. A pure byte permutation; rows = 0 or cols = 0 is a no-op.
 */
MLAQ_API size_t mxfp8_swizzled_scale_bytes(int64_t rows, int64_t cols);
MLAQ_API int mxfp8_swizzle_scales(int64_t rows, int64_t cols, const uint8_t *in, int64_t ld_in,
                                  uint8_t *out, void *stream);

/*
 * Device self-test of the bounded pipeline waits behind MLA_ERR_TIMEOUT.
 * The pages define no such operation. It checks the library's own contract:
 * no device wait spins forever, and a wait that gives up is reported in the
 * status word with the context still usable. One CTA of two roles, with the
 * kernels' wait routine: role 0 waits on an mbarrier that only arrive != 0
 * completes, role 1 on one that only role 0's success completes. With
 * arrive == 0, role 0 gives up after limit_ns of %globaltimer and sets the
 * CTA's abort flag, role 1 leaves through that flag, and MLA_ERR_TIMEOUT is
 * written to *dev_status (if it held 0); with arrive != 0 nothing is
 * written. No copy or MMA is in flight at any point. limit_ns in
 * [1e6, 1e9] (else MLA_ERR_INVALID_ARG); dev_status: device int, 4-byte
 * aligned, required. Asynchronous on the stream; the kernel ends within
 * 2 * limit_ns of starting.
 */
MLAQ_API int mla_wait_selftest(int arrive, uint64_t limit_ns, int *dev_status, void *stream);

/*
 * The same check for the other kind of device wait, the one on a flag in
 * global memory that another CTA raises (dgrad's stream-K owners wait so
 * for the partial sums of the later CTAs of their column; the pages define
 * no such operation). One CTA: role 0 waits on a flag that role 1 raises
 * only when set != 0, then releases role 1. With set == 0 role 0 gives up
 * after limit_ns of %globaltimer, role 1 leaves through the CTA's abort flag,
 * and MLA_ERR_TIMEOUT is written to *dev_status (if it held 0). The flag is
 * a word of the library's own device memory: calls must not overlap.
 * limit_ns in [1e6, 1e9], dev_status as for mla_wait_selftest.
 */
MLAQ_API int mla_wait_selftest_flag(int set, uint64_t limit_ns, int *dev_status, void *stream);

/*
 * Row-group variant of mxfp8_swizzle_scales: rows in groups of `group`, each
 * group padded to whole 128-row tiles (so a GEMM tile of `group` rows starts
 * at a tile boundary). Chunk i of group g and column tile j is the 512-byte
 * tile ((g * ceil(group/128) + i) * ceil(cols/4) + j); inside it the byte
 * order of mxfp8_swizzle_scales; padding bytes 0. group = 128 is
 * mxfp8_swizzle_scales. out: mxfp8_grouped_scale_bytes(rows, cols, group)
 * bytes, 16-byte aligned. A pure byte permutation (TransformerEngine PR "Add
 * support for fused Q Up-Proj GEMM/RoPE/Quant": the GEMM scale swizzle among
 * its MXFP8 helpers), used to tile W's scales for MLA_WEIGHT_MXFP8_TILED.
 */
MLAQ_API size_t mxfp8_grouped_scale_bytes(int64_t rows, int64_t cols, int64_t group);
MLAQ_API int mxfp8_swizzle_scales_grouped(int64_t rows, int64_t cols, int64_t group, const uint8_t *in,
                                          int64_t ld_in, uint8_t *out, void *stream);

/* The row group of W's tiled scales for MLA_WEIGHT_MXFP8_TILED at this shape
 * (the forward's channel tile with MXFP8 weights), or 0 when the shape is
 * invalid or not tiled. */
MLAQ_API int64_t mla_q_uproj_w_scale_group(const mla_q_shape *shape);

/* which: 0 = forward, 1 = dgrad, 2 = wgrad, 3 = MXFP8 backward, 4 = the
 * least workspace dgrad accepts. Bytes of device workspace the call needs
 * for this shape (0 = pass NULL). Of the bf16 calls only dgrad ever needs
 * any (see mla_q_uproj_bwd_dgrad; its sizes depend on the current device):
 * with 1's size it takes its fastest path, with at least 4's a slower one
 * that needs less. Returns 0 for an invalid shape or, for which = 1 and 4,
 * when no CUDA device is usable. */
MLAQ_API size_t mla_q_uproj_workspace_size(const mla_q_shape *shape, int which);

/* Static, human-readable name of a status code. */
MLAQ_API const char *mla_status_string(int status);

/* ABI version of this header (major * 10000 + minor * 100 + patch). */
MLAQ_API int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLAQ_H */
