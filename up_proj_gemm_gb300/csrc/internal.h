// Declarations shared by the translation units of libmlaq.so (host side).
#pragma once
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "mlaq.h"

namespace mlaq {

// Device properties of the current device, cached per device.
struct DeviceInfo {
    int device = -1;
    int num_sms = 0;
    int max_smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
};
int current_device_info(DeviceInfo* out);  // returns an mla status

// cuTensorMapEncodeTiled, resolved through the runtime's driver entry point.
// 2-D, row-major tensor: dims {inner, outer}, row pitch in bytes, box
// {box_inner, box_outer}, 128-byte swizzle when swizzle128 (64-byte
// swizzle when swizzle64), else none. dtype: 0 = uint8, 1 = bf16.
int make_tmap_2d(void* tmap_out /* CUtensorMap, 64 B aligned */, const void* base, int dtype,
                 uint64_t inner, uint64_t outer, uint64_t row_pitch_bytes, uint32_t box_inner,
                 uint32_t box_outer, bool swizzle128, bool swizzle64 = false);

// 3-D view of a row-major bf16 matrix [rows, cols] as 64-column chunks:
// dims {64, rows, cols / 64} with strides {row pitch, 128 bytes}; a box
// {64, box_rows, box_chunks} lands in shared memory as box_chunks
// consecutive [box_rows][64] blocks (128-byte swizzle), the MN-major
// operand layout of the tensor cores. cols must be a multiple of 64.
int make_tmap_chunks(void* tmap_out, const void* base, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_chunks);

// General 3-D bf16 map, 128-byte swizzle: dims {d0 (contiguous), d1, d2},
// byte strides of d1 and d2, box {b0, b1, b2} (b0 * 2 bytes == 128).
int make_tmap_3d(void* tmap_out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                 uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2);

// ------------------------------------------------------------- launchers
// All launchers assume arguments were validated by the API layer.
int launch_mxfp8_swizzle(int64_t rows, int64_t cols, int64_t group, const uint8_t* in, int64_t ld, uint8_t* out,
                         cudaStream_t stream);
int launch_mxfp8_quantize_cols(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                               uint8_t* codes_t, uint8_t* scales_t, cudaStream_t stream);
// The same with output row pitches: codes_t [C, ld_codes >= R], scales_t
// [C, ld_scales >= ceil(R/32)] (bytes past R / ceil(R/32) are not written,
// except scale bytes inside the 4-byte word of a row's last 128-row tile,
// which are written as 0).
int launch_mxfp8_quantize_cols_ld(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                  uint8_t* codes_t, int64_t ld_codes, uint8_t* scales_t, int64_t ld_scales,
                                  cudaStream_t stream);
// The same with the scales in the GEMM's tiled order (sf_tiled_offset with
// rows = C, cols = ceil(R/32), groups of sf_group rows; every byte of the
// ceil(R/128) K steps written, 0 past R). Needs the 16-byte fast path (in
// 16-byte aligned, ld_in and C multiples of the 16-byte vector), else
// MLA_ERR_UNSUPPORTED.
int launch_mxfp8_quantize_cols_tiled_sf(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                        uint8_t* codes_t, int64_t ld_codes, uint8_t* scales_t, int64_t sf_group,
                                        cudaStream_t stream);
// sf_group > 0: scales in the GEMM's tiled order with row groups of sf_group
// (padding zero-filled); 0: row-major [R, ceil(C/32)].
int launch_mxfp8_quantize(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                          uint8_t* codes, uint8_t* scales, cudaStream_t stream, int64_t sf_group = 0);

struct FwdArgs {
    int64_t T, K;
    int H, Dn, Dr;
    int64_t cs_rows, cs_width;
    int weight_mode, out_mode;
    const void* x;
    const uint8_t* x_scales;
    const void* W;
    const uint8_t* w_scales;
    const void* bias;
    const float* cos_tab;
    const float* sin_tab;
    const void* rope_packed = nullptr;  // mla_rope_table_pack's layout, used instead of cos/sin when set
    const int32_t* pos;
    void* q_out;
    uint8_t* q_scales;
    int* status;
    // Row pitches of the MXFP8 operands (codes: bytes, scales: bytes; 0 = dense
    // K and K / 32). With Dr == 0 (H = 1, Dn = the output width) the kernel is
    // a plain block-scaled GEMM q = x W^T with a bf16 output and no rotation,
    // its tiles walked with the output-channel tile fastest;
    // the operand rows may then be longer than K (reads past K are zero codes
    // from the tensor map; their scale bytes must be finite).
    int64_t ld_x = 0, ld_w = 0, ld_scale = 0;
    // MXFP8 scales already in the GEMM's tiled order (sf_tiled_offset): x's
    // with G = 128 over ceil(T/128) chunks, W's with G = sf_group, which must
    // equal the tile width the kernel picks for this shape (else
    // MLA_ERR_UNSUPPORTED); ld_scale is then unused.
    int sf_tiled = 0, sf_group = 0;
};
int launch_fwd(const FwdArgs& a, cudaStream_t stream);
// The packed rotary table (see mla_rope_table_pack).
int launch_rope_table_pack(int64_t rows, int64_t width, int Dr, const float* cos_tab, const float* sin_tab,
                           void* packed, cudaStream_t stream);

struct KvArgs {
    int64_t T, K;
    int H, Dn, Dv, Dr;
    int64_t cs_rows, cs_width;
    const void* c_kv;
    const void* W;
    const void* k_pe;
    const float* cos_tab;
    const float* sin_tab;
    const int32_t* pos;
    void* o_key;
    void* o_value;
    int* status;
};
int launch_kv_fwd(const KvArgs& a, cudaStream_t stream);

struct BwdArgs {
    int64_t T, K;
    int H, Dn, Dr;
    int64_t cs_rows, cs_width;
    const void* dq;
    const void* W;   // dgrad
    const void* x;   // wgrad
    const float* cos_tab;
    const float* sin_tab;
    const int32_t* pos;
    void* dx;        // dgrad
    void* dW;        // wgrad
    void* db;        // wgrad, nullable
    void* rope_out;       // dgrad, nullable: rotated rope channels [T, H, Dr] bf16
    const void* rope_in;  // wgrad, nullable: the same buffer, read instead of rotating dq
    void* workspace; // dgrad split partials (see dgrad_workspace_bytes)
    size_t ws_bytes;
    int* status;
    // MXFP8 backward only: W's columnwise MXFP8 copy prepared by the caller
    // (wt [K, N] codes, scales in the GEMM's tiled order); W is then unused
    const uint8_t* wt = nullptr;
    const uint8_t* wt_s = nullptr;
};
int launch_dgrad(const BwdArgs& a, cudaStream_t stream);
// dgrad's split of the channel reduction for this shape on a device with
// num_sms SMs, and the fp32 workspace it needs (0 when not split).
int dgrad_ksplit(int64_t T, int64_t K, int64_t N, int num_sms);
// Best split count (1..4, each part >= 32 K steps) for this many tiles.
int best_ksplit(int64_t tiles, int64_t k_tiles, int num_sms);
// Workspace of the fused dgrad (split partials only).
size_t dgrad_workspace_bytes_fused(int64_t T, int64_t K, int64_t N, int num_sms);
// Workspace that lets dgrad take its fastest path for this shape (for the
// pre-rotated path: its split partials plus the rotated rope channels).
size_t dgrad_workspace_bytes(int64_t T, int64_t K, int H, int Dn, int Dr, int num_sms);
// The pre-rotated path's workspace for this shape ((size_t)-1: no such path).
size_t dgrad_pre_shape_bytes(int64_t T, int64_t K, int H, int Dn, int Dr, int num_sms, bool have_rope_out);
// The least workspace dgrad accepts for this shape (the smaller of the two
// paths' needs; the path is then chosen by the workspace given).
size_t dgrad_min_workspace_bytes(int64_t T, int64_t K, int H, int Dn, int Dr, int num_sms, bool have_rope_out);
int launch_wgrad(const BwdArgs& a, cudaStream_t stream);
// The checks of mla_q_uproj_bwd_dgrad that do not involve the workspace.
int dgrad_check_args(const mla_q_shape* shape, const void* dq, const void* W, const float* cos_tab,
                     const float* sin_tab, const int32_t* pos, const void* dx, const void* dq_pre_rope,
                     const int* dev_status);

// MXFP8 backward (see mla_q_uproj_bwd_mxfp8): workspace carve-up and launch.
struct Mxfp8BwdLayout {
    int64_t Tp;  // tokens rounded up to 128 (row pitch of the token-blocked operands)
    int64_t G;   // GEMM tile width over K (the rows of each B operand's scale group)
    size_t qa, qa_s, qb, qb_s, wt, wt_s, xt, xt_s, dbp, total;
};
int bwd_mxfp8_layout(int64_t T, int64_t K, int64_t N, Mxfp8BwdLayout* out);
int launch_bwd_mxfp8(const BwdArgs& a, cudaStream_t stream);

// Tile width (channels) of the forward kernel for this shape: the largest
// multiple of `step` that is <= max_bn, divides N and keeps every rope region
// and every 32-channel pass-through block inside one tile; 0 if none.
int fwd_tile_n(int64_t N, int D, int Dn, int Dr, int max_bn, int step);

}  // namespace mlaq
