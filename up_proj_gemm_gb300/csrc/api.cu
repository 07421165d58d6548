// C ABI of libmlaq.so: argument validation, then the kernel launchers.
//
// Every check below runs on the host before any CUDA call, so a rejected
// call touches neither the device nor the stream. The order of checks fixes
// which status a call with several faults returns: missing/invalid
// arguments, table width, positions, tiling support, alignment, aliasing.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "mx.cuh"

namespace mlaq {

// ------------------------------------------------------------- device info
int current_device_info(DeviceInfo* out) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = cache[dev];
    if (d.device != dev) {
        DeviceInfo n;
        n.device = dev;
        if (cudaDeviceGetAttribute(&n.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&n.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return MLA_ERR_CUDA;
        d = n;
    }
    *out = d;
    // The kernels are built for sm_103a only.
    if (d.cc_major != 10 || d.cc_minor != 3) return MLA_ERR_CUDA;
    return MLA_OK;
}

// ------------------------------------------------------------- tensor maps
int make_tmap_2d(void* tmap_out, const void* base, int dtype, uint64_t inner, uint64_t outer,
                 uint64_t row_pitch_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128,
                 bool swizzle64) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode) return MLA_ERR_CUDA;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap_out),
                        dtype == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : (swizzle64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

int make_tmap_3d(void* tmap_out, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t stride1,
                 uint64_t stride2, uint32_t b0, uint32_t b1, uint32_t b2) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode) return MLA_ERR_CUDA;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1, stride2};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

int make_tmap_chunks(void* tmap_out, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                     uint32_t box_chunks) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    if (!encode || cols % 64) return MLA_ERR_CUDA;
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, box_chunks};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(reinterpret_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_CUDA;
}

namespace {

struct Range {
    uintptr_t lo = 0, hi = 0;  // [lo, hi); empty when lo == hi
};

Range rng(const void* p, int64_t bytes) {
    Range r;
    if (p && bytes > 0) {
        r.lo = reinterpret_cast<uintptr_t>(p);
        r.hi = r.lo + (uintptr_t)bytes;
    }
    return r;
}

bool overlap(const Range& a, const Range& b) {
    return a.lo != a.hi && b.lo != b.hi && a.lo < b.hi && b.lo < a.hi;
}

template <size_t NO, size_t NI>
bool any_alias(const Range (&outs)[NO], const Range (&ins)[NI]) {
    for (size_t i = 0; i < NO; ++i) {
        for (size_t j = 0; j < NI; ++j)
            if (overlap(outs[i], ins[j])) return true;
        for (size_t j = i + 1; j < NO; ++j)
            if (overlap(outs[i], outs[j])) return true;
    }
    return false;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int64_t kI32Max = 0x7fffffffLL;

// Checks shared by every mla_q_uproj_* call. On success fills D and N.
int check_shape(const mla_q_shape* s, int* D, int64_t* N) {
    if (!s) return MLA_ERR_INVALID_ARG;
    if (s->T < 0 || s->K <= 0 || s->H <= 0 || s->Dn < 0 || s->Dr <= 0 || (s->Dr & 1) ||
        s->cs_rows < 0 || s->cs_width < 0 || s->reserved != 0)
        return MLA_ERR_INVALID_ARG;
    const int64_t d = (int64_t)s->Dn + s->Dr;
    const int64_t n = d * s->H;
    if (d > kI32Max || n > kI32Max || s->T > kI32Max || s->K > kI32Max) return MLA_ERR_INVALID_ARG;
    // positions are int32, so no row past INT32_MAX is reachable; both bounds
    // keep the table's byte extent (rows * width * 4) inside int64
    if (s->cs_rows > kI32Max || s->cs_width > kI32Max) return MLA_ERR_INVALID_ARG;
    *D = (int)d;
    *N = n;
    return MLA_OK;
}

int check_table_and_positions(const mla_q_shape* s, const float* cos_tab, const float* sin_tab,
                              const int32_t* pos) {
    if (s->cs_width < s->Dr) return MLA_ERR_ROPE_WIDTH;
    if (s->T > 0 && (!cos_tab || !sin_tab)) return MLA_ERR_INVALID_ARG;
    if (!pos && s->T > s->cs_rows) return MLA_ERR_POS_RANGE;
    if (s->cs_rows == 0 && s->T > 0) return MLA_ERR_POS_RANGE;
    (void)pos;
    return MLA_OK;
}

bool rope_dim_supported(int Dr) { return Dr == 16 || Dr == 32 || Dr == 64; }

}  // namespace
}  // namespace mlaq

using namespace mlaq;

extern "C" {

MLAQ_API int mla_version(void) { return 10000; }

MLAQ_API const char* mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "MLA_OK";
        case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
        case MLA_ERR_ROPE_WIDTH: return "MLA_ERR_ROPE_WIDTH";
        case MLA_ERR_ALIGNMENT: return "MLA_ERR_ALIGNMENT";
        case MLA_ERR_ALIAS: return "MLA_ERR_ALIAS";
        case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
        case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
        case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
        case MLA_ERR_POS_RANGE: return "MLA_ERR_POS_RANGE";
        case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
        default: return "MLA_ERR_UNKNOWN";
    }
}

MLAQ_API size_t mla_q_uproj_workspace_size(const mla_q_shape* shape, int which) {
    int D;
    int64_t N;
    if (check_shape(shape, &D, &N) != MLA_OK || which < 0 || which > 4) return 0;
    if (which == 3) {  // MXFP8 backward: the quantized operands and the db partials
        Mxfp8BwdLayout L;
        if (shape->T == 0 || bwd_mxfp8_layout(shape->T, shape->K, N, &L) != MLA_OK) return 0;
        return L.total;
    }
    if ((which != 1 && which != 4) || shape->T == 0) return 0;  // only dgrad needs device scratch
    DeviceInfo di;
    if (current_device_info(&di) != MLA_OK) return 0;
    return which == 1 ? dgrad_workspace_bytes(shape->T, shape->K, shape->H, shape->Dn, shape->Dr, di.num_sms)
                      : dgrad_min_workspace_bytes(shape->T, shape->K, shape->H, shape->Dn, shape->Dr, di.num_sms,
                                                  false);
}

// The forward behind mla_q_uproj_fwd (cos_tab, sin_tab) and
// mla_q_uproj_fwd_packed (packed, the mla_rope_table_pack layout).
static int fwd_entry(const mla_q_shape* shape, int weight_mode, int out_mode, const void* x,
                     const uint8_t* x_scales, const void* W, const uint8_t* w_scales, const void* bias,
                     const float* cos_tab, const float* sin_tab, const float* packed, const int32_t* pos,
                     void* q_out, uint8_t* q_scales_out, int* dev_status, void* stream) {
    int D;
    int64_t N;
    int st = check_shape(shape, &D, &N);
    if (st != MLA_OK) return st;
    const mla_q_shape& s = *shape;
    if (weight_mode != MLA_WEIGHT_BF16 && weight_mode != MLA_WEIGHT_MXFP8 && weight_mode != MLA_WEIGHT_MXFP8_TILED)
        return MLA_ERR_INVALID_ARG;
    const bool tiled = weight_mode == MLA_WEIGHT_MXFP8_TILED;
    if (out_mode != MLA_OUT_BF16 && out_mode != MLA_OUT_MXFP8 && out_mode != MLA_OUT_MXFP8_BHSD &&
        out_mode != MLA_OUT_MXFP8_BHSD_SWIZZLED)
        return MLA_ERR_INVALID_ARG;
    const bool mxw = weight_mode != MLA_WEIGHT_BF16, mxo = out_mode != MLA_OUT_BF16;
    if (mxw != (x_scales != nullptr) || mxw != (w_scales != nullptr)) return MLA_ERR_INVALID_ARG;
    if (mxo != (q_scales_out != nullptr)) return MLA_ERR_INVALID_ARG;
    if (s.T > 0 && (!x || !W || !q_out)) return MLA_ERR_INVALID_ARG;
    if (mxw && (s.K % 32)) return MLA_ERR_INVALID_ARG;  // scales are per 32 along K
    st = packed ? check_table_and_positions(&s, packed, packed, pos)
                : check_table_and_positions(&s, cos_tab, sin_tab, pos);
    if (st != MLA_OK) return st;
    if (s.T == 0) return MLA_OK;

    if (!rope_dim_supported(s.Dr) || s.Dn % 32) return MLA_ERR_UNSUPPORTED;
    if (mxw && s.K % 128) return MLA_ERR_UNSUPPORTED;
    const int bn = fwd_tile_n(N, D, s.Dn, s.Dr, mxw ? 192 : 256, mxw ? 32 : 16);
    if (bn == 0) return MLA_ERR_UNSUPPORTED;
    // tiled scales arrive by 16-byte bulk copies
    if (tiled && (!aligned(x_scales, 16) || !aligned(w_scales, 16))) return MLA_ERR_ALIGNMENT;

    const int64_t esz = mxw ? 1 : 2;
    if ((s.K * esz) % 16) return MLA_ERR_ALIGNMENT;
    if (!aligned(x, 16) || !aligned(W, 16) || !aligned(q_out, 16) || !aligned(x_scales, 4) ||
        !aligned(w_scales, 4) || !aligned(bias, 16) || !aligned(cos_tab, 4) || !aligned(sin_tab, 4) ||
        !aligned(packed, 16) || !aligned(pos, 4) || !aligned(dev_status, 4))
        return MLA_ERR_ALIGNMENT;

    const int64_t NB = (D + 31) / 32;
    // the table's byte extent: rows x width fp32 each, or the packed rows x Dr fp32
    const int64_t table = packed ? s.cs_rows * s.Dr * 4 : s.cs_rows * s.cs_width * 4;
    if (packed) cos_tab = sin_tab = packed;  // (extents for the overlap check only)
    const int64_t qs_bytes = out_mode == MLA_OUT_MXFP8_BHSD_SWIZZLED
                                 ? (int64_t)s.H * (int64_t)mxfp8_swizzled_scale_bytes(s.T, NB)
                                 : s.T * s.H * NB;
    const Range outs[] = {rng(q_out, s.T * N * (mxo ? 1 : 2)), rng(q_scales_out, qs_bytes),
                          rng(dev_status, 4)};
    const int64_t xs_bytes = tiled ? (int64_t)sf_tiled_bytes(s.T, s.K / 32, 128) : s.T * (s.K / 32);
    const int64_t ws_bytes = tiled ? (int64_t)sf_tiled_bytes(N, s.K / 32, bn) : N * (s.K / 32);
    const Range ins[] = {rng(x, s.T * s.K * esz), rng(x_scales, xs_bytes),
                         rng(W, N * s.K * esz),   rng(w_scales, ws_bytes),
                         rng(bias, N * 2),        rng(cos_tab, table),
                         rng(sin_tab, table),     rng(pos, s.T * 4)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;

    FwdArgs a{};
    a.T = s.T;
    a.K = s.K;
    a.H = s.H;
    a.Dn = s.Dn;
    a.Dr = s.Dr;
    a.cs_rows = s.cs_rows;
    a.cs_width = s.cs_width;
    a.weight_mode = mxw ? MLA_WEIGHT_MXFP8 : MLA_WEIGHT_BF16;
    a.out_mode = out_mode;
    if (tiled) {
        a.sf_tiled = 1;
        a.sf_group = bn;
    }
    a.x = x;
    a.x_scales = x_scales;
    a.W = W;
    a.w_scales = w_scales;
    a.bias = bias;
    a.cos_tab = packed ? nullptr : cos_tab;
    a.sin_tab = packed ? nullptr : sin_tab;
    a.rope_packed = packed;
    a.pos = pos;
    a.q_out = q_out;
    a.q_scales = q_scales_out;
    a.status = dev_status;
    return launch_fwd(a, static_cast<cudaStream_t>(stream));
}

MLAQ_API int mla_q_uproj_fwd(const mla_q_shape* shape, int weight_mode, int out_mode, const void* x,
                             const uint8_t* x_scales, const void* W, const uint8_t* w_scales,
                             const void* bias, const float* cos_tab, const float* sin_tab,
                             const int32_t* pos, void* q_out, uint8_t* q_scales_out, int* dev_status,
                             void* stream) {
    return fwd_entry(shape, weight_mode, out_mode, x, x_scales, W, w_scales, bias, cos_tab, sin_tab, nullptr, pos,
                     q_out, q_scales_out, dev_status, stream);
}

MLAQ_API int mla_q_uproj_fwd_packed(const mla_q_shape* shape, int weight_mode, int out_mode, const void* x,
                                    const uint8_t* x_scales, const void* W, const uint8_t* w_scales,
                                    const void* bias, const float* rope_packed, const int32_t* pos, void* q_out,
                                    uint8_t* q_scales_out, int* dev_status, void* stream) {
    return fwd_entry(shape, weight_mode, out_mode, x, x_scales, W, w_scales, bias, nullptr, nullptr, rope_packed,
                     pos, q_out, q_scales_out, dev_status, stream);
}

MLAQ_API size_t mla_rope_table_packed_bytes(int64_t cs_rows, int Dr) {
    if (cs_rows < 0 || cs_rows > kI32Max || Dr <= 0 || (Dr & 1)) return 0;
    return (size_t)cs_rows * (size_t)(Dr / 2) * 16;
}

MLAQ_API int mla_rope_table_pack(int64_t cs_rows, int64_t cs_width, int Dr, const float* cos_tab,
                                 const float* sin_tab, float* packed, void* stream) {
    if (cs_rows < 0 || cs_width < 0 || cs_rows > kI32Max || cs_width > kI32Max || Dr <= 0 || (Dr & 1))
        return MLA_ERR_INVALID_ARG;
    if (cs_width < Dr) return MLA_ERR_ROPE_WIDTH;
    if (cs_rows == 0) return MLA_OK;
    if (!cos_tab || !sin_tab || !packed) return MLA_ERR_INVALID_ARG;
    if (!aligned(cos_tab, 4) || !aligned(sin_tab, 4) || !aligned(packed, 16)) return MLA_ERR_ALIGNMENT;
    const int64_t table = cs_rows * cs_width * 4;
    const Range outs[] = {rng(packed, (int64_t)mla_rope_table_packed_bytes(cs_rows, Dr))};
    const Range ins[] = {rng(cos_tab, table), rng(sin_tab, table)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    return launch_rope_table_pack(cs_rows, cs_width, Dr, cos_tab, sin_tab, packed, static_cast<cudaStream_t>(stream));
}

static int check_bwd(const mla_q_shape* shape, const void* dq, const void* op, const float* cos_tab,
                     const float* sin_tab, const int32_t* pos, const void* out, void* workspace,
                     size_t ws_bytes, int which, int* D, int64_t* N) {
    int st = check_shape(shape, D, N);
    if (st != MLA_OK) return st;
    const mla_q_shape& s = *shape;
    if (s.T > 0 && (!dq || !op || !out)) return MLA_ERR_INVALID_ARG;
    st = check_table_and_positions(&s, cos_tab, sin_tab, pos);
    if (st != MLA_OK) return st;
    if (which == 2 && ws_bytes < mla_q_uproj_workspace_size(shape, which)) return MLA_ERR_WORKSPACE;
    if (!rope_dim_supported(s.Dr) || s.Dn % s.Dr) return MLA_ERR_UNSUPPORTED;
    if ((s.K * 2) % 16 || ((*N) * 2) % 16) return MLA_ERR_ALIGNMENT;
    return MLA_OK;
}

extern "C++" {
namespace mlaq {
// dgrad's checks that do not involve the workspace (shape, table, positions,
// support, alignment), in the order both dgrad entry points run them.
int dgrad_check_args(const mla_q_shape* shape, const void* dq, const void* W, const float* cos_tab,
                     const float* sin_tab, const int32_t* pos, const void* dx, const void* dq_pre_rope,
                     const int* dev_status) {
    int D;
    int64_t N;
    int st = check_bwd(shape, dq, W, cos_tab, sin_tab, pos, dx, nullptr, 0, 1, &D, &N);
    if (st != MLA_OK) return st;
    if (!aligned(dq, 16) || !aligned(W, 16) || !aligned(dx, 16) || !aligned(cos_tab, 4) ||
        !aligned(sin_tab, 4) || !aligned(pos, 4) || !aligned(dev_status, 4) || !aligned(dq_pre_rope, 16))
        return MLA_ERR_ALIGNMENT;
    return MLA_OK;
}
}  // namespace mlaq
}  // extern "C++"

MLAQ_API int mla_q_uproj_bwd_dgrad(const mla_q_shape* shape, const void* dq, const void* W,
                                   const float* cos_tab, const float* sin_tab, const int32_t* pos,
                                   void* dx, void* dq_pre_rope, void* workspace, size_t ws_bytes,
                                   int* dev_status, void* stream) {
    int st = dgrad_check_args(shape, dq, W, cos_tab, sin_tab, pos, dx, dq_pre_rope, dev_status);
    if (st != MLA_OK) return st;
    if (!aligned(workspace, 16)) return MLA_ERR_ALIGNMENT;
    const mla_q_shape& s = *shape;
    const int64_t N = (int64_t)s.H * (s.Dn + s.Dr);
    const int64_t table = s.cs_rows * s.cs_width * 4;
    // the least workspace dgrad takes (the fused path's); with at least
    // mla_q_uproj_workspace_size(shape, 1) bytes it takes the pre-rotated path
    // (without a usable device the sizes are unknown here; the launch reports it)
    size_t least = 0, fast = (size_t)-1;
    DeviceInfo di;
    if (s.T > 0 && current_device_info(&di) == MLA_OK) {
        least = dgrad_min_workspace_bytes(s.T, s.K, s.H, s.Dn, s.Dr, di.num_sms, dq_pre_rope != nullptr);
        fast = dgrad_pre_shape_bytes(s.T, s.K, s.H, s.Dn, s.Dr, di.num_sms, dq_pre_rope != nullptr);
    }
    if (ws_bytes < least || (least > 0 && !workspace)) return MLA_ERR_WORKSPACE;
    const size_t need = (fast != (size_t)-1 && ws_bytes >= fast && (fast == 0 || workspace)) ? fast : least;
    const Range outs[] = {rng(dx, s.T * s.K * 2), rng(dev_status, 4), rng(workspace, (int64_t)need),
                          rng(dq_pre_rope, s.T * s.H * s.Dr * 2)};
    const Range ins[] = {rng(dq, s.T * N * 2), rng(W, N * s.K * 2), rng(cos_tab, table),
                         rng(sin_tab, table), rng(pos, s.T * 4)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    if (s.T == 0) return MLA_OK;
    BwdArgs a{};
    a.T = s.T;
    a.K = s.K;
    a.H = s.H;
    a.Dn = s.Dn;
    a.Dr = s.Dr;
    a.cs_rows = s.cs_rows;
    a.cs_width = s.cs_width;
    a.dq = dq;
    a.W = W;
    a.cos_tab = cos_tab;
    a.sin_tab = sin_tab;
    a.pos = pos;
    a.dx = dx;
    a.rope_out = dq_pre_rope;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    a.status = dev_status;
    return launch_dgrad(a, static_cast<cudaStream_t>(stream));
}

MLAQ_API int mla_q_uproj_bwd_wgrad(const mla_q_shape* shape, const void* dq, const void* dq_pre_rope,
                                   const void* x, const float* cos_tab, const float* sin_tab,
                                   const int32_t* pos, void* dW, void* db, void* workspace,
                                   size_t ws_bytes, int* dev_status, void* stream) {
    int D;
    int64_t N;
    int st = check_bwd(shape, dq, x, cos_tab, sin_tab, pos, dW, workspace, ws_bytes, 2, &D, &N);
    if (st != MLA_OK) return st;
    const mla_q_shape& s = *shape;
    if (!aligned(dq, 16) || !aligned(x, 16) || !aligned(dW, 16) || !aligned(db, 4) ||
        !aligned(cos_tab, 4) || !aligned(sin_tab, 4) || !aligned(pos, 4) || !aligned(dev_status, 4) ||
        !aligned(dq_pre_rope, 16))
        return MLA_ERR_ALIGNMENT;
    const int64_t table = s.cs_rows * s.cs_width * 4;
    const Range outs[] = {rng(dW, N * s.K * 2), rng(db, N * 2), rng(dev_status, 4)};
    const Range ins[] = {rng(dq, s.T * N * 2), rng(x, s.T * s.K * 2), rng(cos_tab, table),
                         rng(sin_tab, table), rng(pos, s.T * 4), rng(dq_pre_rope, s.T * s.H * s.Dr * 2)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    BwdArgs a{};
    a.T = s.T;
    a.K = s.K;
    a.H = s.H;
    a.Dn = s.Dn;
    a.Dr = s.Dr;
    a.cs_rows = s.cs_rows;
    a.cs_width = s.cs_width;
    a.dq = dq;
    a.rope_in = dq_pre_rope;
    a.x = x;
    a.cos_tab = cos_tab;
    a.sin_tab = sin_tab;
    a.pos = pos;
    a.dW = dW;
    a.db = db;
    a.status = dev_status;
    // T == 0 still defines dW = 0 and db = 0: the kernel writes zeros.
    return launch_wgrad(a, static_cast<cudaStream_t>(stream));
}

MLAQ_API int mla_q_uproj_bwd_mxfp8_layout(const mla_q_shape* shape, mla_mxfp8_bwd_layout* out) {
    int D;
    int64_t N;
    int st = check_shape(shape, &D, &N);
    if (st != MLA_OK) return st;
    if (!out) return MLA_ERR_INVALID_ARG;
    Mxfp8BwdLayout L;
    st = bwd_mxfp8_layout(shape->T, shape->K, N, &L);
    if (st != MLA_OK) return st;
    out->t_pad = L.Tp;
    out->b_group = L.G;
    out->qa = L.qa;
    out->qa_scales = L.qa_s;
    out->qb = L.qb;
    out->qb_scales = L.qb_s;
    out->wt = L.wt;
    out->wt_scales = L.wt_s;
    out->xt = L.xt;
    out->xt_scales = L.xt_s;
    out->db_partials = L.dbp;
    out->total = shape->T == 0 ? 0 : L.total;
    return MLA_OK;
}

}  // extern "C"

// The MXFP8 backward, with W or (wt, wt_s), its columnwise MXFP8 copy.
static int bwd_mxfp8_call(const mla_q_shape* shape, const void* dq, const void* W, const uint8_t* wt,
                          const uint8_t* wt_s, const void* x, const float* cos_tab, const float* sin_tab,
                          const int32_t* pos, void* dx, void* dW, void* db, void* workspace, size_t ws_bytes,
                          int* dev_status, void* stream) {
    int D;
    int64_t N;
    int st = check_shape(shape, &D, &N);
    if (st != MLA_OK) return st;
    const mla_q_shape& s = *shape;
    if (!dx && !dW && !db) return MLA_ERR_INVALID_ARG;
    const bool prepared = wt != nullptr || wt_s != nullptr;
    if (prepared && (!wt || !wt_s || W)) return MLA_ERR_INVALID_ARG;
    if (s.T > 0 && (!dq || (dx && !W && !prepared) || (dW && !x))) return MLA_ERR_INVALID_ARG;
    st = check_table_and_positions(&s, cos_tab, sin_tab, pos);
    if (st != MLA_OK) return st;
    const size_t need = mla_q_uproj_workspace_size(shape, 3);
    if (s.T > 0 && (ws_bytes < need || !workspace)) return MLA_ERR_WORKSPACE;
    if (!rope_dim_supported(s.Dr) || s.Dn % 32 || D % 32 || N % 128 || s.K % 32) return MLA_ERR_UNSUPPORTED;
    if (fwd_tile_n(s.K, (int)s.K, (int)s.K, 0, 192, 32) == 0) return MLA_ERR_UNSUPPORTED;
    if (!aligned(dq, 16) || !aligned(W, 16) || !aligned(x, 16) || !aligned(dx, 16) || !aligned(dW, 16) ||
        !aligned(db, 4) || !aligned(cos_tab, 4) || !aligned(sin_tab, 4) || !aligned(pos, 4) ||
        !aligned(dev_status, 4) || !aligned(workspace, 16) || !aligned(wt, 16) || !aligned(wt_s, 16))
        return MLA_ERR_ALIGNMENT;
    const int64_t table = s.cs_rows * s.cs_width * 4;
    const int64_t G = fwd_tile_n(s.K, (int)s.K, (int)s.K, 0, 192, 32);
    const int64_t wts = prepared && dx ? (int64_t)sf_tiled_bytes(s.K, N / 32, G) : 0;
    const Range outs[] = {rng(dx, s.T * s.K * 2), rng(dW, N * s.K * 2), rng(db, N * 2), rng(dev_status, 4),
                          rng(workspace, (int64_t)need)};
    const Range ins[] = {rng(dq, s.T * N * 2), rng(W, dx ? N * s.K * 2 : 0), rng(x, dW ? s.T * s.K * 2 : 0),
                         rng(cos_tab, table), rng(sin_tab, table), rng(pos, s.T * 4),
                         rng(wt, prepared && dx ? s.K * N : 0), rng(wt_s, wts)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    BwdArgs a{};
    a.T = s.T;
    a.K = s.K;
    a.H = s.H;
    a.Dn = s.Dn;
    a.Dr = s.Dr;
    a.cs_rows = s.cs_rows;
    a.cs_width = s.cs_width;
    a.dq = dq;
    a.W = dx ? W : nullptr;
    a.x = dW ? x : nullptr;
    a.cos_tab = cos_tab;
    a.sin_tab = sin_tab;
    a.pos = pos;
    a.dx = dx;
    a.dW = dW;
    a.db = db;
    a.workspace = workspace;
    a.ws_bytes = ws_bytes;
    a.status = dev_status;
    a.wt = dx ? wt : nullptr;
    a.wt_s = dx ? wt_s : nullptr;
    // T == 0: dx is empty; dW = 0 and db = 0 are written
    return launch_bwd_mxfp8(a, static_cast<cudaStream_t>(stream));
}

extern "C" {

MLAQ_API int mla_q_uproj_bwd_mxfp8(const mla_q_shape* shape, const void* dq, const void* W, const void* x,
                                   const float* cos_tab, const float* sin_tab, const int32_t* pos, void* dx,
                                   void* dW, void* db, void* workspace, size_t ws_bytes, int* dev_status,
                                   void* stream) {
    return bwd_mxfp8_call(shape, dq, W, nullptr, nullptr, x, cos_tab, sin_tab, pos, dx, dW, db, workspace,
                          ws_bytes, dev_status, stream);
}

MLAQ_API int mla_q_uproj_bwd_mxfp8_prepared(const mla_q_shape* shape, const void* dq, const uint8_t* wt,
                                            const uint8_t* wt_scales, const void* x, const float* cos_tab,
                                            const float* sin_tab, const int32_t* pos, void* dx, void* dW,
                                            void* db, void* workspace, size_t ws_bytes, int* dev_status,
                                            void* stream) {
    return bwd_mxfp8_call(shape, dq, nullptr, wt, wt_scales, x, cos_tab, sin_tab, pos, dx, dW, db, workspace,
                          ws_bytes, dev_status, stream);
}

MLAQ_API int mla_kv_uproj_fwd(const mla_kv_shape* shape, const void* c_kv, const void* W, const void* k_pe,
                              const float* cos_tab, const float* sin_tab, const int32_t* pos, void* o_key,
                              void* o_value, int* dev_status, void* stream) {
    if (!shape) return MLA_ERR_INVALID_ARG;
    const mla_kv_shape& s = *shape;
    if (s.T < 0 || s.K <= 0 || s.H <= 0 || s.Dn < 0 || s.Dv <= 0 || s.Dr <= 0 || (s.Dr & 1) ||
        s.cs_rows < 0 || s.cs_width < 0)
        return MLA_ERR_INVALID_ARG;
    const int64_t dkv = (int64_t)s.Dn + s.Dv, dk = (int64_t)s.Dn + s.Dr;
    if (dkv * s.H > kI32Max || dk * s.H > kI32Max || s.T > kI32Max || s.K > kI32Max) return MLA_ERR_INVALID_ARG;
    if (s.cs_rows > kI32Max || s.cs_width > kI32Max) return MLA_ERR_INVALID_ARG;
    if (s.cs_width < s.Dr) return MLA_ERR_ROPE_WIDTH;
    if (s.T > 0 && (!cos_tab || !sin_tab || !c_kv || !W || !k_pe || !o_key || !o_value))
        return MLA_ERR_INVALID_ARG;
    if (!pos && s.T > s.cs_rows) return MLA_ERR_POS_RANGE;
    if (s.cs_rows == 0 && s.T > 0) return MLA_ERR_POS_RANGE;
    if (s.T == 0) return MLA_OK;
    if (!rope_dim_supported(s.Dr) || s.Dn % 32 || s.Dv % 32 || dkv > 256) return MLA_ERR_UNSUPPORTED;
    if (s.K % 8) return MLA_ERR_ALIGNMENT;
    if (!aligned(c_kv, 16) || !aligned(W, 16) || !aligned(k_pe, 16) || !aligned(o_key, 16) ||
        !aligned(o_value, 16) || !aligned(cos_tab, 4) || !aligned(sin_tab, 4) || !aligned(pos, 4) ||
        !aligned(dev_status, 4))
        return MLA_ERR_ALIGNMENT;
    const int64_t table = s.cs_rows * s.cs_width * 4;
    const Range outs[] = {rng(o_key, s.T * s.H * dk * 2), rng(o_value, s.T * s.H * s.Dv * 2), rng(dev_status, 4)};
    const Range ins[] = {rng(c_kv, s.T * s.K * 2), rng(W, dkv * s.H * s.K * 2), rng(k_pe, s.T * s.Dr * 2),
                         rng(cos_tab, table), rng(sin_tab, table), rng(pos, s.T * 4)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    KvArgs a{};
    a.T = s.T;
    a.K = s.K;
    a.H = s.H;
    a.Dn = s.Dn;
    a.Dv = s.Dv;
    a.Dr = s.Dr;
    a.cs_rows = s.cs_rows;
    a.cs_width = s.cs_width;
    a.c_kv = c_kv;
    a.W = W;
    a.k_pe = k_pe;
    a.cos_tab = cos_tab;
    a.sin_tab = sin_tab;
    a.pos = pos;
    a.o_key = o_key;
    a.o_value = o_value;
    a.status = dev_status;
    return launch_kv_fwd(a, static_cast<cudaStream_t>(stream));
}

MLAQ_API int mxfp8_quantize_rows(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                 uint8_t* codes, uint8_t* scales, void* stream) {
    if (R < 0 || C < 0 || ld_in < C) return MLA_ERR_INVALID_ARG;
    if (in_dtype != MLA_IN_F32 && in_dtype != MLA_IN_BF16) return MLA_ERR_INVALID_ARG;
    if (R == 0 || C == 0) return MLA_OK;
    if (!in || !codes || !scales) return MLA_ERR_INVALID_ARG;
    const int64_t esz = in_dtype == MLA_IN_F32 ? 4 : 2;
    if (!aligned(in, (uintptr_t)esz)) return MLA_ERR_ALIGNMENT;
    const int64_t nb = (C + 31) / 32;
    const Range outs[] = {rng(codes, R * C), rng(scales, R * nb)};
    const Range ins[] = {rng(in, ((R - 1) * ld_in + C) * esz)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    return launch_mxfp8_quantize(R, C, in_dtype, in, ld_in, codes, scales,
                                 static_cast<cudaStream_t>(stream));
}

MLAQ_API int mxfp8_quantize_rows_tiled(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                       uint8_t* codes, uint8_t* scales, int64_t group, void* stream) {
    if (R < 0 || C < 0 || ld_in < C || group <= 0) return MLA_ERR_INVALID_ARG;
    if (in_dtype != MLA_IN_F32 && in_dtype != MLA_IN_BF16) return MLA_ERR_INVALID_ARG;
    if (R == 0 || C == 0) return MLA_OK;
    if (!in || !codes || !scales) return MLA_ERR_INVALID_ARG;
    const int64_t esz = in_dtype == MLA_IN_F32 ? 4 : 2;
    if (!aligned(in, (uintptr_t)esz)) return MLA_ERR_ALIGNMENT;
    const int64_t nb = (C + 31) / 32;
    const Range outs[] = {rng(codes, R * C), rng(scales, (int64_t)sf_tiled_bytes(R, nb, group))};
    const Range ins[] = {rng(in, ((R - 1) * ld_in + C) * esz)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    return launch_mxfp8_quantize(R, C, in_dtype, in, ld_in, codes, scales, static_cast<cudaStream_t>(stream),
                                 group);
}

MLAQ_API int mxfp8_quantize_cols(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                 uint8_t* codes_t, uint8_t* scales_t, void* stream) {
    if (R < 0 || C < 0 || ld_in < C) return MLA_ERR_INVALID_ARG;
    if (in_dtype != MLA_IN_F32 && in_dtype != MLA_IN_BF16) return MLA_ERR_INVALID_ARG;
    if (R == 0 || C == 0) return MLA_OK;
    if (!in || !codes_t || !scales_t) return MLA_ERR_INVALID_ARG;
    const int64_t esz = in_dtype == MLA_IN_F32 ? 4 : 2;
    if (!aligned(in, (uintptr_t)esz)) return MLA_ERR_ALIGNMENT;
    const int64_t nbr = (R + 31) / 32;
    const Range outs[] = {rng(codes_t, C * R), rng(scales_t, C * nbr)};
    const Range ins[] = {rng(in, ((R - 1) * ld_in + C) * esz)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    return launch_mxfp8_quantize_cols(R, C, in_dtype, in, ld_in, codes_t, scales_t,
                                      static_cast<cudaStream_t>(stream));
}

MLAQ_API int mxfp8_quantize_cols_tiled(int64_t R, int64_t C, int in_dtype, const void* in, int64_t ld_in,
                                       uint8_t* codes_t, uint8_t* scales_t, int64_t group, void* stream) {
    if (R < 0 || C < 0 || ld_in < C || group <= 0) return MLA_ERR_INVALID_ARG;
    if (in_dtype != MLA_IN_F32 && in_dtype != MLA_IN_BF16) return MLA_ERR_INVALID_ARG;
    if (R == 0 || C == 0) return MLA_OK;
    if (!in || !codes_t || !scales_t) return MLA_ERR_INVALID_ARG;
    const int64_t esz = in_dtype == MLA_IN_F32 ? 4 : 2;
    if (!aligned(in, (uintptr_t)esz)) return MLA_ERR_ALIGNMENT;
    // the tiled scale order is written by the tiled kernel only (16-byte rows)
    if (!aligned(in, 16) || (ld_in * esz) % 16 || C % (16 / esz)) return MLA_ERR_UNSUPPORTED;
    const int64_t nbr = (R + 31) / 32;
    const int64_t sbytes = (int64_t)sf_tiled_bytes(C, nbr, group);
    const Range outs[] = {rng(codes_t, C * R), rng(scales_t, sbytes)};
    const Range ins[] = {rng(in, ((R - 1) * ld_in + C) * esz)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the kernel writes the real (row, block) entries; padding rows of a
    // group's last 128-row tile and padding columns read as 0
    if (group % 128 || C % group || nbr % 4) {
        if (cudaMemsetAsync(scales_t, 0, (size_t)sbytes, s) != cudaSuccess) return MLA_ERR_CUDA;
    }
    return launch_mxfp8_quantize_cols_tiled_sf(R, C, in_dtype, in, ld_in, codes_t, R, scales_t, group, s);
}

MLAQ_API size_t mxfp8_swizzled_scale_bytes(int64_t rows, int64_t cols) {
    if (rows <= 0 || cols <= 0) return 0;
    return (size_t)((rows + 127) / 128) * 128 * (size_t)((cols + 3) / 4) * 4;
}

MLAQ_API size_t mxfp8_grouped_scale_bytes(int64_t rows, int64_t cols, int64_t group) {
    if (rows <= 0 || cols <= 0 || group <= 0) return 0;
    return (size_t)sf_tiled_bytes(rows, cols, group);
}

MLAQ_API int mxfp8_swizzle_scales_grouped(int64_t rows, int64_t cols, int64_t group, const uint8_t* in,
                                          int64_t ld_in, uint8_t* out, void* stream) {
    if (rows < 0 || cols < 0 || ld_in < cols || group <= 0) return MLA_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return MLA_OK;
    if (!in || !out) return MLA_ERR_INVALID_ARG;
    if (!aligned(out, 16)) return MLA_ERR_ALIGNMENT;
    const Range outs[] = {rng(out, (int64_t)mxfp8_grouped_scale_bytes(rows, cols, group))};
    const Range ins[] = {rng(in, (rows - 1) * ld_in + cols)};
    if (any_alias(outs, ins)) return MLA_ERR_ALIAS;
    return launch_mxfp8_swizzle(rows, cols, group, in, ld_in, out, static_cast<cudaStream_t>(stream));
}

MLAQ_API int mxfp8_swizzle_scales(int64_t rows, int64_t cols, const uint8_t* in, int64_t ld_in, uint8_t* out,
                                  void* stream) {
    return mxfp8_swizzle_scales_grouped(rows, cols, 128, in, ld_in, out, stream);
}

MLAQ_API int64_t mla_q_uproj_w_scale_group(const mla_q_shape* shape) {
    int D;
    int64_t N;
    if (check_shape(shape, &D, &N) != MLA_OK || !rope_dim_supported(shape->Dr) || shape->Dn % 32) return 0;
    return fwd_tile_n(N, D, shape->Dn, shape->Dr, 192, 32);
}

}  // extern "C"
