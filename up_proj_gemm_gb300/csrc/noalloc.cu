// dgrad for callers that cannot allocate device memory.
//
// mla_q_uproj_bwd_dgrad may need a workspace (the partial sums of split
// tiles, and without dq_pre_rope the rotated rope channels), and expects the
// caller to allocate it. Some callers cannot: a host framework that lends a
// plugin only the tensors of a call and owns every other byte of device
// memory, or a latency-critical path that cannot take cudaMalloc's implicit
// device-wide synchronization. This file gives them one entry point that
// takes inputs and outputs only and uses a scratch array of fixed size that
// the library holds in device global memory instead.
//
// The array below is file-scope device memory: every GPU that loads the
// library holds it until the process exits. In host code its name is only a
// host-side stand-in, not a device address, so the host looks the address
// up (cudaGetSymbolAddress, with the device current) the first time this
// entry point runs in a CUDA context, caches it for that context, and passes
// it to the kernels as their workspace.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace mlaq {
namespace {

static __device__ __align__(256) float g_dgrad_scratch[MLA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// The current CUDA context (the driver's handle), or nullptr.
CUcontext current_context() {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get = nullptr;
    std::call_once(once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    });
    CUcontext ctx = nullptr;
    if (!get || get(&ctx) != CUDA_SUCCESS) return nullptr;
    return ctx;
}

// Device address of g_dgrad_scratch in the current context (looked up once
// per device and context: a context created after a device reset gets a new
// lookup), or nullptr with MLA_ERR_CUDA in *err.
void* scratch_address(int* err) {
    static std::mutex mu;
    static void* addr[64] = {};
    static CUcontext ctx_of[64] = {};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *err = MLA_ERR_CUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    CUcontext ctx = current_context();
    if (!addr[dev] || !ctx || ctx_of[dev] != ctx) {
        void* p = nullptr;
        // (the lookup makes the device's primary context current if none is)
        if (cudaGetSymbolAddress(&p, g_dgrad_scratch) != cudaSuccess || !p) {
            *err = MLA_ERR_CUDA;
            return nullptr;
        }
        addr[dev] = p;
        ctx_of[dev] = ctx ? ctx : current_context();
    }
    return addr[dev];
}

}  // namespace
}  // namespace mlaq

extern "C" MLAQ_API int mla_q_uproj_bwd_dgrad_noalloc(const mla_q_shape* shape, const void* dq,
                                                      const void* W, const float* cos_tab,
                                                      const float* sin_tab, const int32_t* pos, void* dx,
                                                      void* dq_pre_rope, int* dev_status, void* stream) {
    // The argument checks of the allocating entry point come first, so both
    // return the same code for a bad argument; then the size limit; then the
    // scratch stands in for the workspace, always whole, and dgrad takes the
    // fastest path whose workspace fits in it.
    int st = mlaq::dgrad_check_args(shape, dq, W, cos_tab, sin_tab, pos, dx, dq_pre_rope, dev_status);
    if (st != MLA_OK) return st;
    if (shape->T == 0)
        return mla_q_uproj_bwd_dgrad(shape, dq, W, cos_tab, sin_tab, pos, dx, dq_pre_rope, nullptr, 0, dev_status,
                                     stream);
    mlaq::DeviceInfo di;
    if (mlaq::current_device_info(&di) != MLA_OK)  // no usable device: the same remaining checks and error
        return mla_q_uproj_bwd_dgrad(shape, dq, W, cos_tab, sin_tab, pos, dx, dq_pre_rope, nullptr, 0, dev_status,
                                     stream);
    const size_t least = mlaq::dgrad_min_workspace_bytes(shape->T, shape->K, shape->H, shape->Dn, shape->Dr,
                                                        di.num_sms, dq_pre_rope != nullptr);
    if (least > MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;  // shape too large for the scratch
    int err = MLA_OK;
    void* scratch = mlaq::scratch_address(&err);
    if (!scratch) return err;
    return mla_q_uproj_bwd_dgrad(shape, dq, W, cos_tab, sin_tab, pos, dx, dq_pre_rope, scratch,
                                 MLA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
