// Device self-test of the bounded pipeline waits.
//
// Every mbarrier wait in the GEMM kernels gives up after a time limit or
// when another role of the CTA has set the abort flag, and the CTA then
// records MLA_ERR_TIMEOUT in the caller's status word and returns. This
// kernel runs that mechanism on its own, with the same wait routine, so a
// test can make a wait run out on the device (a barrier nothing arrives at)
// and read the status on the host, with no copy or MMA in flight and the
// context left usable.
#include "internal.h"
#include "ptx.cuh"

namespace mlaq {
namespace {

// Two roles as in the GEMM kernels. Warp 0 waits for a stage that only
// `arrive` fills (the producer's part); warp 1 waits on a barrier that only
// warp 0's success releases. When warp 0 gives up it sets the abort flag and
// warp 1 leaves through it; warp 1's own limit (twice warp 0's) is a backstop.
__global__ void __launch_bounds__(64) wait_selftest_kernel(int arrive, uint64_t limit_ns, int* status) {
    __shared__ alignas(8) uint64_t bars[2];
    __shared__ int abort_flag;
    const uint32_t full = smem_u32(&bars[0]), done = smem_u32(&bars[1]);
    if (threadIdx.x == 0) {
        mbar_init(full, 1);
        mbar_init(done, 1);
        abort_flag = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    volatile int* ab = &abort_flag;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        if (arrive && lane == 0) mbar_arrive(full);
        __syncwarp();
        const bool ok = mbar_wait(full, 0, ab, limit_ns);
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(done);
    } else {
        mbar_wait(done, 0, ab, 2 * limit_ns);
    }
    __syncthreads();
    if (threadIdx.x == 0 && *ab) record_status(status, MLA_ERR_TIMEOUT);
}

// The cross-CTA flag wait of dgrad's stream-K owners (wait_flag_gpu), run
// on its own: warp 0 waits for a flag in global memory that warp 1 sets only
// when `set` is non-zero; warp 1 then waits on a barrier that only warp 0's
// success releases. One CTA; the flag is the file's own word, reset first.
__device__ unsigned g_selftest_flag;

__global__ void __launch_bounds__(64) flag_selftest_kernel(int set, uint64_t limit_ns, int* status) {
    __shared__ alignas(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t done = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        abort_flag = 0;
        fence_mbarrier_init();
        st_release_gpu(&g_selftest_flag, 0u);
    }
    __syncthreads();
    volatile int* ab = &abort_flag;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0) {
        bool ok = true;
        if (lane == 0) ok = wait_flag_gpu(&g_selftest_flag, 1u, ab, limit_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (ok && lane == 0) mbar_arrive(done);
    } else {
        if (set && lane == 0) st_release_gpu(&g_selftest_flag, 1u);
        mbar_wait(done, 0, ab, 2 * limit_ns);
    }
    __syncthreads();
    if (threadIdx.x == 0 && *ab) record_status(status, MLA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace mlaq

extern "C" MLAQ_API int mla_wait_selftest_flag(int set, uint64_t limit_ns, int* dev_status, void* stream) {
    if (dev_status == nullptr || (reinterpret_cast<uintptr_t>(dev_status) & 3)) return MLA_ERR_INVALID_ARG;
    if (limit_ns < 1000000ull || limit_ns > 1000000000ull) return MLA_ERR_INVALID_ARG;
    mlaq::flag_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(set != 0, limit_ns, dev_status);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

extern "C" MLAQ_API int mla_wait_selftest(int arrive, uint64_t limit_ns, int* dev_status, void* stream) {
    if (dev_status == nullptr || (reinterpret_cast<uintptr_t>(dev_status) & 3)) return MLA_ERR_INVALID_ARG;
    if (limit_ns < 1000000ull || limit_ns > 1000000000ull) return MLA_ERR_INVALID_ARG;
    mlaq::wait_selftest_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(arrive != 0, limit_ns,
                                                                                 dev_status);
    return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
