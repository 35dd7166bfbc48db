// selftest.cu -- moe_selftest_wait_timeout: runs the bounded mbarrier waits of the tensor-core
// kernels on a barrier that nothing ever completes, so the failure path (give up after the
// limit, raise the abort flag, report MOE_DEVERR_TIMEOUT in the workspace error word, return
// with the context intact) can be checked on a GPU without hanging or faulting it.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

__global__ void __launch_bounds__(64)
wait_timeout_kernel(uint64_t timeout_ns, int32_t* err) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);                 // count 1, and nobody will arrive
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    bool ok1 = true, okw = true;
    if (threadIdx.x == 0)                   // the single-thread wait (producer / MMA roles)
        ok1 = wait1(&bar, 0, &abort_flag, timeout_ns, true);
    if (threadIdx.x >= 32)                  // the warp-wide wait (epilogue role)
        okw = waitw(&bar, 0, &abort_flag, timeout_ns);
    __syncthreads();
    if (threadIdx.x == 0 && (!ok1 || abort_flag)) atomicOr(err, MOE_DEVERR_TIMEOUT);
    if (threadIdx.x == 32 && !okw) atomicOr(err, MOE_DEVERR_TIMEOUT);
}

}  // namespace
}  // namespace moe

extern "C" MOE_API moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes,
                                                        uint32_t timeout_us, void* stream) {
    if (!ws || reinterpret_cast<uintptr_t>(ws) % 256 || ws_bytes < 256) return MOE_ERR_WORKSPACE;
    if (timeout_us == 0 || timeout_us > 2000000u) return MOE_ERR_INVALID_ARG;
    moe::wait_timeout_kernel<<<1, 64, 0, (cudaStream_t)stream>>>((uint64_t)timeout_us * 1000ull,
                                                                  static_cast<int32_t*>(ws));
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
