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

// ------------------------------------------------------------------ backward GEMM engine

#include "bwd_internal.cuh"

namespace moe {
namespace {
__global__ void selftest_plan_kernel(int32_t* plan, int K) {
    if (threadIdx.x == 0) {
        plan[0] = K;        // rows of the single group
        plan[1] = 0;        // a_off
        plan[2] = K;
        plan[3] = 0;        // c_off
        plan[4] = K;
        plan[5] = 0;        // dense_off
    }
}
}  // namespace
}  // namespace moe

extern "C" MOE_API moe_status moe_selftest_gemm(int32_t a_mn, int32_t b_mn, int32_t M, int32_t N,
                                                int32_t K, const void* A, const void* B, float* C,
                                                void* ws, size_t ws_bytes, void* stream) {
    if (!ws || reinterpret_cast<uintptr_t>(ws) % 256 || ws_bytes < 512) return MOE_ERR_WORKSPACE;
    if (M <= 0 || N <= 0 || K <= 0 || (a_mn != 0 && a_mn != 1) || (b_mn != 0 && b_mn != 1))
        return MOE_ERR_INVALID_ARG;
    if (!A || !B || !C || reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16 ||
        reinterpret_cast<uintptr_t>(C) % 16)
        return MOE_ERR_INVALID_ARG;
    // 16-byte rows of the two bf16 operands and of C
    if ((a_mn ? M : K) % 8 || (b_mn ? N : K) % 8 || N % 4) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int32_t* plan = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + 256);
    moe::selftest_plan_kernel<<<1, 32, 0, s>>>(plan, K);
    cudaError_t e = moe::tb_selftest(a_mn != 0, b_mn != 0, M, N, K, (const __nv_bfloat16*)A,
                                     (const __nv_bfloat16*)B, C, plan, static_cast<int32_t*>(ws), s);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
