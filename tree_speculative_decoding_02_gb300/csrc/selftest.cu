// selftest.cu -- ddt_wait_selftest: the failure path of the bounded device waits.
//
// Every pipeline barrier of the tensor-core kernels is waited on with a limit (tc::mbar_wait:
// about one second of SM clock cycles, then an abort flag and an error status instead of a
// hang).  This kernel runs that same wait on an mbarrier that nothing arrives on, so the
// limit is reached on purpose and the outcome can be checked from the host, with no fault
// and no stuck SM: the kernel returns normally after the wait gives up.
#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace ddt {

__global__ void k_wait_selftest(int32_t* __restrict__ status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    tc::mbar_init(&bar, 1);  // one arrival expected; none ever comes
    abort_flag = 0;
    tc::fence_mbar_init();
    const bool done = tc::mbar_wait(&bar, 0, &abort_flag);
    status[0] = done ? DDT_OK : (abort_flag ? DDT_ERR_TIMEOUT : DDT_ERR_CUDA);
}

cudaError_t launch_wait_selftest(int32_t* status, cudaStream_t st) {
    k_wait_selftest<<<counted(1), 1, 0, st>>>(status);
    return cudaGetLastError();
}

}  // namespace ddt
