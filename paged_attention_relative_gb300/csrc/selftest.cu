// Self-test of the bounded-wait path: one thread waits on an mbarrier that
// nothing ever arrives on, gives up after the given time, records its site in
// the device error word and returns, exactly as the attention kernels do when
// a hand-off never comes.  Declared in include/rel_attn_profile.h.

#include "common.cuh"
#include "rel_attn.h"
#include "rel_attn_profile.h"

namespace relattn {

int* device_error_word();
void set_last_error_message(const char* msg);

namespace {

__global__ void wait_timeout_kernel(uint64_t timeout_ns, int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, timeout_ns, kSiteSelfTest, err);  // never satisfied
    __syncthreads();
}

}  // namespace
}  // namespace relattn

extern "C" rel_attn_status rel_attn_check_wait_timeout(int32_t timeout_ms, rel_attn_stream stream) {
    using namespace relattn;
    if (timeout_ms < 1 || timeout_ms > 10000) {
        set_last_error_message("rel_attn_check_wait_timeout: timeout_ms must be in [1, 10000]");
        return REL_ATTN_ERR_INVALID_ARGUMENT;
    }
    int* err = device_error_word();
    if (!err) return REL_ATTN_ERR_CUDA;  // the message names the failing CUDA call
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>((uint64_t)timeout_ms * 1000000ull, err);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_last_error_message(cudaGetErrorString(e));
        return REL_ATTN_ERR_CUDA;
    }
    return REL_ATTN_OK;
}
