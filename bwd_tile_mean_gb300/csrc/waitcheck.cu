// waitcheck.cu -- exercises the bounded mbarrier wait that every tcgen05
// kernel of the library uses, on a barrier that nothing ever arrives on:
// the wait gives up after the given wall time, records its site code in
// the caller's status word and returns, leaving the context usable. Used
// to test the failure path without faulting or hanging the GPU.
#include "sm103_ptx.cuh"
#include "vsa.h"
#include "vsa_internal.h"

namespace vsa {
namespace {

constexpr unsigned kSiteSelfTest = 0x7E57;

__global__ void __launch_bounds__(32) k_wait_timeout(unsigned *err, unsigned long long limit_ns, int *out) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);  // one arrival expected, none ever made
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncwarp();
    const bool ok = ptx::mbar_wait(&bar, 0, &abort_flag, err, kSiteSelfTest, limit_ns);
    if (threadIdx.x == 0) out[0] = ok ? 1 : 0;
}

}  // namespace
}  // namespace vsa

using namespace vsa;

extern "C" vsa_status vsa_check_wait_timeout(void *workspace, unsigned long long limit_ns, int32_t *completed,
                                             vsa_stream_t stream) {
    if (!workspace || !completed) return VSA_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return VSA_ERR_WORKSPACE;
    if (limit_ns == 0 || limit_ns > 10000000000ull) return VSA_ERR_SHAPE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    prof_begin("wait_timeout_check", s);
    // the status word is the workspace's first 4 bytes; `completed` gets 1 if
    // the wait (wrongly) saw its phase complete, 0 after the timeout
    k_wait_timeout<<<1, 32, 0, s>>>(static_cast<unsigned *>(workspace), limit_ns, completed);
    prof_end(s);
    return status_from_cuda(cudaGetLastError());
}
