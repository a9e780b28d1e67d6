// selftest.cu -- hypic_selftest_bounded_wait: runs the bounded mbarrier wait
// and abort protocol of the pipelined kernels against a barrier that nothing
// completes, so that its failure path can be tested without a fault.
#include "kernels.h"
#include "tc_util.cuh"

namespace hypic {
int report_error(int code, const char *msg);  // api.cu: sets hypic_last_error()
int async_status_word(int **out);             // api.cu: this device's status word
}

namespace {

// Thread 0 waits with the given limit and gives up first, raising the CTA's
// abort flag; thread 32 (another warp) waits on the same barrier with a limit
// 64 times longer and must leave as soon as it sees the flag.  Status bits: 1
// the flag was raised, 2 the second waiter left without the phase completing.
__global__ void wait_probe_kernel(int *status, long long max_cycles)
{
    __shared__ __align__(8) uint64_t mbar;
    __shared__ int abort_flag;
    const int tid = threadIdx.x;
    const uint32_t mb = hypic::tc::smem_u32(&mbar);
    if (tid == 0) {
        hypic::tc::mbar_init(mb, 1);
        abort_flag = 0;
        hypic::tc::fence_mbar_init();
    }
    __syncthreads();
    volatile int *af = &abort_flag;
    bool ok = true;
    if (tid == 0) ok = hypic::tc::wait_bounded(mb, 0, af, max_cycles);
    else if (tid == 32) ok = hypic::tc::wait_bounded(mb, 0, af, 64 * max_cycles);
    __syncthreads();
    if (tid == 0 && *af) atomicOr(status, 1);
    if (tid == 32 && !ok) atomicOr(status, 2);
}

}  // namespace

extern "C" int hypic_selftest_bounded_wait(void *workspace, int64_t max_cycles, hypic_stream stream)
{
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255) != 0)
        return hypic::report_error(HYPIC_ERR_WORKSPACE, "workspace must be a 256-byte aligned device pointer");
    if (max_cycles < 1 || max_cycles > ((int64_t)1 << 34))
        return hypic::report_error(HYPIC_ERR_SHAPE, "max_cycles out of [1, 2^34]");
    // with a workspace: its status word (read by hypic_workspace_status); without:
    // the device's word that compose and seam advance report to (hypic_async_status)
    int *status = nullptr;
    if (workspace) {
        status = reinterpret_cast<int *>(static_cast<char *>(workspace) + 128);
    } else {
        const int rc = hypic::async_status_word(&status);
        if (rc != HYPIC_OK) return rc;
    }
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), (cudaStream_t)stream);
    if (e == cudaSuccess) {
        wait_probe_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(status, (long long)max_cycles);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return hypic::report_error(HYPIC_ERR_CUDA, cudaGetErrorString(e));
    hypic::report_error(HYPIC_OK, "");
    return HYPIC_OK;
}
