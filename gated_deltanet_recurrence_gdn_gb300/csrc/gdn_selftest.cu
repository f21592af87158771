// gdn_selftest.cu -- device self-test of the bounded waits (gdn_selftest.h).
//
// One CTA waits, through the control block the pipelined kernels use (Ctl),
// on an mbarrier phase and on a release/acquire counter in shared memory.
// Either the CTA completes both itself before waiting (the waits must
// succeed, no error recorded), or nothing ever completes them (each wait
// must give up after its poll limit and record a timeout in the device error
// word).  No fault, trap or unbounded loop is involved: the failure is a
// phase that nobody completes, and the kernel always returns.
#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_selftest.h"
#include "gdn_internal.h"
#include "tc_common.cuh"

namespace gdn {
namespace {

constexpr long long kMaxSelftestLimit = 1LL << 22;

// whether each wait succeeded (1) or gave up (0), for the host to read back
__device__ int g_selftest_out[2];

__global__ void __launch_bounds__(32, 1)
k_wait_selftest(int complete, uint32_t limit, int *err, int *out) {
    __shared__ uint64_t bar[1];
    __shared__ uint32_t counter;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar, 1);
        counter = 0;
        abort_flag = 0;
        ptx::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    if (complete) {
        ptx::mbar_arrive(bar);              // the one expected arrival: phase 0 completes
        ptx::st_release_cta(&counter, 1u);
    }
    const tcx::Ctl ctl{bar, &abort_flag, err, limit};
    const bool bar_ok = ctl.wait(0, 0);
    abort_flag = 0;                         // let the second wait run as well
    const bool flag_ok = ctl.flag(&counter, 1u);
    out[0] = bar_ok ? 1 : 0;
    out[1] = flag_ok ? 1 : 0;
}

}  // namespace
}  // namespace gdn

extern "C" gdn_status gdn_selftest_wait(int complete, long long limit, int *waits_ok,
                                        void *stream) {
    if ((complete != 0 && complete != 1) || limit < 1 || limit > gdn::kMaxSelftestLimit)
        return GDN_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int *err = gdn::device_error_word();
    int *out = nullptr;
    if (!err || cudaGetSymbolAddress(reinterpret_cast<void **>(&out), gdn::g_selftest_out) !=
                    cudaSuccess)
        return GDN_ERR_CUDA;
    gdn::k_wait_selftest<<<1, 32, 0, st>>>(complete, static_cast<uint32_t>(limit), err, out);
    gdn::count_launch();
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    int host[2] = {0, 0};
    if (cudaMemcpyAsync(host, out, sizeof(host), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
        return GDN_ERR_CUDA;
    if (waits_ok) {
        waits_ok[0] = host[0];
        waits_ok[1] = host[1];
    }
    return GDN_OK;
}
