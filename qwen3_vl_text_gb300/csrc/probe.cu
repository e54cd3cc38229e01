// Failure-detection self-test: a one-thread kernel that waits, through the same
// bounded-wait helpers every kernel of the library uses, on something that may
// never happen (a device flag or an mbarrier nobody arrives on).  When the wait
// gives up it records ST_TIMEOUT in the status word and returns, so the host
// learns of the stall from the status and the CUDA context stays usable.  No
// counterpart on the pages: it tests the library's own failure detection.
#include "../../include/h3enc_ops.h"
#include "common.cuh"
#include "kernels.h"

namespace {

__global__ void wait_probe_kernel(const uint32_t *flag, uint32_t expect, int use_mbarrier, int32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int never;
    if (use_mbarrier) {
        h3::mbar_init(&bar, 1);   // expects one arrival; none comes
        never = 0;
        h3::fence_barrier_init();
        if (!h3::mbar_wait(&bar, 0, &never)) h3::report(status, h3::ST_TIMEOUT);
        return;
    }
    const long long t0 = clock64();
    while (*reinterpret_cast<const volatile uint32_t *>(flag) != expect) {
        if (clock64() - t0 > h3::kSpinLimitCycles) {
            h3::report(status, h3::ST_TIMEOUT);
            return;
        }
    }
}

}  // namespace

extern "C" {

H3ENC_API h3enc_status h3enc_op_wait_probe(const uint32_t *flag, uint32_t expect, int32_t use_mbarrier,
                                           int32_t *status, void *stream) {
    if (!status || (!use_mbarrier && !flag)) return H3ENC_ERR_INVALID_ARG;
    wait_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(flag, expect, use_mbarrier, status);
    return cudaGetLastError() == cudaSuccess ? H3ENC_OK : H3ENC_ERR_CUDA;
}

}  // extern "C"
