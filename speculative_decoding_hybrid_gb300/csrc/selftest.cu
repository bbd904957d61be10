// Self-test of the bounded wait used by every kernel that waits on an
// asynchronous copy or tensor-core operation: one thread waits on an mbarrier
// that nothing will ever arrive at, gives up after the given time and reports
// GDN_DEV_TIMEOUT in the status word, leaving the context usable.  No fault,
// trap or unbounded loop is involved.
#include "common.cuh"

namespace {
__global__ void wait_timeout_kernel(uint32_t *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    gdn::mbar_init(&bar, 1);  // expects one arrival that never comes
    if (!gdn::mbar_wait_bounded(&bar, 0, limit_ns)) gdn::set_status(status, GDN_DEV_TIMEOUT);
}
}  // namespace

extern "C" int gdn_selftest_wait_timeout(uint32_t *dev_status, uint64_t limit_ns, void *stream) {
    if (!dev_status) return GDN_ERR_NULL;
    if (limit_ns == 0 || limit_ns > gdn::kWaitLimitNs) return GDN_ERR_ARG;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status, limit_ns);
    return gdn_host::launch_status(cudaGetLastError());
}
