// k_selftest.cu -- self-test of the bounded waits every tensor-core kernel
// uses: one thread waits on a shared-memory barrier that nothing arrives at.
// The wait must give up after its limit, latch the timeout status bit and let
// the kernel return, leaving the CUDA context usable.
#include "gdn_internal.cuh"
#include "tc.cuh"

namespace gdn {
namespace {

__global__ void wait_timeout_kernel(int32_t *status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    const uint64_t t0 = tc::globaltimer();
    const bool landed = tc::mbar_wait_ns(&bar, 0, limit_ns);  // no arrival will ever come
    const uint64_t waited = tc::globaltimer() - t0;
    if (!landed) atomicOr(status + 2, kStatusTimeout);
    status[3] = (int32_t)(waited / 1000000ull);  // milliseconds waited
}

}  // namespace
}  // namespace gdn

using namespace gdn;

extern "C" gdn_status gdn_selftest_wait_timeout(int32_t *status, int32_t limit_ms, void *stream) {
    if (!status) return GDN_ERR_NULL;
    if (limit_ms < 1 || limit_ms > 2000) return GDN_ERR_SHAPE;
    if (cudaMemsetAsync(status, 0, 4 * sizeof(int32_t), (cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(status, (uint64_t)limit_ms * 1000000ull);
    if (cudaGetLastError() != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    int32_t host[4];
    if (cudaMemcpy(host, status, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess) return GDN_ERR_CUDA;
    // as designed: the wait gave up (timeout bit) after at least its limit
    return ((host[2] & kStatusTimeout) && host[3] >= limit_ms) ? GDN_OK : GDN_ERR_DEVICE;
}
