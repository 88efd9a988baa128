// Failure-detection self-test (gdn_selftest_wait_timeout): exercises the path a
// kernel takes when one of its bounded waits runs out, without any fault.  One
// thread waits on an mbarrier that nothing ever arrives on, with the same
// bounded wait the kernels use; when the limit passes it records GDN_ERR_TIMEOUT
// in the device status word and the kernel returns normally, so the context
// stays usable and gdn_last_error() reports the timeout.
#include "../../include/gdn.h"
#include "gdn_internal.h"
#include "ptx.cuh"

namespace gdn {
namespace {

__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !ptx::mbar_wait(ptx::smem_u32(&bar), 0, limit_ns)) report_device_error(status, kTimeout);
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_selftest_wait_timeout(unsigned int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 10000000u) return GDN_ERR_INVALID_ARG;
  unsigned int* status = gdn::device_status_word();
  if (!status) return GDN_ERR_CUDA;
  gdn::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status,
                                                                              1000ull * timeout_us);
  return cudaGetLastError() == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}
