// Self-test of the failure path: a kernel whose mbarrier wait can never
// complete, bounded exactly as the attention kernels bound their waits. The
// wait gives up, records its site in the workspace status word and returns;
// the host reads the status and the context stays usable. Nothing faults or
// hangs: this is how a stuck pipeline (a lost TMA transaction, a missing
// arrival) is reported instead of hanging the GPU.
#include "internal.h"
#include "ptx.cuh"
#include "flashmask.h"

namespace fm {
namespace {

// CTA 0 waits with `short_ns`; every other CTA with the library's own limit and
// leaves as soon as CTA 0's failure appears in the status word.
__global__ void __launch_bounds__(32) selftest_timeout_kernel(int32_t* status, uint64_t short_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none ever comes
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  const bool ok = blockIdx.x == 0 ? mbar_wait_for(b, 0, status, short_ns)
                                  : mbar_wait(b, 0, status);
  if (!ok) record_failure(status, kStatusTimeout, kSiteSelftest);
}

}  // namespace
}  // namespace fm

extern "C" fm_status flashmask_selftest_timeout(void* ws, size_t ws_bytes, long long limit_ns,
                                                int ctas, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 16)
    return FM_ERR_WORKSPACE;
  if (limit_ns < 1000000LL || limit_ns > 2000000000LL || ctas < 1 || ctas > 1024)
    return FM_ERR_INVALID_ARG;
  fm::selftest_timeout_kernel<<<ctas, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<int32_t*>(ws), static_cast<uint64_t>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? FM_OK : FM_ERR_CUDA;
}
