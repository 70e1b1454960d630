// Test hooks of libmgg that launch kernels of their own (declared in include/mgg_testing.h).
//
// mgg_test_wait_timeout: a kernel that waits on an mbarrier which nothing ever arrives on, through
// the same bounded-wait code the grouped GEMM pipelines use, with a caller-chosen limit.  The wait
// gives up after that limit, records MGG_ERR_DEVICE_TIMEOUT with the waiting role's code in the
// status word, raises the CTA's abort flag, and the kernel returns: it issues no TMA copy and no
// MMA, and nothing in it can wait without a limit.
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "mgg.h"
#include "mgg_internal.h"
#include "mgg_ptx.cuh"
#include "mgg_testing.h"

namespace mgg {
namespace {

// status[0..3] = {status, where, detail, flags}; flags bit 0: the first wait returned false, bit 1:
// a second wait after the abort returned false at once, bit 2: that second wait left the status
// word as the first one wrote it.
__global__ void wait_timeout_probe_kernel(int* status, unsigned long long limit_ns, int where, int cluster) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    if (blockIdx.x == 0) {
      status[0] = status[1] = status[2] = status[3] = 0;
    }
  }
  __syncthreads();
  if (threadIdx.x != 0 || blockIdx.x != 0) return;  // one waiting thread (the other CTA of a cluster idles)
  const WaitGuard g{&abort_flag, status};
  const uint32_t a = smem_u32(&bar);
  // nothing arrives on `bar`: phase 0 never completes
  const bool ok1 = cluster ? mbar_wait_bounded<true>(a, 0, g, where, limit_ns)
                           : mbar_wait_bounded<false>(a, 0, g, where, limit_ns);
  const int where_after_first = status[1];
  // the abort flag is up: a later wait of this CTA returns false without polling to its limit
  const unsigned long long t0 = globaltimer_ns();
  const bool ok2 = mbar_wait_bounded<false>(a, 0, g, where + 1, limit_ns);
  const bool quick = globaltimer_ns() - t0 < limit_ns;
  status[3] = (ok1 ? 0 : 1) | ((!ok2 && quick) ? 2 : 0) | (status[1] == where_after_first ? 4 : 0);
}

// One thread checks `value` against [0, limit) exactly as the kernels check their indices: in the
// bounds-checked build a value outside records MGG_ERR_DEVICE_BOUNDS (where 501, the value) and the
// guarded "access" (status[3] = 1) is skipped; in the normal build the check compiles away.
__global__ void bounds_probe_kernel(int* status, long long value, long long limit) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  if (MGG_IN_BOUNDS(status, value >= 0 && value < limit, 501, value)) status[3] = 1;
}

}  // namespace
}  // namespace mgg

using namespace mgg;

extern "C" mgg_status mgg_test_bounds_check(void* status_dev, int64_t value, int64_t limit, void* stream) {
  if (status_dev == nullptr || (reinterpret_cast<uintptr_t>(status_dev) & 15u) != 0) {
    set_last_error("status_dev must be a 16-byte aligned device buffer of 4 int32");
    return MGG_ERR_VALUE;
  }
  bounds_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int*>(status_dev),
                                                                       (long long)value, (long long)limit);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_last_error(std::string("bounds probe launch: ") + cudaGetErrorString(e));
    return MGG_ERR_RUNTIME;
  }
  return MGG_OK;
}

extern "C" mgg_status mgg_test_wait_timeout(void* status_dev, int64_t limit_ns, int32_t where, int32_t cluster,
                                            void* stream) {
  if (status_dev == nullptr || (reinterpret_cast<uintptr_t>(status_dev) & 15u) != 0) {
    set_last_error("status_dev must be a 16-byte aligned device buffer of 4 int32");
    return MGG_ERR_VALUE;
  }
  if (limit_ns <= 0 || limit_ns > 100000000) {  // at most 0.1 s
    set_last_error("limit_ns must be in (0, 1e8]");
    return MGG_ERR_VALUE;
  }
  if (cluster != 0 && cluster != 1) {
    set_last_error("cluster must be 0 or 1");
    return MGG_ERR_VALUE;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(cluster ? 2u : 1u, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = static_cast<cudaStream_t>(stream);
  if (cluster) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const cudaError_t e = cudaLaunchKernelEx(&cfg, wait_timeout_probe_kernel, static_cast<int*>(status_dev),
                                           (unsigned long long)limit_ns, (int)where, (int)cluster);
  if (e != cudaSuccess) {
    set_last_error(std::string("wait-timeout probe launch: ") + cudaGetErrorString(e));
    return MGG_ERR_RUNTIME;
  }
  return MGG_OK;
}

extern "C" int mgg_test_build_flags(void) {
#ifdef MGG_CHECKED
  return 1;
#else
  return 0;
#endif
}
