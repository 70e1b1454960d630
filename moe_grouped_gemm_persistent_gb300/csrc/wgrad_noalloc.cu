// mgg_wgrad_noalloc: the grouped wgrad for callers that cannot allocate device memory.
//
// Some callers cannot obtain a workspace: a plugin running inside a host program whose own
// memory manager owns the whole device heap (and forbids allocations behind its back), or a
// code path that must never call cudaMalloc because the allocation would synchronise the
// device in the middle of its work.  This entry point runs the same wgrad kernels with their
// scratch (status word, per-expert tensor maps, expert order) in a fixed array that lives in
// device memory as part of this library.
//
// Properties a caller must know:
// * The array holds kNoAllocScratchBytes bytes, enough for the largest expert count the
//   operation accepts (1024); every GPU on which the library is loaded keeps it until the
//   process exits.
// * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
//   with that device current; make that first call before any stream capture begins.
// * All calls share the one array and it keeps the contents of the last call.  Calls whose
//   work may overlap on the GPU (other streams, other threads) race on it: order them.
// * Nothing in the array has to start at zero: the preparation kernel of every call rewrites
//   the status word, the expert order and the tensor map of every non-empty expert before the
//   main kernel reads them, so stale contents from an earlier call are never used.
// * No allocation happens: no cudaMalloc, cudaFree or allocating library call.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "mgg.h"
#include "mgg_internal.h"

namespace {

constexpr int kNoAllocMaxExperts = 1024;
// 256-byte header + 3 tensor maps (128 B) per expert + 4-byte expert order entry, rounded to 256.
constexpr size_t kNoAllocScratchBytes =
    ((256 + 3 * 128 * (size_t)kNoAllocMaxExperts + 4 * (size_t)kNoAllocMaxExperts) + 255) / 256 * 256;

static __device__ __align__(256) unsigned char g_wgrad_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" mgg_status mgg_wgrad_noalloc(const mgg_wgrad_args* args, void* stream) {
  if (args == nullptr) {
    mgg::set_last_error("args is NULL");
    return MGG_ERR_VALUE;
  }
  if (args->L > kNoAllocMaxExperts || mgg_wgrad_workspace_size(args->L) > kNoAllocScratchBytes) {
    mgg::set_last_error("mgg_wgrad_noalloc: " + std::to_string((long long)args->L) +
                        " experts exceed its fixed scratch (" + std::to_string(kNoAllocMaxExperts) + " experts, " +
                        std::to_string(kNoAllocScratchBytes) + " bytes)");
    return MGG_ERR_VALUE;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    mgg::set_last_error(std::string("mgg_wgrad_noalloc: no usable CUDA device: ") + cudaGetErrorString(e));
    return MGG_ERR_ARCH;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_wgrad_scratch);
      if (e != cudaSuccess || p == nullptr) {
        mgg::set_last_error(std::string("mgg_wgrad_noalloc: cannot resolve the scratch array on device ") +
                            std::to_string(dev) + ": " + cudaGetErrorString(e));
        return MGG_ERR_RUNTIME;
      }
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  mgg_wgrad_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = (int64_t)kNoAllocScratchBytes;
  return mgg_wgrad(&a, stream);
}
