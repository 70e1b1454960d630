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
// * The first call on a device (set-up) looks up the array's device address
//   (cudaGetSymbolAddress) with that device current and remembers it together with the device's
//   current CUDA context.  A later call whose current context differs (the context was torn down
//   and created again, after cudaDeviceReset say, which can move the array) looks it up again, so
//   no call receives a stale address.  The set-up must not happen while the call's stream is being
//   captured: make one call on the device (and again after a context reset) before any capture.
// * All calls share the one array and it keeps the contents of the last call.  Calls whose
//   work may overlap on the GPU (other streams, other threads) race on it: order them.
// * Nothing in the array has to start at zero: the preparation kernel of every call rewrites
//   the status word, the expert order and the tensor map of every non-empty expert before the
//   main kernel reads them, so stale contents from an earlier call are never used.
// * No allocation happens: no cudaMalloc, cudaFree or allocating library call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "mgg.h"
#include "mgg_internal.h"

namespace {

constexpr int kNoAllocMaxExperts = 1024;
// The workspace of a 1024-expert mgg_wgrad call (header, three tensor maps and one order entry
// per expert), from the same formula mgg_wgrad_workspace_size uses.
constexpr size_t kNoAllocScratchBytes = mgg::wgrad_workspace_bytes(kNoAllocMaxExperts);
static_assert(kNoAllocScratchBytes == 397568, "the size stated in include/mgg.h");
static_assert(kNoAllocScratchBytes % 256 == 0, "the workspace alignment mgg_wgrad checks");

static __device__ __align__(256) unsigned char g_wgrad_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};  // the context each address was looked up in

// cuCtxGetCurrent through the runtime's driver entry point (the library links no driver stub).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

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
  // the runtime makes the device's primary context current on first use; cudaFree(0) is the
  // usual idiom for that, but it is an allocator call: the symbol lookup below does the same
  CtxGetCurrentFn get_ctx = ctx_get_current();
  if (get_ctx == nullptr) {
    mgg::set_last_error("mgg_wgrad_noalloc: cuCtxGetCurrent is not available from the CUDA driver");
    return MGG_ERR_RUNTIME;
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;
    if (g_scratch_addr[dev] == nullptr || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
      cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
      e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
      if (e != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
        mgg::set_last_error("mgg_wgrad_noalloc: the first call on a device (and the first after a context "
                            "reset) must come before any stream capture");
        return e != cudaSuccess ? MGG_ERR_RUNTIME : MGG_ERR_VALUE;
      }
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_wgrad_scratch);
      if (e != cudaSuccess || p == nullptr) {
        mgg::set_last_error(std::string("mgg_wgrad_noalloc: cannot resolve the scratch array on device ") +
                            std::to_string(dev) + ": " + cudaGetErrorString(e));
        return MGG_ERR_RUNTIME;
      }
      if (get_ctx(&ctx) != CUDA_SUCCESS) ctx = nullptr;  // the lookup made the primary context current
      g_scratch_addr[dev] = p;
      g_scratch_ctx[dev] = ctx;
    }
    scratch = g_scratch_addr[dev];
  }
  mgg_wgrad_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = (int64_t)kNoAllocScratchBytes;
  return mgg_wgrad(&a, stream);
}
