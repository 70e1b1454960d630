// C ABI of libmgg: host-side validation, TMA descriptor encoding, device checks, launch.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <string>

#include "mgg.h"
#include "mgg_internal.h"
#include "mgg_testing.h"

namespace mgg {
namespace {

thread_local std::string g_err;

mgg_status fail(mgg_status s, const std::string& msg) {
  g_err = msg;
  return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// `p`, or the (always valid) workspace when `p` is NULL: the base of a tensor map that no copy uses.
const void* or_ws(const void* p, const void* workspace) { return p != nullptr ? p : workspace; }
void* or_ws(void* p, void* workspace) { return p != nullptr ? p : workspace; }

size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

// ---------------------------------------------------------------- driver entry point
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

CUtensorMapDataType tmap_dtype(int d) {
  return d == MGG_FP32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                       : d == MGG_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
}

// Tiled map with 128-byte swizzle; dims[0] innermost; strides in bytes for dims 1..rank-1.
// `promotion`: how much L2 fetches around a missed line (256 bytes suits the operands, whose next
// k-slice reads the neighbouring 128 bytes of each row a moment later).
mgg_status encode_map(CUtensorMap* map, int dtype, const void* addr, int rank, const uint64_t* dims,
                      const uint64_t* strides, const uint32_t* box, const char* what,
                      CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(MGG_ERR_RUNTIME, "cuTensorMapEncodeTiled is not available from the CUDA driver");
  if (rank < 1 || rank > 4) return fail(MGG_ERR_RUNTIME, std::string("tensor map rank out of range for the ") + what);
  cuuint64_t gdim[4], gstr[3];
  cuuint32_t bdim[4], estr[4] = {1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) gstr[i] = strides[i];
  const CUresult r = fn(map, tmap_dtype(dtype), (cuuint32_t)rank, const_cast<void*>(addr), gdim, gstr,
                        bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        promotion, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MGG_ERR_RUNTIME, std::string("cuTensorMapEncodeTiled rejected the ") + what + " map (CUresult " +
                                     std::to_string((int)r) + ")");
  return MGG_OK;
}

mgg_status encode_bf16(CUtensorMap* map, const void* addr, int rank, const uint64_t* dims, const uint64_t* strides,
                       const uint32_t* box, const char* what) {
  return encode_map(map, MGG_BF16, addr, rank, dims, strides, box, what);
}

// One NVTX range per ABI call (host side: validation, descriptor encoding and the launches), so a
// profiler timeline shows which call queued which kernels.  Costs nothing without a tool attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

// ---------------------------------------------------------------- device check
struct DevInfo {
  int num_sms;
  int device;
};

mgg_status check_device(DevInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MGG_ERR_ARCH, std::string("no CUDA device: ") + cudaGetErrorString(e));
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(MGG_ERR_ARCH, "libmgg is built for sm_103a; the current device has compute capability " +
                                  std::to_string(major) + "." + std::to_string(minor));
  info->num_sms = sms;
  info->device = dev;
  return MGG_OK;
}

bool valid_dtype(int d) { return d == MGG_BF16 || d == MGG_FP16 || d == MGG_FP32; }

// ---------------------------------------------------------------- dGLU validation
mgg_status validate_dglu(const mgg_dglu_bwd_args& a) {
  if (a.L < 1 || a.L > 1024) return fail(MGG_ERR_VALUE, "expert count L must be in [1, 1024]");
  if (a.M < 0 || a.M % 256 != 0) return fail(MGG_ERR_VALUE, "M (padded rows) must be a non-negative multiple of 256");
  if (a.M > (int64_t)1 << 30) return fail(MGG_ERR_UNSUPPORTED, "M above 2^30 rows is not supported");
  if (a.K < 8 || a.K % 8 != 0) return fail(MGG_ERR_VALUE, "K must be a positive multiple of 8 (16-byte rows)");
  if (a.K > (int64_t)1 << 24) return fail(MGG_ERR_UNSUPPORTED, "K above 2^24 is not supported");
  if (a.N < 32 || a.N % 32 != 0) return fail(MGG_ERR_VALUE, "N must be a positive multiple of 32");
  if (a.N > (int64_t)1 << 24) return fail(MGG_ERR_UNSUPPORTED, "N above 2^24 is not supported");
  if ((a.b == nullptr) == (a.b_ptrs == nullptr))
    return fail(MGG_ERR_VALUE, "exactly one of the dense weights b and the pointer array b_ptrs must be given");
  if (a.b_major != MGG_MAJOR_K && a.b_major != MGG_MAJOR_MN) return fail(MGG_ERR_VALUE, "b_major must be K or MN");
  if (a.b != nullptr && a.b_major != MGG_MAJOR_K) return fail(MGG_ERR_VALUE, "dense weights (N, K, L) are K-major");
  if (!valid_dtype(a.c_dtype) || !valid_dtype(a.d_dtype)) return fail(MGG_ERR_VALUE, "c_dtype/d_dtype out of range");
  if (a.act != MGG_ACT_DSWIGLU && a.act != MGG_ACT_DGEGLU && a.act != MGG_ACT_DSITUGLU)
    return fail(MGG_ERR_VALUE, "act must be DSWIGLU, DGEGLU or DSITUGLU");
  if (a.act == MGG_ACT_DSITUGLU) {
    const float b[2] = {a.situ_beta1, a.situ_beta2};
    for (float v : b)
      if (v != 0.0f && !(v > 0.0f && v < 3.0e38f))
        return fail(MGG_ERR_VALUE, "situ_beta1 / situ_beta2 must be positive finite (0 = default)");
  }
  if (a.geglu_filter != MGG_FILTER_VALUE && a.geglu_filter != MGG_FILTER_INDICATOR)
    return fail(MGG_ERR_VALUE, "geglu_filter must be VALUE or INDICATOR");
  if (a.gate_first != 0 && a.gate_first != 1) return fail(MGG_ERR_VALUE, "gate_first must be 0 or 1");
  if (a.sched != MGG_SCHED_STATIC && a.sched != MGG_SCHED_DYNAMIC) return fail(MGG_ERR_VALUE, "sched out of range");
  if (a.cta_mode != MGG_CTA_AUTO && a.cta_mode != MGG_CTA_SINGLE && a.cta_mode != MGG_CTA_PAIR)
    return fail(MGG_ERR_VALUE, "cta_mode out of range");
  const void* req[] = {a.a, a.c, a.padded_offsets, a.alpha, a.beta, a.prob, a.dprob, a.d_row, a.workspace};
  const char* names[] = {"a", "c", "padded_offsets", "alpha", "beta", "prob", "dprob", "d_row", "workspace"};
  const bool per_row[] = {true, true, false, false, false, true, true, true, false};
  for (int i = 0; i < 9; ++i) {
    if (req[i] == nullptr && per_row[i] && a.M == 0) continue;  // no rows: nothing is read or written there
    if (req[i] == nullptr) return fail(MGG_ERR_VALUE, std::string(names[i]) + " must not be NULL");
    if (!aligned16(req[i])) return fail(MGG_ERR_VALUE, std::string(names[i]) + " must be 16-byte aligned");
  }
  if (a.b && !aligned16(a.b)) return fail(MGG_ERR_VALUE, "b must be 16-byte aligned");
  if (a.b_ptrs && !aligned16(a.b_ptrs)) return fail(MGG_ERR_VALUE, "b_ptrs must be 16-byte aligned");
  if (a.dbias && !aligned16(a.dbias)) return fail(MGG_ERR_VALUE, "dbias must be 16-byte aligned");
  if (a.d_col && !aligned16(a.d_col)) return fail(MGG_ERR_VALUE, "d_col must be 16-byte aligned");
  if (a.amax && !aligned16(a.amax)) return fail(MGG_ERR_VALUE, "amax must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(a.workspace) & 255u) != 0)
    return fail(MGG_ERR_VALUE, "workspace must be 256-byte aligned");
  if ((size_t)a.workspace_bytes < mgg_dglu_bwd_workspace_size(a.L, a.N))
    return fail(MGG_ERR_VALUE, "workspace too small: need " + std::to_string(mgg_dglu_bwd_workspace_size(a.L, a.N)) +
                                   " bytes");
  if (a.tile_log != nullptr) {
    if (!aligned16(a.tile_log)) return fail(MGG_ERR_VALUE, "tile_log must be 16-byte aligned");
    if (a.tile_log_capacity < mgg_dglu_bwd_num_tiles(a.M, a.N))
      return fail(MGG_ERR_VALUE, "tile_log_capacity smaller than the number of tiles");
  }
  return MGG_OK;
}

// ---------------------------------------------------------------- dsReLU validation
mgg_status validate_dsrelu(const mgg_dsrelu_bwd_args& a) {
  if (a.L < 1 || a.L > 1024) return fail(MGG_ERR_VALUE, "expert count L must be in [1, 1024]");
  if (a.M < 0 || a.M % 256 != 0) return fail(MGG_ERR_VALUE, "M (padded rows) must be a non-negative multiple of 256");
  if (a.M > (int64_t)1 << 30) return fail(MGG_ERR_UNSUPPORTED, "M above 2^30 rows is not supported");
  if (a.K < 8 || a.K % 8 != 0) return fail(MGG_ERR_VALUE, "K must be a positive multiple of 8 (16-byte rows)");
  if (a.K > (int64_t)1 << 24) return fail(MGG_ERR_UNSUPPORTED, "K above 2^24 is not supported");
  if (a.N < 32 || a.N % 32 != 0) return fail(MGG_ERR_VALUE, "N must be a positive multiple of 32");
  if (a.N > (int64_t)1 << 24) return fail(MGG_ERR_UNSUPPORTED, "N above 2^24 is not supported");
  if ((a.b == nullptr) == (a.b_ptrs == nullptr))
    return fail(MGG_ERR_VALUE, "exactly one of the dense weights b and the pointer array b_ptrs must be given");
  if (a.b_major != MGG_MAJOR_K && a.b_major != MGG_MAJOR_MN) return fail(MGG_ERR_VALUE, "b_major must be K or MN");
  if (a.b != nullptr && a.b_major != MGG_MAJOR_K) return fail(MGG_ERR_VALUE, "dense weights (N, K, L) are K-major");
  if (!valid_dtype(a.c_dtype) || !valid_dtype(a.d_dtype)) return fail(MGG_ERR_VALUE, "c_dtype/d_dtype out of range");
  if (a.c_dtype == MGG_FP32) return fail(MGG_ERR_UNSUPPORTED, "the dsReLU epilogue takes a 16-bit C (bf16 or fp16)");
  if (a.sched != MGG_SCHED_STATIC && a.sched != MGG_SCHED_DYNAMIC) return fail(MGG_ERR_VALUE, "sched out of range");
  if (a.cta_mode != MGG_CTA_AUTO && a.cta_mode != MGG_CTA_SINGLE && a.cta_mode != MGG_CTA_PAIR)
    return fail(MGG_ERR_VALUE, "cta_mode out of range");
  if (a.reserved != 0) return fail(MGG_ERR_VALUE, "reserved field must be 0");
  const void* req[] = {a.a, a.c, a.padded_offsets, a.alpha, a.prob, a.dprob, a.d_row, a.workspace};
  const char* names[] = {"a", "c", "padded_offsets", "alpha", "prob", "dprob", "d_row", "workspace"};
  const bool per_row[] = {true, true, false, false, true, true, true, false};
  for (int i = 0; i < 8; ++i) {
    if (req[i] == nullptr && per_row[i] && a.M == 0) continue;  // no rows: nothing is read or written there
    if (req[i] == nullptr) return fail(MGG_ERR_VALUE, std::string(names[i]) + " must not be NULL");
    if (!aligned16(req[i])) return fail(MGG_ERR_VALUE, std::string(names[i]) + " must be 16-byte aligned");
  }
  if (a.b && !aligned16(a.b)) return fail(MGG_ERR_VALUE, "b must be 16-byte aligned");
  if (a.b_ptrs && !aligned16(a.b_ptrs)) return fail(MGG_ERR_VALUE, "b_ptrs must be 16-byte aligned");
  if (a.d_col && !aligned16(a.d_col)) return fail(MGG_ERR_VALUE, "d_col must be 16-byte aligned");
  if (a.amax && !aligned16(a.amax)) return fail(MGG_ERR_VALUE, "amax must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(a.workspace) & 255u) != 0)
    return fail(MGG_ERR_VALUE, "workspace must be 256-byte aligned");
  if ((size_t)a.workspace_bytes < mgg_dsrelu_bwd_workspace_size(a.L))
    return fail(MGG_ERR_VALUE, "workspace too small: need " + std::to_string(mgg_dsrelu_bwd_workspace_size(a.L)) +
                                   " bytes");
  if (a.tile_log != nullptr) {
    if (!aligned16(a.tile_log)) return fail(MGG_ERR_VALUE, "tile_log must be 16-byte aligned");
    if (a.tile_log_capacity < mgg_dglu_bwd_num_tiles(a.M, a.N))
      return fail(MGG_ERR_VALUE, "tile_log_capacity smaller than the number of tiles");
  }
  return MGG_OK;
}

// ---------------------------------------------------------------- wgrad validation
mgg_status validate_wgrad(const mgg_wgrad_args& a) {
  if (a.L < 1 || a.L > 1024) return fail(MGG_ERR_VALUE, "expert count L must be in [1, 1024]");
  if (a.hidden < 8 || a.hidden % 8 != 0) return fail(MGG_ERR_VALUE, "hidden must be a positive multiple of 8");
  if (a.inter < 8 || a.inter % 8 != 0) return fail(MGG_ERR_VALUE, "intermediate must be a positive multiple of 8");
  if (a.hidden > (int64_t)1 << 24 || a.inter > (int64_t)1 << 24)
    return fail(MGG_ERR_UNSUPPORTED, "hidden/intermediate above 2^24 is not supported");
  if (a.tokens_sum < 0 || a.tokens_sum % 256 != 0)
    return fail(MGG_ERR_VALUE, "tokens_sum must be a non-negative multiple of 256");
  if (a.tokens_sum > (int64_t)1 << 30) return fail(MGG_ERR_UNSUPPORTED, "tokens_sum above 2^30 is not supported");
  if ((a.out == nullptr) == (a.out_ptrs == nullptr))
    return fail(MGG_ERR_VALUE, "exactly one of the dense output and the pointer array out_ptrs must be given");
  if (a.a_major != MGG_MAJOR_K && a.a_major != MGG_MAJOR_MN) return fail(MGG_ERR_VALUE, "a_major must be K or MN");
  if (a.b_major != MGG_MAJOR_K && a.b_major != MGG_MAJOR_MN) return fail(MGG_ERR_VALUE, "b_major must be K or MN");
  if (a.input_order != MGG_ORDER_TENSOR2D && a.input_order != MGG_ORDER_TENSOR_RAGGED)
    return fail(MGG_ERR_VALUE, "input_order out of range");
  if (!valid_dtype(a.out_dtype)) return fail(MGG_ERR_VALUE, "out_dtype out of range");
  if (a.accumulate != 0 && a.accumulate != 1) return fail(MGG_ERR_VALUE, "accumulate must be 0 or 1");
  if (a.sched != MGG_SCHED_STATIC && a.sched != MGG_SCHED_DYNAMIC) return fail(MGG_ERR_VALUE, "sched out of range");
  if (a.cta_mode != MGG_CTA_AUTO && a.cta_mode != MGG_CTA_SINGLE && a.cta_mode != MGG_CTA_PAIR)
    return fail(MGG_ERR_VALUE, "cta_mode out of range");
  if (a.cta_mode == MGG_CTA_PAIR && a.hidden % 256 != 0)
    return fail(MGG_ERR_VALUE, "cta_mode PAIR needs hidden to be a multiple of 256");
  if (a.reserved1 != 0) return fail(MGG_ERR_VALUE, "reserved field must be 0");
  const void* req[] = {a.a, a.b, a.offsets, a.workspace};
  const char* names[] = {"a", "b", "offsets", "workspace"};
  for (int i = 0; i < 4; ++i) {
    if (req[i] == nullptr && i < 2 && a.tokens_sum == 0) continue;  // no tokens: the operands are never read
    if (req[i] == nullptr) return fail(MGG_ERR_VALUE, std::string(names[i]) + " must not be NULL");
    if (!aligned16(req[i])) return fail(MGG_ERR_VALUE, std::string(names[i]) + " must be 16-byte aligned");
  }
  if (a.out && !aligned16(a.out)) return fail(MGG_ERR_VALUE, "out must be 16-byte aligned");
  if (a.out_ptrs && !aligned16(a.out_ptrs)) return fail(MGG_ERR_VALUE, "out_ptrs must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(a.workspace) & 255u) != 0)
    return fail(MGG_ERR_VALUE, "workspace must be 256-byte aligned");
  if ((size_t)a.workspace_bytes < mgg_wgrad_workspace_size(a.L))
    return fail(MGG_ERR_VALUE, "workspace too small: need " + std::to_string(mgg_wgrad_workspace_size(a.L)) + " bytes");
  if (a.tile_log != nullptr) {
    if (!aligned16(a.tile_log)) return fail(MGG_ERR_VALUE, "tile_log must be 16-byte aligned");
    if (a.tile_log_capacity < mgg_wgrad_num_tiles(a.L, a.hidden, a.inter))
      return fail(MGG_ERR_VALUE, "tile_log_capacity smaller than the number of tiles");
  }
  return MGG_OK;
}

// AUTO picks CTA pairs where they measured faster on GB300.  For the dgrad that is every shape
// (M is a multiple of 256): a pair's halved B slot leaves room for eight epilogue warps with the
// C ring and five operand stages (Mixtral-shaped: 1552 vs 1397 TFLOP/s single; DeepSeek-shaped
// K = 7168: 1486 vs 1300; dGeGLU with fp32 D: 975 vs 845).
bool dglu_pair(const mgg_dglu_bwd_args& a) { return a.cta_mode != MGG_CTA_SINGLE; }

// For the wgrad AUTO takes pairs whenever hidden allows them (a multiple of 256): a pair loads
// 32 KB of operands per SM and k-slice instead of 48 KB, and the SM's operand loads, not the tensor
// pipe, bound these layers (DeepSeek-shaped, ~630 tokens per expert: 3.79 vs 4.17 ms on one box;
// Zipf-shaped dense accumulate, ~1000 tokens per expert: 0.312 vs 0.343 ms).
bool wgrad_pair(const mgg_wgrad_args& a) {
  if (a.hidden % 256 != 0) return false;
  if (a.cta_mode != MGG_CTA_AUTO) return a.cta_mode == MGG_CTA_PAIR;
  return true;
}

mgg_status from_cuda(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return MGG_OK;
  return fail(MGG_ERR_RUNTIME, std::string(what) + ": " + cudaGetErrorString(e));
}

}  // namespace

void set_last_error(const std::string& msg) { g_err = msg; }

}  // namespace mgg

using namespace mgg;

extern "C" {

int mgg_abi_version(void) { return MGG_ABI_VERSION; }

size_t mgg_sizeof_dglu_bwd_args(void) { return sizeof(mgg_dglu_bwd_args); }

size_t mgg_sizeof_dsrelu_bwd_args(void) { return sizeof(mgg_dsrelu_bwd_args); }

size_t mgg_sizeof_wgrad_args(void) { return sizeof(mgg_wgrad_args); }

int mgg_args_field_offsets(int which, size_t* out, int cap) {
#define MGG_OFF(S, f) offsetof(S, f)
  static const size_t dglu[] = {
      MGG_OFF(mgg_dglu_bwd_args, M), MGG_OFF(mgg_dglu_bwd_args, K), MGG_OFF(mgg_dglu_bwd_args, N),
      MGG_OFF(mgg_dglu_bwd_args, L), MGG_OFF(mgg_dglu_bwd_args, a), MGG_OFF(mgg_dglu_bwd_args, b),
      MGG_OFF(mgg_dglu_bwd_args, b_ptrs), MGG_OFF(mgg_dglu_bwd_args, c), MGG_OFF(mgg_dglu_bwd_args, padded_offsets),
      MGG_OFF(mgg_dglu_bwd_args, alpha), MGG_OFF(mgg_dglu_bwd_args, beta), MGG_OFF(mgg_dglu_bwd_args, prob),
      MGG_OFF(mgg_dglu_bwd_args, dprob), MGG_OFF(mgg_dglu_bwd_args, d_row), MGG_OFF(mgg_dglu_bwd_args, dbias),
      MGG_OFF(mgg_dglu_bwd_args, d_col), MGG_OFF(mgg_dglu_bwd_args, amax), MGG_OFF(mgg_dglu_bwd_args, workspace),
      MGG_OFF(mgg_dglu_bwd_args, tile_log), MGG_OFF(mgg_dglu_bwd_args, workspace_bytes),
      MGG_OFF(mgg_dglu_bwd_args, tile_log_capacity), MGG_OFF(mgg_dglu_bwd_args, b_major),
      MGG_OFF(mgg_dglu_bwd_args, c_dtype), MGG_OFF(mgg_dglu_bwd_args, d_dtype), MGG_OFF(mgg_dglu_bwd_args, act),
      MGG_OFF(mgg_dglu_bwd_args, geglu_filter), MGG_OFF(mgg_dglu_bwd_args, gate_first),
      MGG_OFF(mgg_dglu_bwd_args, sched), MGG_OFF(mgg_dglu_bwd_args, cta_mode), MGG_OFF(mgg_dglu_bwd_args, situ_beta1),
      MGG_OFF(mgg_dglu_bwd_args, situ_beta2)};
  static const size_t dsrelu[] = {
      MGG_OFF(mgg_dsrelu_bwd_args, M), MGG_OFF(mgg_dsrelu_bwd_args, K), MGG_OFF(mgg_dsrelu_bwd_args, N),
      MGG_OFF(mgg_dsrelu_bwd_args, L), MGG_OFF(mgg_dsrelu_bwd_args, a), MGG_OFF(mgg_dsrelu_bwd_args, b),
      MGG_OFF(mgg_dsrelu_bwd_args, b_ptrs), MGG_OFF(mgg_dsrelu_bwd_args, c),
      MGG_OFF(mgg_dsrelu_bwd_args, padded_offsets), MGG_OFF(mgg_dsrelu_bwd_args, alpha),
      MGG_OFF(mgg_dsrelu_bwd_args, prob), MGG_OFF(mgg_dsrelu_bwd_args, dprob), MGG_OFF(mgg_dsrelu_bwd_args, d_row),
      MGG_OFF(mgg_dsrelu_bwd_args, d_col), MGG_OFF(mgg_dsrelu_bwd_args, amax), MGG_OFF(mgg_dsrelu_bwd_args, workspace),
      MGG_OFF(mgg_dsrelu_bwd_args, tile_log), MGG_OFF(mgg_dsrelu_bwd_args, workspace_bytes),
      MGG_OFF(mgg_dsrelu_bwd_args, tile_log_capacity), MGG_OFF(mgg_dsrelu_bwd_args, b_major),
      MGG_OFF(mgg_dsrelu_bwd_args, c_dtype), MGG_OFF(mgg_dsrelu_bwd_args, d_dtype),
      MGG_OFF(mgg_dsrelu_bwd_args, sched), MGG_OFF(mgg_dsrelu_bwd_args, cta_mode),
      MGG_OFF(mgg_dsrelu_bwd_args, reserved)};
  static const size_t wgrad[] = {
      MGG_OFF(mgg_wgrad_args, hidden), MGG_OFF(mgg_wgrad_args, inter), MGG_OFF(mgg_wgrad_args, L),
      MGG_OFF(mgg_wgrad_args, tokens_sum), MGG_OFF(mgg_wgrad_args, a), MGG_OFF(mgg_wgrad_args, b),
      MGG_OFF(mgg_wgrad_args, offsets), MGG_OFF(mgg_wgrad_args, out), MGG_OFF(mgg_wgrad_args, out_ptrs),
      MGG_OFF(mgg_wgrad_args, workspace), MGG_OFF(mgg_wgrad_args, tile_log), MGG_OFF(mgg_wgrad_args, workspace_bytes),
      MGG_OFF(mgg_wgrad_args, tile_log_capacity), MGG_OFF(mgg_wgrad_args, a_major), MGG_OFF(mgg_wgrad_args, b_major),
      MGG_OFF(mgg_wgrad_args, input_order), MGG_OFF(mgg_wgrad_args, out_dtype), MGG_OFF(mgg_wgrad_args, accumulate),
      MGG_OFF(mgg_wgrad_args, sched), MGG_OFF(mgg_wgrad_args, cta_mode), MGG_OFF(mgg_wgrad_args, reserved1)};
#undef MGG_OFF
  const size_t* tab = which == 0 ? dglu : which == 1 ? dsrelu : which == 2 ? wgrad : nullptr;
  const int n = which == 0 ? (int)(sizeof(dglu) / sizeof(size_t))
              : which == 1 ? (int)(sizeof(dsrelu) / sizeof(size_t))
              : which == 2 ? (int)(sizeof(wgrad) / sizeof(size_t)) : -1;
  if (tab == nullptr) return -1;
  for (int i = 0; i < n && i < cap && out != nullptr; ++i) out[i] = tab[i];
  return n;
}

const char* mgg_last_error(void) { return g_err.c_str(); }

const char* mgg_status_string(int s) {
  switch (s) {
    case MGG_OK: return "MGG_OK";
    case MGG_ERR_VALUE: return "MGG_ERR_VALUE";
    case MGG_ERR_UNSUPPORTED: return "MGG_ERR_UNSUPPORTED";
    case MGG_ERR_RUNTIME: return "MGG_ERR_RUNTIME";
    case MGG_ERR_ARCH: return "MGG_ERR_ARCH";
    case MGG_ERR_DEVICE_OFFSETS: return "MGG_ERR_DEVICE_OFFSETS";
    case MGG_ERR_DEVICE_POINTER: return "MGG_ERR_DEVICE_POINTER";
    case MGG_ERR_DEVICE_TIMEOUT: return "MGG_ERR_DEVICE_TIMEOUT";
    case MGG_ERR_DEVICE_BOUNDS: return "MGG_ERR_DEVICE_BOUNDS";
    default: return "MGG_UNKNOWN_STATUS";
  }
}

size_t mgg_dglu_bwd_workspace_size(int64_t L, int64_t N) {
  if (L < 0 || N < 0) return 0;
  return round_up(kWsHeaderBytes + kTmapBytes * (size_t)L + sizeof(float) * (size_t)L * 2 * (size_t)N, 256);
}

size_t mgg_dsrelu_bwd_workspace_size(int64_t L) {
  if (L < 0) return 0;
  return round_up(kWsHeaderBytes + kTmapBytes * (size_t)L, 256);
}

size_t mgg_wgrad_workspace_size(int64_t L) {
  if (L < 0) return 0;
  return wgrad_workspace_bytes((size_t)L);
}

int64_t mgg_dglu_bwd_num_tiles(int64_t M, int64_t N) {
  if (M < 0 || N < 0) return 0;
  return (M / 128) * ((N + kDgluTileN - 1) / kDgluTileN);
}

int64_t mgg_wgrad_num_tiles(int64_t L, int64_t hidden, int64_t inter) {
  if (L < 0 || hidden < 0 || inter < 0) return 0;
  const int64_t bn = wgrad_tile_n(inter);
  return L * ((hidden + 127) / 128) * ((inter + bn - 1) / bn);
}

void mgg_dglu_bwd_tile_shape(int32_t* tile_m, int32_t* tile_n) {
  if (tile_m) *tile_m = 128;
  if (tile_n) *tile_n = kDgluTileN;
}

void mgg_wgrad_tile_shape(int64_t inter, int32_t* tile_m, int32_t* tile_n) {
  if (tile_m) *tile_m = 128;
  if (tile_n) *tile_n = wgrad_tile_n(inter);
}

}  // extern "C"

namespace mgg {
namespace {

// Maps of one grouped-GEMM epilogue call: A (M, K); B (N, K) per expert (dense, or the
// discrete template); C and D_row / D_col of `cd_cols` columns (2N for dGLU, N for dsReLU).
mgg_status build_epi_maps(DgluLaunch& Lc, const void* a_ptr, const void* b, const int64_t* b_ptrs, int b_major,
                          const void* c, int c_dtype, void* d_row, void* d_col, int d_dtype, int64_t M_, int64_t K_,
                          int64_t N_, int64_t L_, uint64_t cd_cols) {
  mgg_status s;
  const uint32_t b_rows = (uint32_t)(Lc.pair ? kDgluTileN / 2 : kDgluTileN);  // B rows one CTA loads
  const uint64_t M = (uint64_t)(M_ > 0 ? M_ : 256), K = (uint64_t)K_, N = (uint64_t)N_, L = (uint64_t)L_;
  {
    const uint64_t dims[2] = {K, M}, strides[1] = {K * 2};
    const uint32_t box[2] = {64, 128};
    if ((s = encode_bf16(&Lc.tmap_a, a_ptr, 2, dims, strides, box, "A")) != MGG_OK) return s;
  }
  if (b != nullptr) {
    const uint64_t dims[3] = {K, N, L}, strides[2] = {K * 2, N * K * 2};
    const uint32_t box[3] = {64, b_rows, 1};
    if ((s = encode_bf16(&Lc.tmap_b, b, 3, dims, strides, box, "dense B")) != MGG_OK) return s;
  } else if (b_major == MGG_MAJOR_K) {
    const uint64_t dims[2] = {K, N}, strides[1] = {K * 2};
    const uint32_t box[2] = {64, b_rows};
    if ((s = encode_bf16(&Lc.tmap_b, a_ptr, 2, dims, strides, box, "discrete K-major B")) != MGG_OK) return s;
  } else {
    // N a multiple of 64: a 3-D template of 64-column blocks (dims {64, K, N/64}, strides
    // {N*2, 128} bytes) so one box fills a ring slot; else one 64 x 64 box per 64 columns
    (void)b_ptrs;
    if (N % 64 == 0) {
      const uint64_t dims[3] = {64, K, N / 64}, strides[2] = {N * 2, 128};
      const uint32_t box[3] = {64, 64, b_rows / 64};
      const std::string saved = g_err;
      Lc.b_blocked = encode_bf16(&Lc.tmap_b, a_ptr, 3, dims, strides, box, "discrete N-major B (blocked)") == MGG_OK;
      if (!Lc.b_blocked) g_err = saved;
    }
    if (!Lc.b_blocked) {
      const uint64_t dims[2] = {N, K}, strides[1] = {N * 2};
      const uint32_t box[2] = {64, 64};
      if ((s = encode_bf16(&Lc.tmap_b, a_ptr, 2, dims, strides, box, "discrete N-major B")) != MGG_OK) return s;
    }
  }
  {  // D_row / D_col (M, cd_cols): 32-row boxes of one 128-byte row of columns
    const uint64_t esz = d_dtype == MGG_FP32 ? 4 : 2;
    const uint64_t dims[2] = {cd_cols, M}, strides[1] = {cd_cols * esz};
    const uint32_t box[2] = {(uint32_t)(128 / esz), 32};
    if ((s = encode_map(&Lc.tmap_d, d_dtype, d_row, 2, dims, strides, box, "D_row")) != MGG_OK) return s;
    if (d_col != nullptr && (s = encode_map(&Lc.tmap_dcol, d_dtype, d_col, 2, dims, strides, box, "D_col")) != MGG_OK)
      return s;
  }
  if (c_dtype != MGG_FP32) {  // C (M, cd_cols): 32-row boxes of 64 columns
    const uint64_t dims[2] = {cd_cols, M}, strides[1] = {cd_cols * 2};
    const uint32_t box[2] = {64, 32};
    // 128-byte promotion: C is read once, 128 bytes per row and box, and the row's next 128 bytes
    // belong to a later use or another warp; fetched early (256-byte promotion) under the loads'
    // evict-first hint they were often dropped again before that use (Mixtral-shaped layer: DRAM
    // reads 3.75 -> 3.43 GB, 2.224 -> 2.210 ms)
    if ((s = encode_map(&Lc.tmap_c, c_dtype, c, 2, dims, strides, box, "C", CU_TENSOR_MAP_L2_PROMOTION_L2_128B)) !=
        MGG_OK)
      return s;
  }
  return MGG_OK;
}

}  // namespace
}  // namespace mgg

extern "C" {

mgg_status mgg_dglu_bwd(const mgg_dglu_bwd_args* args, void* stream) {
  g_err.clear();
  const NvtxRange range("mgg_dglu_bwd");
  if (args == nullptr) return fail(MGG_ERR_VALUE, "args is NULL");
  const mgg_dglu_bwd_args& a = *args;
  mgg_status s = validate_dglu(a);
  if (s != MGG_OK) return s;
  DevInfo dev;
  if ((s = check_device(&dev)) != MGG_OK) return s;

  DgluLaunch Lc;
  memset(&Lc, 0, sizeof(Lc));
  Lc.args = args;
  Lc.num_sms = dev.num_sms;
  Lc.device = dev.device;
  Lc.tile_n = kDgluTileN;
  Lc.pair = dglu_pair(a);
  // with no rows (M == 0) the per-row operands may be NULL: their maps, never used, point at the workspace
  if ((s = build_epi_maps(Lc, or_ws(a.a, a.workspace), a.b, a.b_ptrs, a.b_major, or_ws(a.c, a.workspace), a.c_dtype,
                          or_ws(a.d_row, a.workspace), a.d_col, a.d_dtype, a.M, a.K, a.N, a.L,
                          2 * (uint64_t)a.N)) != MGG_OK)
    return s;
  return from_cuda(launch_dglu_bwd(Lc, static_cast<cudaStream_t>(stream)), "mgg_dglu_bwd launch");
}

mgg_status mgg_dsrelu_bwd(const mgg_dsrelu_bwd_args* args, void* stream) {
  g_err.clear();
  const NvtxRange range("mgg_dsrelu_bwd");
  if (args == nullptr) return fail(MGG_ERR_VALUE, "args is NULL");
  const mgg_dsrelu_bwd_args& a = *args;
  mgg_status s = validate_dsrelu(a);
  if (s != MGG_OK) return s;
  DevInfo dev;
  if ((s = check_device(&dev)) != MGG_OK) return s;

  DgluLaunch Lc;
  memset(&Lc, 0, sizeof(Lc));
  Lc.args = nullptr;
  Lc.num_sms = dev.num_sms;
  Lc.device = dev.device;
  Lc.tile_n = kDgluTileN;
  Lc.pair = a.cta_mode != MGG_CTA_SINGLE;  // AUTO: pairs, as for the dGLU dgrad
  if ((s = build_epi_maps(Lc, or_ws(a.a, a.workspace), a.b, a.b_ptrs, a.b_major, or_ws(a.c, a.workspace), a.c_dtype,
                          or_ws(a.d_row, a.workspace), a.d_col, a.d_dtype, a.M, a.K, a.N, a.L,
                          (uint64_t)a.N)) != MGG_OK)
    return s;
  return from_cuda(launch_dsrelu_bwd(Lc, a, static_cast<cudaStream_t>(stream)), "mgg_dsrelu_bwd launch");
}

mgg_status mgg_wgrad(const mgg_wgrad_args* args, void* stream) {
  g_err.clear();
  const NvtxRange range("mgg_wgrad");
  if (args == nullptr) return fail(MGG_ERR_VALUE, "args is NULL");
  const mgg_wgrad_args& a = *args;
  mgg_status s = validate_wgrad(a);
  if (s != MGG_OK) return s;
  DevInfo dev;
  if ((s = check_device(&dev)) != MGG_OK) return s;

  WgradLaunch Lc;
  memset(&Lc, 0, sizeof(Lc));
  Lc.args = args;
  Lc.num_sms = dev.num_sms;
  Lc.device = dev.device;
  Lc.tile_n = wgrad_tile_n(a.inter);
  Lc.pair = wgrad_pair(a);
  const bool ragged = a.input_order == MGG_ORDER_TENSOR_RAGGED;
  Lc.a_ragged = ragged && a.a_major == MGG_MAJOR_K;
  Lc.b_ragged = ragged && a.b_major == MGG_MAJOR_K;
  const uint64_t T = (uint64_t)(a.tokens_sum > 0 ? a.tokens_sum : 256), H = (uint64_t)a.hidden, I = (uint64_t)a.inter;
  // with no tokens the operands may be NULL: their maps, never used, point at the workspace
  const void* A = or_ws(a.a, a.workspace);
  const void* B = or_ws(a.b, a.workspace);
  // An MN-major operand whose MN extent is a multiple of 64 is also a 3-D tensor of 64-wide
  // blocks: dims {64, T, extent/64}, strides {extent*2, 128} bytes.  One box of that map fills a
  // whole ring slot (its 64 x 64 blocks land 8 KB apart, as the MMA descriptors expect), so the
  // producer issues one TMA copy per operand and slot instead of one per 64 columns.
  auto blocked = [&](CUtensorMap* map, const void* base, uint64_t extent, uint32_t blocks, const char* what) {
    if (extent % 64 != 0) return false;
    const uint64_t dims[3] = {64, T, extent / 64}, strides[2] = {extent * 2, 128};
    const uint32_t box[3] = {64, 64, blocks};
    const std::string saved = g_err;
    if (encode_bf16(map, base, 3, dims, strides, box, what) == MGG_OK) return true;
    g_err = saved;  // the driver refused the blocked view: the 2-D map is used instead
    return false;
  };
  const uint32_t b_cols = (uint32_t)(Lc.pair ? Lc.tile_n / 2 : Lc.tile_n);  // B columns one CTA loads
  if (a.a_major == MGG_MAJOR_K) {  // (hidden, T), T contiguous
    const uint64_t dims[2] = {T, H}, strides[1] = {T * 2};
    const uint32_t box[2] = {64, 128};
    if ((s = encode_bf16(&Lc.tmap_a, A, 2, dims, strides, box, "A (K-major)")) != MGG_OK) return s;
  } else if (!(Lc.a_blocked = blocked(&Lc.tmap_a, A, H, 2, "A (M-major, blocked)"))) {
    // (hidden, T) with hidden contiguous: rows of T
    const uint64_t dims[2] = {H, T}, strides[1] = {H * 2};
    const uint32_t box[2] = {64, 64};
    if ((s = encode_bf16(&Lc.tmap_a, A, 2, dims, strides, box, "A (M-major)")) != MGG_OK) return s;
  }
  if (a.b_major == MGG_MAJOR_MN) {  // (T, inter), inter contiguous
    if (!(Lc.b_blocked = blocked(&Lc.tmap_b, B, I, b_cols / 64, "B (N-major, blocked)"))) {
      const uint64_t dims[2] = {I, T}, strides[1] = {I * 2};
      const uint32_t box[2] = {64, 64};
      if ((s = encode_bf16(&Lc.tmap_b, B, 2, dims, strides, box, "B (N-major)")) != MGG_OK) return s;
    }
  } else {  // (T, inter) with T contiguous: rows of T
    const uint64_t dims[2] = {T, I}, strides[1] = {T * 2};
    const uint32_t box[2] = {64, b_cols};
    if ((s = encode_bf16(&Lc.tmap_b, B, 2, dims, strides, box, "B (K-major)")) != MGG_OK) return s;
  }
  {  // outputs: 32-row boxes of one 128-byte row of columns
    const uint64_t esz = a.out_dtype == MGG_FP32 ? 4 : 2, L = (uint64_t)a.L;
    const uint32_t cw = (uint32_t)(128 / esz);
    // FP32 outputs with inter % 64 == 0 are also viewed as 32-column blocks (dims {32, hidden,
    // inter/32 [, L]}, strides {inter*4, 128 [, hidden*inter*4]} bytes): one box of two blocks
    // stores the two 32-column chunks of one 64-column TMEM load (8 KB) with a single TMA copy.
    if (a.out_dtype == MGG_FP32 && I % 64 == 0) {
      const std::string saved = g_err;
      if (a.out != nullptr) {
        const uint64_t dims[4] = {32, H, I / 32, L}, strides[3] = {I * 4, 128, H * I * 4};
        const uint32_t box[4] = {32, 32, 2, 1};
        Lc.out_blocked = encode_map(&Lc.tmap_out, a.out_dtype, a.out, 4, dims, strides, box, "dense output (blocked)") == MGG_OK;
      } else {
        const uint64_t dims[3] = {32, H, I / 32}, strides[2] = {I * 4, 128};
        const uint32_t box[3] = {32, 32, 2};
        Lc.out_blocked = encode_map(&Lc.tmap_out, a.out_dtype, A, 3, dims, strides, box, "per-expert output (blocked)") == MGG_OK;
      }
      if (!Lc.out_blocked) g_err = saved;  // the driver refused the blocked view: the plain map is used
    }
    if (!Lc.out_blocked && a.out != nullptr) {
      const uint64_t dims[3] = {I, H, L}, strides[2] = {I * esz, H * I * esz};
      const uint32_t box[3] = {cw, 32, 1};
      if ((s = encode_map(&Lc.tmap_out, a.out_dtype, a.out, 3, dims, strides, box, "dense output")) != MGG_OK)
        return s;
    } else if (!Lc.out_blocked) {  // per-expert template; the preparation kernel substitutes each expert's address
      const uint64_t dims[2] = {I, H}, strides[1] = {I * esz};
      const uint32_t box[2] = {cw, 32};
      if ((s = encode_map(&Lc.tmap_out, a.out_dtype, A, 2, dims, strides, box, "per-expert output")) != MGG_OK)
        return s;
    }
  }
  return from_cuda(launch_wgrad(Lc, static_cast<cudaStream_t>(stream)), "mgg_wgrad launch");
}

mgg_status mgg_read_device_status(const void* workspace, void* stream) {
  g_err.clear();
  if (workspace == nullptr) return fail(MGG_ERR_VALUE, "workspace is NULL");
  int h[4] = {0, 0, 0, 0};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(h, workspace, sizeof(h), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return from_cuda(e, "reading the device status");
  if (h[0] != 0) {
    g_err = std::string(mgg_status_string(h[0])) + " (where=" + std::to_string(h[1]) +
            ", detail=" + std::to_string(h[2]) + ")";
  }
  return static_cast<mgg_status>(h[0]);
}

mgg_status mgg_test_encode_tmap_2d(void* out128, const void* addr, uint64_t dim0, uint64_t dim1,
                                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1) {
  g_err.clear();
  if (out128 == nullptr || (reinterpret_cast<uintptr_t>(out128) & 63u) != 0)
    return fail(MGG_ERR_VALUE, "out128 must be 64-byte aligned host memory");
  const uint64_t dims[2] = {dim0, dim1}, strides[1] = {stride1_bytes};
  const uint32_t box[2] = {box0, box1};
  return encode_bf16(static_cast<CUtensorMap*>(out128), addr, 2, dims, strides, box, "test");
}

mgg_status mgg_test_tmap_replace(const void* tmpl128, void* out_dev128, const void* addr, uint32_t dim0,
                                 uint64_t stride1_bytes, int fields, void* stream) {
  g_err.clear();
  if (tmpl128 == nullptr || out_dev128 == nullptr) return fail(MGG_ERR_VALUE, "NULL descriptor");
  if ((reinterpret_cast<uintptr_t>(out_dev128) & 127u) != 0)
    return fail(MGG_ERR_VALUE, "out_dev128 must be 128-byte aligned");
  CUtensorMap t;
  memcpy(&t, tmpl128, sizeof(t));
  return from_cuda(launch_tmap_replace_probe(t, out_dev128, addr, dim0, stride1_bytes, fields,
                                             static_cast<cudaStream_t>(stream)),
                   "tensormap replace probe");
}

}  // extern "C"
