// Host-side declarations shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "mgg.h"

namespace mgg {

// Workspace header (first 256 bytes of every workspace):
//   int32 [0] status (0 = ok, else an mgg_status), [1] where, [2] detail,
//   [3] dynamic tile counter, [4] number of active experts (wgrad)
constexpr size_t kWsHeaderBytes = 256;
constexpr size_t kTmapBytes = 128;

// Workspace bytes of one mgg_wgrad call with L experts: the header, three tensor maps per expert
// (ragged A, ragged B, discrete output) and the expert order (int32 per expert), rounded to 256.
constexpr size_t wgrad_workspace_bytes(size_t L) {
  return (kWsHeaderBytes + 3 * kTmapBytes * L + sizeof(int32_t) * L + 255) / 256 * 256;
}

struct DgluLaunch {
  CUtensorMap tmap_a;
  CUtensorMap tmap_b;  // dense 3-D map, or the per-expert template (discrete)
  CUtensorMap tmap_d;  // D_row store map
  CUtensorMap tmap_c;  // C load map (16-bit C only)
  CUtensorMap tmap_dcol;  // D_col store map (when requested)
  const mgg_dglu_bwd_args* args;  // null for mgg_dsrelu_bwd
  int num_sms;
  int device;      // ordinal of the current device (keys the per-device occupancy caches)
  int tile_n;
  bool pair;       // 256-row tiles on CTA pairs (B maps load half a tile's columns)
  bool b_blocked;  // discrete N-major B as a 3-D map of 64-column blocks (one box per slot)
};

struct WgradLaunch {
  CUtensorMap tmap_a;  // tensor2d map, or the per-expert template (ragged K-major)
  CUtensorMap tmap_b;
  CUtensorMap tmap_out;  // dense output (3-D) map, or the per-expert template (discrete)
  const mgg_wgrad_args* args;
  int num_sms;
  int device;      // ordinal of the current device
  int tile_n;
  bool a_ragged;  // per-expert A maps built on the device
  bool b_ragged;
  bool pair;      // 256-row tiles on CTA pairs (B maps load half a tile's columns)
  bool a_blocked; // M-major A as a 3-D map of 64-row blocks (one box per slot), else 2-D
  bool b_blocked; // N-major B likewise
  bool out_blocked; // FP32 output as 32-column blocks (one TMA copy per two chunks), else plain
};

// Launchers (queue the prep kernel, the persistent kernel and finalisers on `stream`).
cudaError_t launch_dglu_bwd(const DgluLaunch& L, cudaStream_t stream);
cudaError_t launch_dsrelu_bwd(const DgluLaunch& L, const mgg_dsrelu_bwd_args& a, cudaStream_t stream);
cudaError_t launch_wgrad(const WgradLaunch& L, cudaStream_t stream);

// Test hook: copies `tmpl` into `out` on the device and replaces address / dim0 / stride of
// dimension 1 there with tensormap.replace (the same code path the prep kernels use).
cudaError_t launch_tmap_replace_probe(const CUtensorMap& tmpl, void* out, const void* addr, uint32_t dim0,
                                      uint64_t stride1, int fields, cudaStream_t stream);

// Sets the calling thread's mgg_last_error() message.
void set_last_error(const std::string& msg);

constexpr int kDgluTileN = 256;
// Largest K for which a single CTA stages 16-bit C through a TMA ring (one operand stage less).
constexpr int64_t kTmaCMaxK = 4095;
int wgrad_tile_n(int64_t inter);

}  // namespace mgg
