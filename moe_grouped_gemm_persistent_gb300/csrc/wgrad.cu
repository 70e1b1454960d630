// Grouped weight gradient ("Grouped GEMM + WGrad (Unified)", "Operation"):
//
//   Wgrad[e] = A[:, begin:end] @ B[begin:end, :]    begin = offsets[e-1] (0 for e = 0), end = offsets[e]
//
// with A (hidden, T) and B (T, inter) in bf16, fp32 accumulation in TMEM, and the result
// written (overwrite; zeros for an empty expert) or added (accumulate_on_output) to a
// dense (L, hidden, inter) tensor or to per-expert output pointers.
//
// Scheduling: the preparation kernel orders experts by decreasing token count; the
// persistent CTAs walk the (expert, hidden tile, inter tile) space in that order
// (longest-processing-time-first), the dynamic schedule drawing from both of its ends.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mgg_internal.h"
#include "mgg_pipeline.cuh"

namespace mgg {

// Workspace status word holding the number of experts whose tiles have work (prep kernel).
constexpr int kWgradActiveWord = 4;

struct WgradParams {
  CUtensorMap tmap_a;          // tensor2d A: K-major dims {T, h} box {64, 128}; M-major dims {h, T} box {64, 64}
  CUtensorMap tmap_b;          // tensor2d B: N-major dims {i, T} box {64, 64}; K-major dims {T, i} box {64, BN}
  CUtensorMap tmap_out;        // dense output: dims {i, h, L}, box {128 B of columns, 32, 1}, 128B swizzle;
                               // blocked FP32: dims {32, h, i/32, L}, box {32, 32, 2, 1}
  const CUtensorMap* a_maps;   // tensor_ragged K-major A: per-expert maps (dims {K_e, h}), else null
  const CUtensorMap* b_maps;   // tensor_ragged K-major B: per-expert maps (dims {K_e, i}), else null
  const CUtensorMap* out_maps; // discrete outputs: per-expert maps (dims {i, h}), else null
  const int32_t* offsets;
  const int32_t* order;        // experts by decreasing token count (workspace)
  const int64_t* out_ptrs;
  const void* out;
  int* status;
  int32_t* tile_log;
  long long tile_log_cap;
  long long total_tiles;
  int dynamic;                  // 1: tiles claimed from the workspace counter
  int hidden, inter, L;
  int tiles_n, tiles_per_expert;
  int a_mn, b_mn, out_dtype, accumulate;
  int a_blocked, b_blocked;     // MN-major operand as a 3-D map of 64-wide blocks (one box per slot)
  int out_blocked;              // FP32 output map of 32-column blocks: one store per 64-column load
};

constexpr int kWgradEpiWarps = 4;
constexpr int kWgradStgBytes = 8192;  // 4 KB staging boxes per epilogue warp (a ring of two)

__device__ __forceinline__ uint32_t swz128w(int r, int c16) { return (uint32_t)(r * 128 + ((c16 ^ (r & 7)) << 4)); }

// OS: output element size in bytes (2 = bf16/fp16, 4 = fp32).  PAIR: 256-row tiles computed by a
// CTA pair (hidden is then a multiple of 256), each CTA loading half of the tile's B columns.
// Four epilogue warps, one per TMEM sub-partition, each draining every column of its 32 rows.
// (Eight warps, two per sub-partition, each reading half of the columns into registers and freeing
// the accumulator before its stores, measured 5% slower on the DeepSeek-shaped layer: the larger
// staging costs a pair one of its six operand stages.)
template <int BN, int OS, bool PAIR>
struct WgradPolicy {
  static constexpr int kTileM = PAIR ? 2 * BM : BM;
  static constexpr int kBLoad = PAIR ? BN / 2 : BN;
  static constexpr int EPI_WARPS = kWgradEpiWarps;
  static constexpr int STG_BYTES = kWgradStgBytes;
  static constexpr int CW = 128 / OS;  // output columns per staged chunk (one 128-byte row)
  const WgradParams& p;
  static constexpr int kBoxes = STG_BYTES / 4096;
  mutable uint32_t stg_uses = 0;  // staging boxes this warp has filled (box = stg_uses % kBoxes)
  long long total_tiles;
  int* status;
  int a_mn, b_mn;
  int dynamic;
  // The scheduler thread's decode cache: the expert slot last decoded at each end of the LPT order
  // (the dynamic schedule draws from both ends, the static one uses end 0) with its
  // expert and token range, so consecutive tiles of one expert read no global memory.
  struct ExpertRange {
    int slot = -1, e = 0, begin = 0, end = 0;
  };
  mutable ExpertRange c_long, c_short;

  // Expert slot `slot` of the order with its token range, from the cache `c` or global memory.
  __device__ __forceinline__ void decode(ExpertRange& c, int slot, bool slot_ok) const {
    if (slot == c.slot) return;
    const int e = slot_ok ? __ldg(p.order + slot) : 0;
    c.slot = slot;
    c.e = e;
    c.begin = (e > 0 && e < p.L) ? __ldg(p.offsets + e - 1) : 0;
    c.end = (e >= 0 && e < p.L) ? __ldg(p.offsets + e) : 0;
  }

  __device__ WgradPolicy(const WgradParams& prm)
      : p(prm), total_tiles(prm.total_tiles), status(prm.status), a_mn(prm.a_mn), b_mn(prm.b_mn),
        dynamic(prm.dynamic) {}

  // The tiles of the experts that have work (all of them when overwriting; in accumulate mode the
  // preparation kernel counts the non-empty ones, which the LPT order puts first), so the two ends
  // of the dynamic schedule are a long and a short tile with work rather than skipped ones.
  __device__ void on_prep_done() {
    total_tiles = min(p.total_tiles, (long long)__ldcg(p.status + kWgradActiveWord) * p.tiles_per_expert);
  }

  // Tiles in LPT order (experts by decreasing token count).  The dynamic schedule hands them out
  // from both ends of that order, so each SM interleaves MMA-bound long reductions with
  // epilogue-bound short ones: one tile from the long end, then kShortPerLong from the short end.
  // When overwriting, one short tile per long one; when accumulating, five: the epilogue's
  // reduce-add also reads every output tile, and spreading the short tiles' read-modify-write
  // traffic over the whole run beats leaving a tail of short tiles only.  The static schedule
  // deals the tiles round-robin.
  __device__ TileWork tile(long long t) const {
    const long long per = p.accumulate ? 6 : 2;  // claims per long-end tile (1 + kShortPerLong)
    const long long grp = t / per, j = t - grp * per;
    const bool short_end = j != 0;
    const long long idx = !p.dynamic ? t : short_end ? total_tiles - 1 - (grp * (per - 1) + j - 1) : grp;
    const int slot = (int)(idx / p.tiles_per_expert);
    const int local = (int)(idx % p.tiles_per_expert);
    TileWork w;
    // checked build: an expert slot or order entry outside [0, L) makes the tile a skipped one
    const bool slot_ok = MGG_IN_BOUNDS(p.status, slot >= 0 && slot < p.L, 411, slot);
    int e, begin, end;
    if (p.dynamic && short_end) {  // the short end of the order
      decode(c_short, slot, slot_ok);
      e = c_short.e, begin = c_short.begin, end = c_short.end;
    } else {
      decode(c_long, slot, slot_ok);
      e = c_long.e, begin = c_long.begin, end = c_long.end;
    }
    if (!MGG_IN_BOUNDS(p.status, e >= 0 && e < p.L, 412, e) || !slot_ok) {
      w = TileWork{0, 0, 0, 0, 0, 0};
      return w;
    }
    w.expert = e;
    w.active = (end > begin) || !p.accumulate;
    w.m0 = (local / p.tiles_n) * kTileM;
    w.n0 = (local % p.tiles_n) * BN;
    w.k0 = begin;
    w.num_kb = (end - begin) / BK;
    if (!(MGG_IN_BOUNDS(p.status, w.m0 < p.hidden, 413, w.m0) && MGG_IN_BOUNDS(p.status, w.n0 < p.inter, 414, w.n0)))
      w.active = 0;
    return w;
  }

  static __device__ __forceinline__ void load2(uint32_t dst, const void* map, uint32_t bar, int x, int y) {
    if constexpr (PAIR) tma_load_2d_pair(dst, map, bar, x, y);
    else tma_load_2d(dst, map, bar, x, y);
  }
  static __device__ __forceinline__ void load3(uint32_t dst, const void* map, uint32_t bar, int x, int y, int z) {
    if constexpr (PAIR) tma_load_3d_pair(dst, map, bar, x, y, z);
    else tma_load_3d(dst, map, bar, x, y, z);
  }

  // This CTA's 128 rows of A (m0 + 128 * rank) and its kBLoad columns of B (n0 + kBLoad * rank;
  // a narrow tile's N = BN/2 MMA takes BN/4 columns from each CTA of a pair, so the odd CTA's
  // start at n0 + BN/4; the loads keep their full box sizes, the columns past those unused).
  __device__ void issue_loads(const TileWork& w, int kb, uint32_t sa, uint32_t sb, uint32_t bar, int rank,
                              const MapAcquired& acq) const {
    const int k = w.k0 + kb * BK;
    const int mrow = w.m0 + rank * BM;
    const int ncol = w.n0 + rank * (narrow(w) ? kBLoad / 2 : kBLoad);
    if (kb == 0 && (p.a_maps != nullptr || p.b_maps != nullptr) && acq.first_use(w.expert)) {
      if (p.a_maps != nullptr) tmap_acquire(p.a_maps + w.expert);
      if (p.b_maps != nullptr) tmap_acquire(p.b_maps + w.expert);
    }
    if (p.a_maps != nullptr) {
      const CUtensorMap* m = p.a_maps + w.expert;
      load2(sa, m, bar, kb * BK, mrow);
    } else if (!p.a_mn) {
      load2(sa, &p.tmap_a, bar, k, mrow);
    } else if (p.a_blocked) {
      load3(sa, &p.tmap_a, bar, 0, k, mrow / 64);
    } else {
      load2(sa, &p.tmap_a, bar, mrow, k);
      load2(sa + 8192, &p.tmap_a, bar, mrow + 64, k);
    }
    if (p.b_maps != nullptr) {
      load2(sb, p.b_maps + w.expert, bar, kb * BK, ncol);
    } else if (p.b_mn && p.b_blocked) {
      load3(sb, &p.tmap_b, bar, 0, k, ncol / 64);
    } else if (p.b_mn) {
#pragma unroll
      for (int j = 0; j < kBLoad / 64; ++j) load2(sb + j * 8192, &p.tmap_b, bar, ncol + 64 * j, k);
    } else {
      load2(sb, &p.tmap_b, bar, k, ncol);
    }
  }

  // The last column tile of an output whose width leaves at most 128 columns there (inter % 256 in
  // (0, 128]) runs N = 128 MMAs: half the tensor work of a full tile for the same result.
  __device__ __forceinline__ bool narrow(const TileWork& w) const { return BN == 256 && p.inter - w.n0 <= BN / 2; }

  __device__ void prologue(const TileWork&, long long, const EpiCtx&) const {}

  // Writes 64 accumulator columns of this lane's row, starting at tile column `tc` (a multiple of
  // 64; `n` of them lie inside the output), held in v: added to the old values for 16-bit
  // accumulation, staged through the warp's shared-memory boxes and sent out by TMA (a bulk
  // reduce-add for fp32 accumulation).  Lane 0 issues the copies.
  __device__ __forceinline__ void drain64(const TileWork& w, const EpiCtx& ctx, float (&v)[64], int tc, int n,
                                          const CUtensorMap* map) const {
    const int lane = ctx.lane, e = w.expert;
    const int row0 = w.m0 + ctx.rank * BM + ctx.q * 32;
    const int row = row0 + lane;
    const uint32_t stg = smem_u32(ctx.stg);
    const bool discrete = p.out_maps != nullptr;
    // fp32 accumulation is a bulk reduce-add at the memory side; 16-bit accumulation reads the old values
    const bool reduce = p.accumulate && OS == 4;
    const bool add_old = p.accumulate && OS == 2;
    if (row0 >= p.hidden || n <= 0) return;  // rows past hidden (single-CTA tiles only): nothing to write
    if constexpr (OS == 4) {
      if (p.out_blocked) {  // inter % 64 == 0: both 32-column chunks exist; one 8 KB store for the pair
        if (lane == 0) bulk_wait_read<0>();  // both boxes of the ring have been read
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int i = 0; i < 8; ++i)
            st_shared_v4(stg + j * 4096u + swz128w(lane, i), __float_as_uint(v[32 * j + 4 * i]),
                         __float_as_uint(v[32 * j + 4 * i + 1]), __float_as_uint(v[32 * j + 4 * i + 2]),
                         __float_as_uint(v[32 * j + 4 * i + 3]));
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          const int blk = (w.n0 + tc) >> 5;  // first 32-column block of the pair
          if (discrete) {
            if (reduce) tma_reduce_add_3d(map, stg, 0, row0, blk);
            else tma_store_3d(map, stg, 0, row0, blk);
          } else {
            if (reduce) tma_reduce_add_4d(map, stg, 0, row0, blk, e);
            else tma_store_4d(map, stg, 0, row0, blk, e);
          }
          bulk_commit_group();
        }
        return;
      }
    }
#pragma unroll
    for (int j = 0; j < 64 / CW; ++j) {
      if (j * CW >= n) break;
      const int col0 = w.n0 + tc + j * CW;
      if (add_old && row < p.hidden && MGG_IN_BOUNDS(p.status, e < p.L && col0 < p.inter, 202, col0)) {
        const char* base = discrete ? reinterpret_cast<const char*>(__ldg(p.out_ptrs + e))
                                    : static_cast<const char*>(p.out) + (size_t)e * p.hidden * (size_t)p.inter * OS;
        const int nc = p.inter - col0 < CW ? p.inter - col0 : CW;
        const size_t idx = (size_t)row * p.inter + col0;
#pragma unroll
        for (int h = 0; h < CW / 32; ++h) {
          float old[32];
          load32_n(base, p.out_dtype, idx + 32 * h, old, nc - 32 * h);
#pragma unroll
          for (int k = 0; k < 32; ++k) v[CW * j + 32 * h + k] += old[k];
        }
      }
      // the box was last filled kBoxes stores ago: wait until at most kBoxes - 1 stores still read
      const uint32_t box = stg + (stg_uses % kBoxes) * 4096u;
      ++stg_uses;
      if (lane == 0) bulk_wait_read<kBoxes - 1>();
      __syncwarp();
      const float* vc = v + CW * j;
      if constexpr (OS == 4) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_shared_v4(box + swz128w(lane, i), __float_as_uint(vc[4 * i]), __float_as_uint(vc[4 * i + 1]),
                       __float_as_uint(vc[4 * i + 2]), __float_as_uint(vc[4 * i + 3]));
      } else {
        const int dt = p.out_dtype;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          st_shared_v4(box + swz128w(lane, i), pack2(vc[8 * i], vc[8 * i + 1], dt),
                       pack2(vc[8 * i + 2], vc[8 * i + 3], dt), pack2(vc[8 * i + 4], vc[8 * i + 5], dt),
                       pack2(vc[8 * i + 6], vc[8 * i + 7], dt));
      }
      fence_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (discrete) {
          if (reduce) tma_reduce_add_2d(map, box, col0, row0);
          else tma_store_2d(map, box, col0, row0);
        } else {
          if (reduce) tma_reduce_add_3d(map, box, col0, row0, e);
          else tma_store_3d(map, box, col0, row0, e);
        }
        bulk_commit_group();
      }
    }
  }

  // 64 accumulator columns starting at column tc of this warp's TMEM lanes, as fp32 (zeros when
  // the tile has no accumulator: an empty expert written in overwrite mode).
  __device__ __forceinline__ void load64(uint32_t taddr, bool have_acc, int tc, float (&v)[64]) const {
    if (have_acc) {
      uint32_t r[64];
      // BN is a multiple of 64: never past this accumulator
      tmem_load_64cols(taddr + (MGG_IN_BOUNDS(p.status, tc + 64 <= BN, 204, tc) ? tc : 0), r);
#pragma unroll
      for (int k = 0; k < 64; ++k) v[k] = __uint_as_float(r[k]);
    } else {
#pragma unroll
      for (int k = 0; k < 64; ++k) v[k] = 0.f;
    }
  }

  __device__ void epilogue(const TileWork& w, long long t, uint32_t taddr, bool have_acc, const EpiCtx& ctx,
                           AccRelease rel) const {
    const int lane = ctx.lane;
    const int e = w.expert;
    const int ncols = p.inter - w.n0 < BN ? p.inter - w.n0 : BN;
    const bool discrete = p.out_maps != nullptr;
    const CUtensorMap* map = discrete ? p.out_maps + e : &p.tmap_out;
    if (discrete && lane == 0 && ctx.acq.first_use(e)) tmap_acquire(map);
    // one TMEM load per 64 accumulator columns (tcgen05.ld 32x32b.x64), the accumulator freed
    // after the last load
#pragma unroll 1
    for (int tc = 0; tc < ncols; tc += 64) {
      float v[64];
      load64(taddr, have_acc, tc, v);
      if (have_acc && tc + 64 >= ncols) rel(lane);
      drain64(w, ctx, v, tc, ncols - tc, map);
    }
    // one entry per CTA tile of 128 rows (a pair's tile logs two)
    const long long idx = PAIR ? 2 * t + ctx.rank : t;
    if (p.tile_log != nullptr && ctx.q == 0 && lane == 0 && idx < p.tile_log_cap) {
      int32_t* l = p.tile_log + 4 * idx;
      l[0] = e;
      l[1] = w.m0 + ctx.rank * BM;
      l[2] = w.n0;
      l[3] = (int32_t)blockIdx.x;
    }
  }
};

template <int BN, int STAGES, int OS, bool PAIR>
__global__ void __launch_bounds__(cta_threads(kWgradEpiWarps), 1) wgrad_kernel(const __grid_constant__ WgradParams prm) {
  WgradPolicy<BN, OS, PAIR> pol(prm);
  persistent_gemm<BN, STAGES, PAIR>(pol);
}

// Checks offsets / output pointers, orders experts by decreasing token count and builds
// the per-expert maps of tensor_ragged K-major operands.
__global__ void wgrad_prep_kernel(const int32_t* offsets, int L, long long T, const int64_t* out_ptrs,
                                  const __grid_constant__ CUtensorMap tmpl_a, const __grid_constant__ CUtensorMap tmpl_b,
                                  const __grid_constant__ CUtensorMap tmpl_out, const void* a, const void* b,
                                  int hidden, int inter, int a_ragged, int b_ragged, CUtensorMap* a_maps,
                                  CUtensorMap* b_maps, CUtensorMap* out_maps, int32_t* order, int* status,
                                  int accumulate) {
  griddep_launch_dependents();  // the GEMM kernel may launch now; it waits for this kernel's results
  __shared__ int s_cnt[1024];
  bool bad_off = false, bad_ptr = false;
  for (int e = threadIdx.x; e < L; e += blockDim.x) {
    const int prev = e ? offsets[e - 1] : 0;
    const int cur = offsets[e];
    if (cur < prev || ((cur - prev) & 255) != 0) bad_off = true;
    if (e == L - 1 && (long long)cur != T) bad_off = true;
    if (out_ptrs != nullptr) {
      const long long ptr = out_ptrs[e];
      if (ptr == 0 || (ptr & 15) != 0) bad_ptr = true;
    }
    s_cnt[e] = cur - prev;
  }
  const int any_off = __syncthreads_or(bad_off);
  const int any_ptr = __syncthreads_or(bad_ptr);
  const int nonempty = __syncthreads_count((int)threadIdx.x < L && s_cnt[threadIdx.x] > 0);
  if (threadIdx.x == 0) {
    status[0] = any_off ? (int)MGG_ERR_DEVICE_OFFSETS : any_ptr ? (int)MGG_ERR_DEVICE_POINTER : 0;
    status[1] = 0;
    status[2] = 0;
    status[3] = 0;
    status[kWgradActiveWord] = (any_off || any_ptr) ? 0 : accumulate ? nonempty : L;  // experts with tiles
  }
  if (any_off || any_ptr) return;
  // stable rank by decreasing count
  for (int e = threadIdx.x; e < L; e += blockDim.x) {
    const int ce = s_cnt[e];
    int rank = 0;
    for (int f = 0; f < L; ++f) {
      const int cf = s_cnt[f];
      rank += (cf > ce) || (cf == ce && f < e);
    }
    order[rank] = e;
  }
  if (!a_ragged && !b_ragged && out_ptrs == nullptr) return;
  for (int e = threadIdx.x; e < L; e += blockDim.x) {
    if (out_ptrs != nullptr) {  // every expert, empty ones included (zero-filled in overwrite mode)
      uint4* dst = reinterpret_cast<uint4*>(out_maps + e);
      const uint4* src = reinterpret_cast<const uint4*>(&tmpl_out);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = src[i];
      tmap_replace_address(out_maps + e, reinterpret_cast<const void*>(out_ptrs[e]));
    }
    const int ke = s_cnt[e];
    if (ke == 0) continue;
    const int begin = e ? offsets[e - 1] : 0;
    if (a_ragged) {
      uint4* dst = reinterpret_cast<uint4*>(a_maps + e);
      const uint4* src = reinterpret_cast<const uint4*>(&tmpl_a);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = src[i];
      tmap_replace_address(a_maps + e, static_cast<const __nv_bfloat16*>(a) + (size_t)begin * hidden);
      tmap_replace_dim(a_maps + e, 0, (uint32_t)ke);
      tmap_replace_stride0(a_maps + e, (uint64_t)ke * 2);
    }
    if (b_ragged) {
      uint4* dst = reinterpret_cast<uint4*>(b_maps + e);
      const uint4* src = reinterpret_cast<const uint4*>(&tmpl_b);
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[i] = src[i];
      tmap_replace_address(b_maps + e, static_cast<const __nv_bfloat16*>(b) + (size_t)begin * inter);
      tmap_replace_dim(b_maps + e, 0, (uint32_t)ke);
      tmap_replace_stride0(b_maps + e, (uint64_t)ke * 2);
    }
  }
  tmap_release();
}

// 128 x 256 tiles keep the tensor pipe fed (128 x 128 tiles are shared-memory-bandwidth bound);
// narrow outputs fall back to 128 columns.
int wgrad_tile_n(int64_t inter) { return inter > 128 ? 256 : 128; }

// Ring depth: as many stages as the shared memory holds, at most 6 (a single CTA loads 48 KB
// (BN = 256) or 32 KB (BN = 128) per stage, a CTA of a pair half of the B part of that).
template <int BN, bool PAIR>
constexpr int wgrad_stages() {
  return max_stages(PAIR ? BN / 2 : BN, kWgradEpiWarps, kWgradStgBytes, num_acc(BN), 6);
}

template <int BN, int OS, bool PAIR>
static cudaError_t launch_wgrad_bn(const WgradLaunch& Lc, WgradParams& prm, cudaStream_t stream) {
  constexpr int STAGES = wgrad_stages<BN, PAIR>();
  using S = SmemLayout<PAIR ? BN / 2 : BN, STAGES, kWgradEpiWarps, kWgradStgBytes, num_acc(BN)>;
  auto kern = wgrad_kernel<BN, STAGES, OS, PAIR>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::DYN_BYTES);
  if (err != cudaSuccess) return err;
  static UnitCache cache;  // co-resident CTAs (pairs) of this variant, asked once per device
  return launch_persistent(kern, prm, prm.total_tiles, Lc.num_sms, PAIR, cta_threads(kWgradEpiWarps), S::DYN_BYTES,
                           cache.slot(Lc.device), stream);
}

cudaError_t launch_wgrad(const WgradLaunch& Lc, cudaStream_t stream) {
  const mgg_wgrad_args& a = *Lc.args;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int* status = reinterpret_cast<int*>(ws);
  CUtensorMap* a_maps = reinterpret_cast<CUtensorMap*>(ws + kWsHeaderBytes);
  CUtensorMap* b_maps = a_maps + a.L;
  CUtensorMap* out_maps = b_maps + a.L;
  int32_t* order = reinterpret_cast<int32_t*>(ws + kWsHeaderBytes + 3 * kTmapBytes * (size_t)a.L);

  // stream order: the optional tile-log fill, the preparation kernel, then the GEMM kernel, which
  // may launch while the preparation kernel runs
  cudaError_t err;
  if (a.tile_log != nullptr && a.tile_log_capacity > 0) {
    err = cudaMemsetAsync(a.tile_log, 0xff, sizeof(int32_t) * 4 * (size_t)a.tile_log_capacity, stream);
    if (err != cudaSuccess) return err;
  }
  wgrad_prep_kernel<<<1, 1024, 0, stream>>>(a.offsets, (int)a.L, (long long)a.tokens_sum, a.out_ptrs, Lc.tmap_a,
                                            Lc.tmap_b, Lc.tmap_out, a.a, a.b, (int)a.hidden, (int)a.inter,
                                            Lc.a_ragged, Lc.b_ragged, a_maps, b_maps, out_maps, order, status,
                                            a.accumulate ? 1 : 0);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;

  const int BN = Lc.tile_n;
  const long long tiles_m = Lc.pair ? a.hidden / (2 * BM) : (a.hidden + BM - 1) / BM;  // pair: hidden % 256 == 0
  const long long tiles_n = (a.inter + BN - 1) / BN;
  const long long total = a.L * tiles_m * tiles_n;
  if (total == 0) return cudaSuccess;
  WgradParams prm;
  prm.tmap_a = Lc.tmap_a;
  prm.tmap_b = Lc.tmap_b;
  prm.tmap_out = Lc.tmap_out;
  prm.a_maps = Lc.a_ragged ? a_maps : nullptr;
  prm.b_maps = Lc.b_ragged ? b_maps : nullptr;
  prm.out_maps = a.out_ptrs != nullptr ? out_maps : nullptr;
  prm.offsets = a.offsets;
  prm.order = order;
  prm.out = a.out;
  prm.out_ptrs = a.out_ptrs;
  prm.status = status;
  prm.tile_log = a.tile_log;
  prm.tile_log_cap = a.tile_log != nullptr ? a.tile_log_capacity : 0;
  prm.total_tiles = total;
  prm.dynamic = a.sched == MGG_SCHED_DYNAMIC;
  prm.hidden = (int)a.hidden;
  prm.inter = (int)a.inter;
  prm.L = (int)a.L;
  prm.tiles_n = (int)tiles_n;
  prm.tiles_per_expert = (int)(tiles_m * tiles_n);
  prm.a_mn = (a.a_major == MGG_MAJOR_MN) ? 1 : 0;
  prm.b_mn = (a.b_major == MGG_MAJOR_MN) ? 1 : 0;
  prm.a_blocked = Lc.a_blocked ? 1 : 0;
  prm.b_blocked = Lc.b_blocked ? 1 : 0;
  prm.out_blocked = Lc.out_blocked ? 1 : 0;
  prm.out_dtype = a.out_dtype;
  prm.accumulate = a.accumulate != 0;
  const bool fp32 = a.out_dtype == MGG_FP32;
  if (Lc.pair) {
    if (BN == 256) return fp32 ? launch_wgrad_bn<256, 4, true>(Lc, prm, stream) : launch_wgrad_bn<256, 2, true>(Lc, prm, stream);
    return fp32 ? launch_wgrad_bn<128, 4, true>(Lc, prm, stream) : launch_wgrad_bn<128, 2, true>(Lc, prm, stream);
  }
  if (BN == 256) return fp32 ? launch_wgrad_bn<256, 4, false>(Lc, prm, stream) : launch_wgrad_bn<256, 2, false>(Lc, prm, stream);
  return fp32 ? launch_wgrad_bn<128, 4, false>(Lc, prm, stream) : launch_wgrad_bn<128, 2, false>(Lc, prm, stream);
}

}  // namespace mgg
