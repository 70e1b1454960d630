// Persistent, warp-specialised grouped GEMM pipeline for sm_103a (one CTA per SM).
//
//   warp 0      TMA producer: one elected thread streams BK-wide slices of the A and
//               B tiles into a STAGES-deep shared-memory ring (full/empty mbarriers).
//   warp 1      MMA issuer: allocates TMEM, one thread issues tcgen05.mma (128 x BN x 16,
//               bf16 in, fp32 accumulate) into one of two TMEM accumulators and commits
//               the ring slots and the finished accumulator to mbarriers.
//   warps 2..5  epilogue: each warp owns one 32-lane TMEM sub-partition (rows
//               32*(warp%4) .. +31 of the tile), reads the accumulator with tcgen05.ld
//               and hands it to the operation's epilogue while the MMA warp already
//               accumulates the next tile into the other TMEM buffer.
//
// The operation supplies a policy object P with
//   total_tiles, status, a_mn, b_mn, dynamic        status[3] is the dynamic scheduler's tile
//                                                   counter (zeroed by the preparation kernel)
//   TileWork tile(long long t)                      same answer for every role
//   issue_loads(w, kb, sa, sb, bar)                 producer thread
//   EPI_WARPS                                       epilogue warps (multiple of 4)
//   STG_BYTES                                       shared memory per epilogue warp
//   prologue(w, t, ctx)                             one epilogue warp, before it waits for the
//                                                   tile's accumulator (e.g. to start input loads)
//   epilogue(w, t, taddr, have_acc, ctx, rel)       one epilogue warp; EPI_WARPS/4 warps share TMEM
//        sub-partition ctx.q and split the tile's 32-column chunks (chunk c belongs to ctx.half =
//        c % (EPI_WARPS/4)); ctx.stg is the warp's 1024-byte aligned STG_BYTES of shared memory,
//        ctx.bars four mbarriers (count 1) it owns; `rel` frees the TMEM accumulator and must be
//        called exactly once per tile when have_acc, after the warp's last tcgen05.ld of it.
#pragma once

#include "mgg_ptx.cuh"

namespace mgg {

constexpr int BM = 128;     // tile rows = UMMA M (cta_group::1)
constexpr int BK = 64;      // K elements per ring slot: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;  // K of one kind::f16 MMA
constexpr int kSchedRing = 8;      // tile indices in flight from the producer to the other roles

// Threads of a CTA with `epi_warps` epilogue warps (a multiple of 4) after the producer and MMA warps.
__host__ __device__ constexpr int cta_threads(int epi_warps) { return 64 + 32 * epi_warps; }

struct TileWork {
  int active;   // 0: the tile is skipped by every role
  int expert;
  int m0, n0;   // tile origin in the output
  int k0;       // first reduction index of the tile (operation-specific meaning)
  int num_kb;   // number of BK slices; 0 = no MMA (the epilogue writes without TMEM)
};

// STG: bytes of output staging per epilogue warp (a multiple of 4 KB: 32 rows x 128 bytes per box).
template <int BN, int STAGES, int EPI_WARPS, int STG>
struct SmemLayout {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_WARPS * STG;
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * kSchedRing + 4 * EPI_WARPS;
  static constexpr int SCHED_OFF = BAR_OFF + NUM_BARS * 8;
  static constexpr int MISC_OFF = SCHED_OFF + kSchedRing * 8;
  static constexpr int BYTES = MISC_OFF + 16;
  static constexpr int DYN_BYTES = BYTES + 1024;  // slack to align the ring to 1024 B
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "ring slots must stay 1024-byte aligned");
  static_assert(DYN_BYTES <= 232448, "shared memory per block");
};

// What one epilogue warp owns.
struct EpiCtx {
  int q;          // TMEM sub-partition (rows 32q .. 32q+31 of the tile)
  int half;       // index among the warps sharing that sub-partition
  int lane;
  uint8_t* stg;   // STG_BYTES of shared memory, 1024-byte aligned
  uint64_t* bars; // four mbarriers initialised with count 1
  WaitGuard wg;
};

// Frees one TMEM accumulator for the MMA warp (called by every lane of an epilogue warp).
struct AccRelease {
  uint64_t* bar;
  __device__ __forceinline__ void operator()(int lane) const {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
  }
};

__host__ __device__ constexpr uint32_t tmem_cols_for(int cols) {
  return cols <= 32 ? 32u : cols <= 64 ? 64u : cols <= 128 ? 128u : cols <= 256 ? 256u : 512u;
}

// Bounded wait used only while tearing down after an abort: ignores the abort flag.
static __device__ __noinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs / 4) return;
  }
}

// Every lane of the warp waits; the warp proceeds only if all lanes saw the phase.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, WaitGuard g, int where) {
  const bool ok = mbar_wait(bar, parity, g, where);
  return __all_sync(0xffffffffu, ok);
}

template <int BN, int STAGES, class P>
__device__ __forceinline__ void persistent_gemm(const P& p) {
  constexpr int kEpiWarps = P::EPI_WARPS;
  static_assert(kEpiWarps % 4 == 0, "whole TMEM sub-partitions");
  using S = SmemLayout<BN, STAGES, kEpiWarps, P::STG_BYTES>;
  constexpr uint32_t TMEM_COLS = tmem_cols_for(2 * BN);
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "UMMA N");

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* done_bar = tempty_bar + 2;
  uint64_t* sfull_bar = done_bar + 1;           // [kSchedRing] a tile index was published
  uint64_t* sempty_bar = sfull_bar + kSchedRing;  // [kSchedRing] every role has read it
  uint64_t* epi_bars = sempty_bar + kSchedRing;   // [4 * kEpiWarps] owned by the epilogue warps
  volatile long long* sched_ring = reinterpret_cast<volatile long long*>(smem + S::SCHED_OFF);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::MISC_OFF + 4);

  // The preparation kernel of this call found invalid device-side arguments.
  if (*reinterpret_cast<volatile int*>(p.status) != 0) return;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(done_bar, 1);
    for (int r = 0; r < kSchedRing; ++r) {
      mbar_init(&sfull_bar[r], 1);
      mbar_init(&sempty_bar[r], 1 + kEpiWarps);  // the MMA thread and every epilogue warp
    }
    for (int b = 0; b < 4 * kEpiWarps; ++b) mbar_init(&epi_bars[b], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const WaitGuard wg{abort_flag, p.status};
  const bool dynamic = p.dynamic != 0;
  const long long kEnd = 0x7fffffffffffffffLL;

  // Static schedule: CTA b takes tiles b, b + grid, ...  Dynamic schedule: the producer thread
  // claims the next tile from the global counter and publishes it to the MMA thread and the
  // epilogue warps through sched_ring; every role sees the same tile sequence.
  auto static_tile = [&](long long n) -> long long { return (long long)blockIdx.x + n * (long long)gridDim.x; };
  auto consume_tile = [&](long long n, bool is_warp) -> long long {
    const int r = (int)(n % kSchedRing);
    const uint32_t ph = (uint32_t)((n / kSchedRing) & 1);
    const bool ok = is_warp ? warp_wait(&sfull_bar[r], ph, wg, 6) : mbar_wait(&sfull_bar[r], ph, wg, 6);
    if (!ok) return kEnd;
    const long long t = sched_ring[r];
    if (is_warp) __syncwarp();
    if (!is_warp || lane == 0) mbar_arrive(&sempty_bar[r]);
    return t;
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      int* counter = p.status + 3;
      auto produce_tile = [&](long long n) -> long long {
        if (!dynamic) return static_tile(n);
        const int r = (int)(n % kSchedRing);
        if (!mbar_wait(&sempty_bar[r], (uint32_t)(((n / kSchedRing) & 1) ^ 1), wg, 5)) return kEnd;
        const long long t = atomicAdd(counter, 1);
        sched_ring[r] = t;
        mbar_arrive(&sfull_bar[r]);
        return t;
      };
      long long n_tile = 0;
      for (long long t = produce_tile(n_tile++); t < p.total_tiles && ok; t = produce_tile(n_tile++)) {
        const TileWork w = p.tile(t);
        if (!w.active) continue;
        for (int kb = 0; kb < w.num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wg, 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full_bar[stage], S::STAGE_BYTES);
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          p.issue_loads(w, kb, sa, sa + S::A_BYTES, smem_u32(&full_bar[stage]));
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {  // let the copies already in flight land before the CTA exits
        const long long n_flight = issued < STAGES ? issued : STAGES;
        for (long long i = 1; i <= n_flight; ++i) {
          const long long n = issued - i;
          mbar_wait_drain(&full_bar[n % STAGES], (uint32_t)((n / STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN, p.a_mn, p.b_mn);
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, a_kstep = p.a_mn ? 2048u : 32u;
      const uint32_t b_lbo = p.b_mn ? 8192u : 16u, b_kstep = p.b_mn ? 2048u : 32u;
      int stage = 0;
      uint32_t phase = 0, local = 0;
      bool ok = true;
      long long n_tile = 0;
      auto next_tile = [&]() { const long long n = n_tile++; return dynamic ? consume_tile(n, false) : static_tile(n); };
      for (long long t = next_tile(); t < p.total_tiles && ok; t = next_tile()) {
        const TileWork w = p.tile(t);
        if (!w.active || w.num_kb == 0) continue;
        const uint32_t acc = local & 1u, use = local >> 1;
        if (!mbar_wait(&tempty_bar[acc], (use & 1u) ^ 1u, wg, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < w.num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, wg, 3)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t sb = sa + S::A_BYTES;
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint64_t ad = smem_desc_sw128(sa + k * a_kstep, a_lbo, 1024u);
            const uint64_t bd = smem_desc_sw128(sb + k * b_kstep, b_lbo, 1024u);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&empty_bar[stage]));  // ring slot free once these MMAs finish
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(smem_u32(&tfull_bar[acc]));  // accumulator complete
        ++local;
      }
      umma_commit(smem_u32(done_bar));  // all MMAs of this CTA retired before TMEM is freed
      mbar_wait_drain(done_bar, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue warps
    const int q = warp & 3;             // TMEM sub-partition this warp may access
    const int half = (warp - 2) >> 2;   // which of the sub-partition's warps
    const EpiCtx ctx{q, half, lane, smem + S::EPI_OFF + (warp - 2) * P::STG_BYTES, epi_bars + 4 * (warp - 2), wg};
    uint32_t local = 0;
    long long n_tile = 0;
    auto next_tile = [&]() { const long long n = n_tile++; return dynamic ? consume_tile(n, true) : static_tile(n); };
    for (long long t = next_tile(); t < p.total_tiles; t = next_tile()) {
      const TileWork w = p.tile(t);
      if (!w.active) continue;
      p.prologue(w, t, ctx);
      if (w.num_kb == 0) {
        p.epilogue(w, t, 0u, false, ctx, AccRelease{nullptr});
        continue;
      }
      const uint32_t acc = local & 1u, use = local >> 1;
      if (!warp_wait(&tfull_bar[acc], use & 1u, wg, 4)) break;
      tc_fence_after();
      p.epilogue(w, t, tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN, true, ctx, AccRelease{&tempty_bar[acc]});
      ++local;
    }
    if (lane == 0) bulk_wait_all();  // bulk stores complete before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------
// epilogue helpers: 32 consecutive elements of one row
// ------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

// Loads 32 elements (dtype 0 bf16, 1 fp16, 2 fp32) starting at element `idx` of `base`.
__device__ __forceinline__ void load32(const void* base, int dtype, size_t idx, float (&v)[32]) {
  if (dtype == MGG_FP32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 x = __ldg(p + i);
      v[4 * i + 0] = x.x;
      v[4 * i + 1] = x.y;
      v[4 * i + 2] = x.z;
      v[4 * i + 3] = x.w;
    }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = __ldg(p + i);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (dtype == MGG_BF16) {
          v[8 * i + 2 * j + 0] = bf16_bits_to_float(w[j] & 0xffffu);
          v[8 * i + 2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
        } else {
          v[8 * i + 2 * j + 0] = __half2float(__ushort_as_half((unsigned short)(w[j] & 0xffffu)));
          v[8 * i + 2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(w[j] >> 16)));
        }
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int dtype) {
  if (dtype == MGG_BF16) {
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
  }
  const uint32_t lo = __half_as_ushort(__float2half_rn(a));
  const uint32_t hi = __half_as_ushort(__float2half_rn(b));
  return lo | (hi << 16);
}

// Stores the first `n` (a multiple of 8, <= 32) of 32 values at element `idx` of `base`.
__device__ __forceinline__ void store32(void* base, int dtype, size_t idx, const float (&v)[32], int n = 32) {
  if (dtype == MGG_FP32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (4 * i < n) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else {
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (8 * i < n)
        p[i] = make_uint4(pack2(v[8 * i], v[8 * i + 1], dtype), pack2(v[8 * i + 2], v[8 * i + 3], dtype),
                          pack2(v[8 * i + 4], v[8 * i + 5], dtype), pack2(v[8 * i + 6], v[8 * i + 7], dtype));
  }
}

// Like load32 but only the first `n` (multiple of 8) elements are read; the rest become 0.
__device__ __forceinline__ void load32_n(const void* base, int dtype, size_t idx, float (&v)[32], int n) {
  if (n >= 32) {
    load32(base, dtype, idx, v);
    return;
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = 0.f;
  if (dtype == MGG_FP32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (4 * i < n) {
        const float4 x = p[i];
        v[4 * i + 0] = x.x;
        v[4 * i + 1] = x.y;
        v[4 * i + 2] = x.z;
        v[4 * i + 3] = x.w;
      }
  } else {
    const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (8 * i < n) {
        const uint4 x = p[i];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (dtype == MGG_BF16) {
            v[8 * i + 2 * j + 0] = bf16_bits_to_float(w[j] & 0xffffu);
            v[8 * i + 2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
          } else {
            v[8 * i + 2 * j + 0] = __half2float(__ushort_as_half((unsigned short)(w[j] & 0xffffu)));
            v[8 * i + 2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(w[j] >> 16)));
          }
        }
      }
  }
}

// Column sums of a 32 x 32 block held one row per lane: after the call lane l holds the
// sum over all 32 lanes of column l (recursive-halving exchange, 31 shuffles).
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < off; ++k) {
      const float send = upper ? v[k] : v[k + off];
      const float keep = upper ? v[k + off] : v[k];
      v[k] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

}  // namespace mgg
