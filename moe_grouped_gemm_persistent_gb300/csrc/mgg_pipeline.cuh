// Persistent, warp-specialised grouped GEMM pipeline for sm_103a.
//
//   warp 0      TMA producer: one elected thread streams BK-wide slices of the A and B tiles
//               into a STAGES-deep shared-memory ring (full/empty mbarriers).
//   warp 1      TMEM allocator and MMA issuer: one thread issues tcgen05.mma (bf16 in, fp32
//               accumulate) into one of the TMEM accumulators (512 / BN of them, at most 4) and
//               commits the ring slots and the finished accumulator to mbarriers.
//   warp 2      scheduler: one thread claims, decodes and publishes the tiles to every role.
//   warps 3..   epilogue: each warp owns one 32-lane TMEM sub-partition (rows 32*(warp%4) ..
//               +31 of its CTA's rows), reads the accumulator with tcgen05.ld and hands it to the
//               operation's epilogue while the MMA already accumulates the next tile.
//
// The kernel is launched with programmatic stream serialization behind its call's preparation
// kernel: it initialises its barriers and allocates TMEM while that kernel may still run, then
// waits for it (griddepcontrol.wait) before reading anything it wrote, and lets the next
// programmatically launched kernel start once its roles have finished.
//
// Single CTA (PAIR = false): one CTA per SM computes 128 x BN tiles with cta_group::1.
// CTA pair (PAIR = true): a cluster of two CTAs on two SMs computes 256 x BN tiles with
// cta_group::2 MMAs issued by the even CTA; each CTA loads its own 128 rows of A and half of the
// BN columns of B, so per SM the B traffic and the ring slot shrink by half, and each CTA's TMEM
// holds the accumulator rows it then writes out.  The even CTA's full barrier counts the bytes of
// both CTAs' loads; its MMA commits arrive on both CTAs' barriers (multicast); both CTAs' epilogue
// warps free the accumulator on the even CTA's barrier.
//
// The operation supplies a policy object P with
//   total_tiles, status, a_mn, b_mn, dynamic        status[3] is the dynamic scheduler's tile
//                                                   counter (zeroed by the preparation kernel)
//   on_prep_done()                                  every thread, once the preparation kernel's
//                                                   writes are visible (before any other use)
//   TileWork tile(long long t)                      called once per tile, by the scheduler thread
//   issue_loads(w, kb, sa, sb, bar, rank, acq)      producer thread; `bar` is the address the
//                                                   loads complete on (the even CTA's in a pair);
//                                                   `acq` records the maps it has acquired
//   bool narrow(w)                                  the tile's valid columns fit in BN/2: its MMAs
//                                                   have N = BN/2 (accumulator columns [0, BN/2);
//                                                   in a pair each CTA then supplies BN/4 of them)
//   EPI_WARPS, STG_BYTES                            epilogue warps (multiple of 4), bytes per warp
//   prologue(w, t, ctx)                             one epilogue warp, before it waits for the
//                                                   tile's accumulator (e.g. to start input loads)
//   epilogue(w, t, taddr, have_acc, ctx, rel)       one epilogue warp; EPI_WARPS/4 warps share TMEM
//        sub-partition ctx.q and split the tile's 32-column chunks (chunk c belongs to ctx.half =
//        c % (EPI_WARPS/4)); ctx.rank is the CTA's rank in the pair (its rows start at
//        m0 + 128*rank); ctx.stg is the warp's 1024-byte aligned STG_BYTES of shared memory,
//        ctx.bars four mbarriers (count 1) it owns; `rel` frees the TMEM accumulator and must be
//        called exactly once per tile when have_acc, after the warp's last tcgen05.ld of it.
#pragma once

#include <atomic>

#include "mgg_ptx.cuh"

namespace mgg {

constexpr int BM = 128;        // accumulator rows per CTA (UMMA M per CTA)
constexpr int BK = 64;         // K elements per ring slot: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;     // K of one kind::f16 MMA
constexpr int kSchedRing = 8;  // published tiles in flight from the scheduler to the other roles
// The scheduler claims the next tile once the producer has kClaimLeadKb (or fewer) k-slices of the
// tiles already published left to issue: early enough to hide the claim's atomic and decode (about
// 1.5 us), so that a run of short tiles does not stall the producer at every tile boundary, and
// late enough to keep the dynamic schedule's load balance (a tile claimed long before it starts
// cannot move).
constexpr int kClaimLeadKb = 10;
constexpr int kSchedEntry = 32; // bytes of one published tile: index + TileWork
constexpr int kMaxExperts = 1024;
constexpr int kAcqWords = kMaxExperts / 32;  // one bit per expert

// Per-thread record of the per-expert tensor maps (built in global memory by the preparation
// kernel) this thread has already acquired for the tensormap proxy.  One acquire per map and
// thread is enough: the maps do not change while the kernel runs, and the fence orders all of
// this thread's later TMA uses of the map after the preparation kernel's writes.
struct MapAcquired {
  uint32_t* bits;  // kAcqWords words of shared memory owned by one thread
  // True the first time expert e is seen: the caller then acquires that expert's maps.
  __device__ __forceinline__ bool first_use(int e) const {
    const uint32_t m = 1u << (e & 31);
    const uint32_t w = bits[e >> 5];
    if (w & m) return false;
    bits[e >> 5] = w | m;
    return true;
  }
};

// Threads of a CTA with `epi_warps` epilogue warps (a multiple of 4) after the producer, MMA and
// scheduler warps.
constexpr int kFirstEpiWarp = 3;
__host__ __device__ constexpr int cta_threads(int epi_warps) { return 32 * (kFirstEpiWarp + epi_warps); }

struct TileWork {
  int active;   // 0: the tile is skipped by every role
  int expert;
  int m0, n0;   // tile origin in the output
  int k0;       // first reduction index of the tile (operation-specific meaning)
  int num_kb;   // number of BK slices; 0 = no MMA (the epilogue writes without TMEM)
};

// TMEM accumulators of BN fp32 columns in the 512 columns of an SM (at most 4 in flight).
__host__ __device__ constexpr int num_acc(int bn) { return 512 / bn < 4 ? 512 / bn : 4; }

// BN_LOAD: B rows (N) this CTA loads per slot (BN, or BN/2 in a pair).
// STG: bytes of output staging per epilogue warp (a multiple of 4 KB: 32 rows x 128 bytes per box).
// NACC: TMEM accumulators (num_acc(BN)).
constexpr int kMaxSmemBytes = 232448;  // dynamic shared memory per block (227 KB)

// Dynamic shared memory of one CTA (the same arithmetic as SmemLayout below).
__host__ __device__ constexpr int smem_bytes(int bn_load, int stages, int epi_warps, int stg, int nacc) {
  return ((stages * (BM + bn_load) * BK * 2 + epi_warps * stg +
           (2 * stages + 2 * nacc + 1 + 2 * kSchedRing + 4 * epi_warps) * 8 + 15) / 16 * 16) +
         kSchedRing * kSchedEntry + (1 + epi_warps) * kAcqWords * 4 + 16 + 1024;
}

// Deepest operand ring (at most `cap` slots) that fits next to the epilogue's shared memory.
__host__ __device__ constexpr int max_stages(int bn_load, int epi_warps, int stg, int nacc, int cap) {
  int s = cap;
  while (s > 1 && smem_bytes(bn_load, s, epi_warps, stg, nacc) > kMaxSmemBytes) --s;
  return s;
}

template <int BN_LOAD, int STAGES, int EPI_WARPS, int STG, int NACC>
struct SmemLayout {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN_LOAD * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int EPI_OFF = STAGES * STAGE_BYTES;
  static constexpr int BAR_OFF = EPI_OFF + EPI_WARPS * STG;
  static constexpr int NUM_BARS = 2 * STAGES + 2 * NACC + 1 + 2 * kSchedRing + 4 * EPI_WARPS;
  static constexpr int SCHED_OFF = (BAR_OFF + NUM_BARS * 8 + 15) / 16 * 16;
  static constexpr int ACQ_OFF = SCHED_OFF + kSchedRing * kSchedEntry;  // producer, then each epilogue warp
  static constexpr int MISC_OFF = ACQ_OFF + (1 + EPI_WARPS) * kAcqWords * 4;
  static constexpr int BYTES = MISC_OFF + 16;  // TMEM address, abort flag, skip flag, issued k-slices
  static constexpr int DYN_BYTES = BYTES + 1024;  // slack to align the ring to 1024 B
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "ring slots must stay 1024-byte aligned");
  static_assert(SCHED_OFF % 16 == 0, "16-byte aligned published tiles");
  static_assert(DYN_BYTES == smem_bytes(BN_LOAD, STAGES, EPI_WARPS, STG, NACC), "layout arithmetic");
  static_assert(DYN_BYTES <= kMaxSmemBytes, "shared memory per block");
};

// What one epilogue warp owns.
struct EpiCtx {
  int q;          // TMEM sub-partition (rows 32q .. 32q+31 of this CTA's rows)
  int half;       // index among the warps sharing that sub-partition
  int lane;
  int rank;       // rank of the CTA in its pair (0 for a single CTA)
  uint8_t* stg;   // STG_BYTES of shared memory, 1024-byte aligned
  uint64_t* bars; // four mbarriers initialised with count 1
  MapAcquired acq;  // the tensor maps lane 0 of this warp has acquired
  WaitGuard wg;
};

// Frees one TMEM accumulator for the MMA thread (called by every lane of an epilogue warp):
// arrives on the accumulator's "empty" barrier, which lives in the even CTA of a pair.  Every
// tcgen05.ld of the accumulator has completed (tcgen05.wait::ld) before this is called, so the MMA
// can no longer change what the warp read: the odd CTA of a pair arrives with a relaxed (fence-free)
// remote arrive.
struct AccRelease {
  uint32_t bar;    // shared::cta address (single CTA) or shared::cluster address (pair)
  bool remote;
  __device__ __forceinline__ void operator()(int lane) const {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      if (remote) mbar_arrive_remote_relaxed(bar);
      else asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
    }
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

// Spins (sleeping briefly between looks) until the producer has at most kClaimLeadKb of the
// `published` k-slices left to issue (`issued` is the producer's running count, modulo 2^32).
// Bounded like the mbarrier waits: an abort of the CTA or the time limit ends it with false.
static __device__ __noinline__ bool wait_claim_lead(const volatile uint32_t* issued, uint32_t published, WaitGuard g,
                                                    int where) {
  if ((int)(published - *issued) <= kClaimLeadKb) return true;
  const unsigned long long t0 = globaltimer_ns();
  while ((int)(published - *issued) > kClaimLeadKb) {
    if (*g.abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_timeout(g, where);
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// Every lane of the warp waits; the warp proceeds only if all lanes saw the phase.
template <bool CLUSTER = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, WaitGuard g, int where) {
  const bool ok = CLUSTER ? mbar_wait_cluster(bar, parity, g, where) : mbar_wait(bar, parity, g, where);
  return __all_sync(0xffffffffu, ok);
}

template <int BN, int STAGES, bool PAIR, class P>
__device__ __forceinline__ void persistent_gemm(P& p) {
  constexpr int kEpiWarps = P::EPI_WARPS;
  static_assert(kEpiWarps % 4 == 0, "whole TMEM sub-partitions");
  constexpr int kBLoad = PAIR ? BN / 2 : BN;
  constexpr int NACC = num_acc(BN);
  using S = SmemLayout<kBLoad, STAGES, kEpiWarps, P::STG_BYTES, NACC>;
  constexpr uint32_t TMEM_COLS = tmem_cols_for(NACC * BN);
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "UMMA N");
  static_assert(!PAIR || BN % 128 == 0, "a pair splits B in 64-column multiples");

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;
  uint64_t* tempty_bar = tfull_bar + NACC;
  uint64_t* done_bar = tempty_bar + NACC;
  uint64_t* sfull_bar = done_bar + 1;             // [kSchedRing] a tile was published
  uint64_t* sempty_bar = sfull_bar + kSchedRing;  // [kSchedRing] every consumer has read it
  uint64_t* epi_bars = sempty_bar + kSchedRing;   // [4 * kEpiWarps] owned by the epilogue warps
  const uint32_t sched_ring = smem_u32(smem + S::SCHED_OFF);  // [kSchedRing] x {t, TileWork}
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::MISC_OFF + 4);
  // k-slices the (even CTA's) producer has issued so far, read by the scheduler thread
  volatile uint32_t* issued_kb = reinterpret_cast<volatile uint32_t*>(smem + S::MISC_OFF + 12);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  volatile int* skip_flag = reinterpret_cast<volatile int*>(smem + S::MISC_OFF + 8);
  // consumers of one published tile: the producer and MMA threads and the epilogue warps of this
  // CTA, plus in a pair the peer's producer thread and epilogue warps (the peer's MMA and
  // scheduler warps are idle)
  constexpr uint32_t kSchedConsumers = PAIR ? 3u + 2u * kEpiWarps : 2u + kEpiWarps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < NACC; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], (PAIR ? 2 : 1) * kEpiWarps);  // one arrival per epilogue warp
    }
    mbar_init(done_bar, 1);
    for (int r = 0; r < kSchedRing; ++r) {
      mbar_init(&sfull_bar[r], 1);
      mbar_init(&sempty_bar[r], kSchedConsumers);
    }
    for (int b = 0; b < 4 * kEpiWarps; ++b) mbar_init(&epi_bars[b], 1);
    uint32_t* acq = reinterpret_cast<uint32_t*>(smem + S::ACQ_OFF);
    for (int i = 0; i < (1 + kEpiWarps) * kAcqWords; ++i) acq[i] = 0u;
    *abort_flag = 0;
    *issued_kb = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  // The launch may overlap the preparation kernel of this call (programmatic stream
  // serialization): the set-up above needs none of its results; what follows does.
  griddep_wait();
  p.on_prep_done();
  // The preparation kernel found invalid device-side arguments: nothing to do.  The CTAs of a
  // pair must agree, so the even CTA's reading decides for both (another pair's timeout may set
  // the word between the two readings).
  if (threadIdx.x == 0 && leader) *skip_flag = *reinterpret_cast<volatile int*>(p.status);
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // barriers of both CTAs initialised before any remote use
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if constexpr (PAIR) {
    const int skip = leader ? *skip_flag : (int)ld_cluster_u32(mapa_shared(smem_u32((const void*)skip_flag), 0));
    if (skip != 0) {
      cluster_sync_all();  // no CTA leaves while its peer may still read its shared memory
      if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
      return;
    }
  } else if (*skip_flag != 0) {
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
    return;
  }
  const WaitGuard wg{abort_flag, p.status};
  const bool dynamic = p.dynamic != 0;
  const long long kEnd = 0x7fffffffffffffffLL;

  // Static schedule: unit u (a CTA, or a pair) takes tiles u, u + units, ...  Dynamic schedule:
  // the next tile comes from the global counter.  Either way the (even CTA's) scheduler thread
  // alone computes each tile's TileWork and publishes {t, TileWork} through the shared-memory
  // ring (into both CTAs of a pair), so the other roles never touch global memory to schedule.
  // The last entry published has t >= total_tiles and ends every role's loop.
  const long long unit = PAIR ? (long long)(blockIdx.x >> 1) : (long long)blockIdx.x;
  const long long units = PAIR ? (long long)(gridDim.x >> 1) : (long long)gridDim.x;
  // Consumers in the odd CTA of a pair release the slot on the even CTA's barrier.
  auto consume_tile = [&](long long n, bool is_warp, TileWork& w) -> long long {
    const int r = (int)(n % kSchedRing);
    const uint32_t ph = (uint32_t)((n / kSchedRing) & 1);
    bool ok;
    // the odd CTA's copy of an entry is written by the even CTA's scheduler (remote stores, then a
    // release at cluster scope): acquire at cluster scope there; the even CTA's own copy is local
    const bool remote_entry = PAIR && !leader;
    if (is_warp) ok = remote_entry ? warp_wait<true>(&sfull_bar[r], ph, wg, 6) : warp_wait<false>(&sfull_bar[r], ph, wg, 6);
    else ok = remote_entry ? mbar_wait_cluster(&sfull_bar[r], ph, wg, 6) : mbar_wait(&sfull_bar[r], ph, wg, 6);
    if (!ok) return kEnd;
    const uint4 e0 = ld_shared_v4(sched_ring + r * kSchedEntry);
    const uint4 e1 = ld_shared_v4(sched_ring + r * kSchedEntry + 16);
    if (is_warp) __syncwarp();
    if (!is_warp || lane == 0) {
      // the odd CTA tells the scheduler it may overwrite this slot: a relaxed arrive whose address
      // depends on both loaded halves of the entry, so it cannot issue before they have returned
      if (PAIR && !leader)
        mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&sempty_bar[r]), 0) + zero_after(e0.x ^ e1.x));
      else mbar_arrive(&sempty_bar[r]);
    }
    w.active = (int)e0.z;
    w.expert = (int)e0.w;
    w.m0 = (int)e1.x;
    w.n0 = (int)e1.y;
    w.k0 = (int)e1.z;
    w.num_kb = (int)e1.w;
    return (long long)(((unsigned long long)e0.y << 32) | e0.x);
  };

  if (warp == 2) {
    // ---------------------------------------------------------------- scheduler (even CTA)
    // Claims tiles (static or from the counter), decodes them and publishes them to every role,
    // so the producer does not wait for a claim's atomic or for the offsets the decode reads.
    // The next tile is claimed once the producer has at most kClaimLeadKb k-slices of the
    // published tiles left to issue.
    if (lane == 0 && leader) {
      int* counter = p.status + 3;
      uint32_t published_kb = 0;  // k-slices of every tile published so far (modulo 2^32)
      for (long long n = 0;; ++n) {
        const int r = (int)(n % kSchedRing);
        const uint32_t eph = (uint32_t)(((n / kSchedRing) & 1) ^ 1);
        if (n >= 1 && !wait_claim_lead(issued_kb, published_kb, wg, 8)) break;
        // in a pair the odd CTA's consumers release the slot remotely: acquire at cluster scope
        if (!(PAIR ? mbar_wait_cluster(&sempty_bar[r], eph, wg, 5) : mbar_wait(&sempty_bar[r], eph, wg, 5))) break;
        long long t = dynamic ? (long long)atomicAdd(counter, 1) : unit + n * units;
        TileWork w;
        if (t >= p.total_tiles) {
          t = p.total_tiles;
          w = TileWork{0, 0, 0, 0, 0, 0};
        } else {
          w = p.tile(t);
        }
        const uint32_t t_lo = (uint32_t)((unsigned long long)t & 0xffffffffu);
        const uint32_t t_hi = (uint32_t)((unsigned long long)t >> 32);
        const uint32_t slot = sched_ring + r * kSchedEntry;
        st_shared_v4(slot, t_lo, t_hi, (uint32_t)w.active, (uint32_t)w.expert);
        st_shared_v4(slot + 16, (uint32_t)w.m0, (uint32_t)w.n0, (uint32_t)w.k0, (uint32_t)w.num_kb);
        if constexpr (PAIR) {  // the odd CTA's copy of the entry, then its "published" barrier
          const uint32_t peer = mapa_shared(slot, 1);
          st_cluster_v4(peer, t_lo, t_hi, (uint32_t)w.active, (uint32_t)w.expert);
          st_cluster_v4(peer + 16, (uint32_t)w.m0, (uint32_t)w.n0, (uint32_t)w.k0, (uint32_t)w.num_kb);
          mbar_arrive_remote(mapa_shared(smem_u32(&sfull_bar[r]), 1));
        }
        mbar_arrive(&sfull_bar[r]);
        if (w.active) published_kb += (uint32_t)w.num_kb;
        if (t >= p.total_tiles) break;
      }
    }
  } else if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      const uint32_t expect = PAIR ? 2u * S::STAGE_BYTES : (uint32_t)S::STAGE_BYTES;
      const MapAcquired acq_producer{reinterpret_cast<uint32_t*>(smem + S::ACQ_OFF)};
      long long n_tile = 0;
      TileWork w;
      for (long long t = consume_tile(n_tile++, false, w); t < p.total_tiles && ok;
           t = consume_tile(n_tile++, false, w)) {
        if (!w.active) continue;
        for (int kb = 0; kb < w.num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, wg, 1)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], expect);
          const uint32_t sa = smem_u32(smem + stage * S::STAGE_BYTES);
          const uint32_t bar = PAIR ? mapa_shared(smem_u32(&full_bar[stage]), 0) : smem_u32(&full_bar[stage]);
          p.issue_loads(w, kb, sa, sa + S::A_BYTES, bar, (int)rank, acq_producer);
          ++issued;
          if (leader) *issued_kb = (uint32_t)issued;  // the scheduler's claim lead
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {  // let the copies already in flight land before the CTA exits
        const long long n_flight = issued < STAGES ? issued : STAGES;
        for (long long i = 1; i <= n_flight; ++i) {
          const long long n = issued - i;
          mbar_wait_drain(&full_bar[n % STAGES], (uint32_t)((n / STAGES) & 1));
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && leader) {
      const uint32_t idesc_full = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, p.a_mn, p.b_mn);
      const uint32_t idesc_half = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN / 2, p.a_mn, p.b_mn);
      const uint32_t a_lbo = p.a_mn ? 8192u : 16u, a_kstep = p.a_mn ? 2048u : 32u;
      const uint32_t b_lbo = p.b_mn ? 8192u : 16u, b_kstep = p.b_mn ? 2048u : 32u;
      int stage = 0;
      uint32_t phase = 0, local = 0;
      bool ok = true;
      long long n_tile = 0;
      TileWork w;
      for (long long t = consume_tile(n_tile++, false, w); t < p.total_tiles && ok;
           t = consume_tile(n_tile++, false, w)) {
        if (!w.active || w.num_kb == 0) continue;
        const uint32_t acc = local % NACC, use = local / NACC;
        if (!mbar_wait(&tempty_bar[acc], (use & 1u) ^ 1u, wg, 2)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const uint32_t idesc = p.narrow(w) ? idesc_half : idesc_full;
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
            if constexpr (PAIR) umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
            else umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          // ring slot free (in both CTAs of a pair) once these MMAs finish
          if constexpr (PAIR) umma_commit_pair_multicast(smem_u32(&empty_bar[stage]), (uint16_t)3);
          else umma_commit(smem_u32(&empty_bar[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        // accumulator complete (in both CTAs' TMEM)
        if constexpr (PAIR) umma_commit_pair_multicast(smem_u32(&tfull_bar[acc]), (uint16_t)3);
        else umma_commit(smem_u32(&tfull_bar[acc]));
        ++local;
      }
      // every MMA of this CTA (pair) retired before TMEM is freed
      if constexpr (PAIR) umma_commit_pair_multicast(smem_u32(done_bar), (uint16_t)1);
      else umma_commit(smem_u32(done_bar));
      mbar_wait_drain(done_bar, 0);
    }
  } else {
    // ---------------------------------------------------------------- epilogue warps (both CTAs)
    const int e = warp - kFirstEpiWarp;     // index among the epilogue warps
    const int q = warp & 3;                 // TMEM sub-partition this warp may access
    const int half = e >> 2;                // which of the sub-partition's warps
    const EpiCtx ctx{q, half, lane, (int)rank, smem + S::EPI_OFF + e * P::STG_BYTES, epi_bars + 4 * e,
                     MapAcquired{reinterpret_cast<uint32_t*>(smem + S::ACQ_OFF) + (1 + e) * kAcqWords}, wg};
    uint32_t local = 0;
    long long n_tile = 0;
    TileWork w;
    for (long long t = consume_tile(n_tile++, true, w); t < p.total_tiles; t = consume_tile(n_tile++, true, w)) {
      if (!w.active) continue;
      p.prologue(w, t, ctx);
      if (w.num_kb == 0) {
        p.epilogue(w, t, 0u, false, ctx, AccRelease{0u, false});
        continue;
      }
      const uint32_t acc = local % NACC, use = local / NACC;
      if (!warp_wait(&tfull_bar[acc], use & 1u, wg, 4)) break;
      tc_fence_after();
      const uint32_t ebar = PAIR ? mapa_shared(smem_u32(&tempty_bar[acc]), 0) : smem_u32(&tempty_bar[acc]);
      p.epilogue(w, t, tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN, true, ctx, AccRelease{ebar, PAIR});
      ++local;
    }
    if (lane == 0) bulk_wait_all();  // bulk stores complete before the CTA exits
    __syncwarp();
  }

  __syncwarp();  // the role branches above split warps 0 and 1; the barriers below are warp-aligned
  griddep_launch_dependents();  // a kernel that reads this one's results may start launching
  tc_fence_before();
  if constexpr (PAIR) cluster_sync_all();  // the pair's MMAs are retired and no peer still signals us
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// Co-resident units (CTAs, or CTA pairs) of one kernel variant, per device ordinal (0 = not yet
// asked): devices of one process may differ in how many clusters they can hold.
struct UnitCache {
  static constexpr int kDevices = 64;
  std::atomic<int> units[kDevices];
  // The cache slot of `device`, or null (ask every time) for an ordinal past the table.
  std::atomic<int>* slot(int device) { return device >= 0 && device < kDevices ? &units[device] : nullptr; }
};

// Launches a persistent kernel: one CTA per SM (single) or one cluster of two CTAs per SM pair,
// never more units than tiles.  `max_units` caches the number of co-resident units of this
// kernel on the current device (0 = not yet known; null = no cache); a pair needs both SMs of a
// cluster slot, so it asks the runtime.
template <class Prm>
inline cudaError_t launch_persistent(void (*kern)(Prm), const Prm& prm, long long total_tiles, int num_sms,
                                     bool pair, int threads, int smem, std::atomic<int>* max_units,
                                     cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  if (pair) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.numAttrs = 1;
  }
  int units = max_units != nullptr ? max_units->load(std::memory_order_relaxed) : 0;
  if (units <= 0) {
    if (pair) {
      cfg.gridDim = dim3(2, 1, 1);
      cudaError_t err = cudaOccupancyMaxActiveClusters(&units, kern, &cfg);
      if (err != cudaSuccess) return err;
      if (units <= 0) return cudaErrorInvalidConfiguration;  // no SM pair can hold the kernel
    } else {
      units = num_sms;
    }
    if (max_units != nullptr) max_units->store(units, std::memory_order_relaxed);
  }
  if (total_tiles < units) units = (int)total_tiles;
  cfg.gridDim = dim3((unsigned)(pair ? 2 * units : units), 1, 1);
  // start while the preparation kernel before it still runs (the kernel waits for its results)
  attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  ++cfg.numAttrs;
  return cudaLaunchKernelEx(&cfg, kern, prm);
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
