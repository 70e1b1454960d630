// Grouped GEMM + dGLU backward ("Grouped GEMM + dGLU (SM100)", BF16 contract):
//
//   R_g = alpha_g^2 * A_g * B_g^T           rows of expert g: [padded_offsets[g-1], padded_offsets[g])
//   X_g = beta_g * C_g                      alternating 32-wide gate / input blocks
//   D_row = interleaved (dgate, dinput)     dSwiGLU or dGeGLU (clamp +-7, filters)
//   dprob[m] += sum_j R[m, j] * act[m, j]   act = unscaled forward activation
//   dbias[g, :] += sum_{m in g} D_row[m, :] (optional)
//
// One persistent kernel computes the GEMM on the tensor cores and applies the whole
// epilogue from TMEM: no intermediate R tensor ever reaches global memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "mgg_internal.h"
#include "mgg_pipeline.cuh"

namespace mgg {

// Per-variant configuration (CS / DS = element bytes of C / D_row; PAIR = CTA-pair tiles).
//  TMA-C (16-bit C): C reaches shared memory by TMA (a 2-box ring of 32 x 64 boxes per epilogue
//            warp, each loaded a chunk ahead of its math); the results go back out of the
//            consumed box (16-bit D in one store; fp32 D as the gate half, then the input half).
//  register-C: C is read per row into registers one chunk ahead.
//  Both use 8 epilogue warps (two per TMEM sub-partition), so each scheduler interleaves two
//  warps' math.  The ring stages take whatever shared memory the epilogue leaves (at most 6): a
//  single CTA loads 48 KB per stage (3 stages next to the TMA-C ring), a CTA of a pair 32 KB
//  (5 stages); a single CTA takes the TMA-C path when K <= kTmaCMaxK.

// EPI: epilogue warps, 8 (two per TMEM sub-partition, each taking every other chunk) or 4.  Four
// leave room for one more operand stage, which pays where the epilogue's per-element work is
// light (dSwiGLU, dSiTU-GLU or dsReLU with 16-bit D_row); the dGeGLU math and fp32 D_row need 8.
template <int CS, int DS, bool TMAC, bool PAIR, int EPI = 8>
struct DgluCfg {
  static_assert(EPI == 4 || EPI == 8, "one or two epilogue warps per TMEM sub-partition");
  static constexpr bool kTmaC = TMAC && CS == 2;
  static constexpr int kEpiWarps = EPI;
  // C boxes per warp (TMA path).  Three boxes would let a refill wait for stores a use older, but
  // cost a pair one of its five operand stages, which measured 5-10% slower on every shape.
  static constexpr int kCRing = 2;
  // bulk groups one use commits on the TMA path: 16-bit D leaves in one store, fp32 D in two
  // (always both: a dsReLU use that ends at N after its first half commits an empty second group)
  static constexpr int kGroups = DS == 4 ? 2 : 1;
  // TMA path: the C ring (results leave through the consumed box); register path: D staging
  static constexpr int kStgBytes = kTmaC ? kCRing * 4096 : (DS == 4 ? 8192 : 4096);
  static constexpr int kStages = max_stages(PAIR ? kDgluTileN / 2 : kDgluTileN, kEpiWarps, kStgBytes,
                                            num_acc(kDgluTileN), 6);
  static_assert(kStages >= 3, "operand ring too shallow");
  static_assert(kCRing == 2, "the C-ring waits are written for any depth, measured and tested at 2");
};

struct DgluParams {
  CUtensorMap tmap_a;           // A (M, K): dims {K, M}, box {64, 128}, 128B swizzle
  CUtensorMap tmap_b;           // dense B (N, K, L): dims {K, N, L}, box {64, BN, 1}
  CUtensorMap tmap_d;           // D_row (M, 2N): dims {2N, M}, box {128 B of columns, 32}, 128B swizzle
  CUtensorMap tmap_c;           // 16-bit C (M, 2N): dims {2N, M}, box {64, 32}, 128B swizzle
  CUtensorMap tmap_dcol;        // optional D_col, same geometry as tmap_d (has_dcol)
  const CUtensorMap* b_maps;    // discrete B: one map per expert in the workspace, else null
  const int32_t* offsets;
  const float* alpha;
  const float* beta;
  const float* prob;
  const void* c;
  float* dprob;
  float* dbias_ws;              // fp32 partial sums (L, 2N), null = no dbias
  float* amax;                  // per-expert |D| maxima ((L, 2) dGLU, (L) dsReLU), zeroed by the prep kernel; or null
  int has_dcol;                 // 1: every D_row box is also stored through tmap_dcol
  int* status;
  int32_t* tile_log;
  long long tile_log_cap;
  long long total_tiles;
  int dynamic;                  // 1: tiles claimed from the workspace counter
  int M, K, N, L;               // dsReLU: N = columns of C / D_row (dGLU: 2N of them)
  int num_n, num_kb;
  int a_mn, b_mn;
  int b_blocked;                // discrete N-major B maps are 3-D (64-column blocks, one box per slot)
  int c_dtype, d_dtype, act, indicator, gate_first;
  float situ_b1, situ_b2, situ_inv_b1, situ_inv_b2;  // dSiTU-GLU scales and their reciprocals
};

// Byte offset of 16-byte chunk `c16` of row `r` in a 128B-swizzled staging box (rows of 128 B).
__device__ __forceinline__ uint32_t swz128(int r, int c16) { return (uint32_t)(r * 128 + ((c16 ^ (r & 7)) << 4)); }

// The epilogue a launch runs on the grouped GEMM result: the dGLU page's (gate/input blocks of C
// and D_row, R = alpha^2 acc) or the dsReLU page's (plain C and D_row of N columns, G = alpha acc).
constexpr int kOpGlu = 0;
constexpr int kOpSrelu = 1;

// CS / DS: element size in bytes of C and D_row (2 = bf16/fp16, 4 = fp32).
template <int BN, int CS, int DS, bool TMAC, bool PAIR, int OP, int EPI>
struct DgluPolicy {
  using Cfg = DgluCfg<CS, DS, TMAC, PAIR, EPI>;
  static constexpr int kTileM = PAIR ? 2 * BM : BM;   // rows of a tile (a pair's tile spans both CTAs)
  static constexpr int kBLoad = PAIR ? BN / 2 : BN;   // B rows this CTA loads
  static constexpr int EPI_WARPS = Cfg::kEpiWarps;
  static constexpr int STG_BYTES = Cfg::kStgBytes;
  static constexpr int kEpiHalves = EPI_WARPS / 4;
  static constexpr int kCRing = Cfg::kCRing;
  static constexpr int CV = 32 * CS / 16;  // 16-byte vectors per 32 elements of C
  const DgluParams& p;
  long long total_tiles;
  int* status;
  int a_mn, b_mn;
  int dynamic;
  mutable uint32_t c_uses = 0;  // TMA path: C boxes this warp has consumed (ring position)
  // The scheduler thread's decode cache: the expert found last and its row range, so consecutive
  // tiles of one expert skip the binary search over the offsets (dependent global loads).
  mutable int c_g = -1, c_begin = 0, c_end = 0;

  __device__ DgluPolicy(const DgluParams& prm)
      : p(prm), total_tiles(prm.total_tiles), status(prm.status), a_mn(0), b_mn(prm.b_mn), dynamic(prm.dynamic) {}

  // Nothing of the preparation kernel's output is cached in the policy.
  __device__ void on_prep_done() {}

  // Tile order: expert-major (tile t belongs to the expert containing row floor(t / num_n) *
  // kTileM; its tiles occupy [begin/kTileM * num_n, end/kTileM * num_n)).  Inside an expert the
  // operand that is re-read across the expert's tiles stays in L2 while the other one streams
  // through once: an expert with at most N rows (A_g no larger than B_g) runs column panel by
  // column panel, each panel over all of the expert's row blocks (A_g re-read per panel from L2,
  // each B panel read once); an expert with more rows runs row block by row block, each over all
  // column panels (B_g re-read per row block from L2, each block of A rows read once).  (Panel
  // order for a DeepSeek-shaped expert of 21248 rows re-read its 304 MB of A rows from DRAM for
  // every one of its 8 panels.)
  __device__ TileWork tile(long long t) const {
    const int row = (int)(t / p.num_n) * kTileM;
    if (c_g < 0 || row < c_begin || row >= c_end) {
      int lo = 0, hi = p.L - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.offsets + mid) > row) hi = mid;
        else lo = mid + 1;
      }
      c_g = lo;
      c_begin = lo ? __ldg(p.offsets + lo - 1) : 0;
      c_end = __ldg(p.offsets + lo);
    }
    const int g = c_g;
    const int begin = c_begin;
    const int mblocks = (c_end - begin) / kTileM;
    const long long u = t - (long long)(begin / kTileM) * p.num_n;
    TileWork w;
    w.active = 1;
    w.expert = g;
    if (c_end - begin <= p.N) {  // panel by panel
      w.n0 = (int)(u / mblocks) * BN;
      w.m0 = begin + (int)(u % mblocks) * kTileM;
    } else {  // row block by row block
      w.n0 = (int)(u % p.num_n) * BN;
      w.m0 = begin + (int)(u / p.num_n) * kTileM;
    }
    w.k0 = 0;
    w.num_kb = p.num_kb;
    // checked build: a tile outside the call's extents is skipped by every role
    if (!(MGG_IN_BOUNDS(p.status, g >= 0 && g < p.L, 401, g) &&
          MGG_IN_BOUNDS(p.status, w.m0 >= begin && w.m0 + kTileM <= p.M, 402, w.m0) &&
          MGG_IN_BOUNDS(p.status, w.n0 >= 0 && w.n0 < p.N, 403, w.n0)))
      w.active = 0;
    return w;
  }

  static __device__ __forceinline__ void load2(uint32_t dst, const void* map, uint32_t bar, int x, int y) {
    if constexpr (PAIR) tma_load_2d_pair(dst, map, bar, x, y);
    else tma_load_2d(dst, map, bar, x, y);
  }

  // This CTA's rows of A (m0 + 128 * rank) and its kBLoad columns of B (n0 + kBLoad * rank).
  __device__ void issue_loads(const TileWork& w, int kb, uint32_t sa, uint32_t sb, uint32_t bar, int rank,
                              const MapAcquired& acq) const {
    const int mrow = w.m0 + rank * BM;
    const int ncol = w.n0 + rank * kBLoad;
    load2(sa, &p.tmap_a, bar, kb * BK, mrow);
    if (p.b_maps == nullptr) {
      if constexpr (PAIR) tma_load_3d_pair(sb, &p.tmap_b, bar, kb * BK, ncol, w.expert);
      else tma_load_3d(sb, &p.tmap_b, bar, kb * BK, ncol, w.expert);
    } else {
      const int e = MGG_IN_BOUNDS(p.status, w.expert < p.L, 301, w.expert) ? w.expert : 0;
      const CUtensorMap* m = p.b_maps + e;
      if (kb == 0 && acq.first_use(e)) tmap_acquire(m);
      if (!p.b_mn) {
        load2(sb, m, bar, kb * BK, ncol);
      } else if (p.b_blocked) {
        if constexpr (PAIR) tma_load_3d_pair(sb, m, bar, 0, kb * BK, ncol / 64);
        else tma_load_3d(sb, m, bar, 0, kb * BK, ncol / 64);
      } else {
#pragma unroll
        for (int j = 0; j < kBLoad / 64; ++j) load2(sb + j * 8192, m, bar, ncol + 64 * j, kb * BK);
      }
    }
  }

  // Raw C of one row for compact columns [j0, j0 + 32): the gate block and the input block.
  __device__ __forceinline__ void load_c(size_t row_off, int j0, uint4 (&g)[CV], uint4 (&in)[CV]) const {
    const int first = 2 * j0, second = 2 * j0 + 32;
    const int gcol = p.gate_first ? first : second;
    const int icol = p.gate_first ? second : first;
    const uint4* pg = reinterpret_cast<const uint4*>(static_cast<const char*>(p.c) + (row_off + gcol) * CS);
    const uint4* pi = reinterpret_cast<const uint4*>(static_cast<const char*>(p.c) + (row_off + icol) * CS);
#pragma unroll
    for (int i = 0; i < CV; ++i) {
      g[i] = __ldg(pg + i);
      in[i] = __ldg(pi + i);
    }
  }

  __device__ __forceinline__ void unpack_c(const uint4 (&raw)[CV], float (&v)[32]) const {
    if constexpr (CS == 4) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[4 * i + 0] = __uint_as_float(raw[i].x);
        v[4 * i + 1] = __uint_as_float(raw[i].y);
        v[4 * i + 2] = __uint_as_float(raw[i].z);
        v[4 * i + 3] = __uint_as_float(raw[i].w);
      }
    } else {
      const bool bf = p.c_dtype == MGG_BF16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (bf) {
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

  // Writes 32 values of this lane's row into the staging box: 16-bit D uses one box of 64
  // columns (block `blk` = chunks 4*blk .. 4*blk+3), fp32 D one box of 32 columns.
  __device__ __forceinline__ void stage_block(uint32_t stg, int lane, int blk, const float (&v)[32]) const {
    if constexpr (DS == 4) {
      (void)blk;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        st_shared_v4(stg + swz128(lane, i), __float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                     __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3]));
    } else {
      const int dt = p.d_dtype;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        st_shared_v4(stg + swz128(lane, 4 * blk + i), pack2(v[8 * i], v[8 * i + 1], dt),
                     pack2(v[8 * i + 2], v[8 * i + 3], dt), pack2(v[8 * i + 4], v[8 * i + 5], dt),
                     pack2(v[8 * i + 6], v[8 * i + 7], dt));
    }
  }

  // The staging box must no longer be read by an earlier bulk store before it is rewritten.
  __device__ __forceinline__ void staging_free(int lane) const {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
  }

  // Bulk store of one staged box to D_row (and to D_col when requested); lane 0 of the warp.
  // D_row (and D_col) are written once: streamed out of L2 ahead of the reused A / B lines.
  __device__ __forceinline__ void store_box(uint32_t stg, int x, int y) const {
    tma_store_2d_evict_first(&p.tmap_d, stg, x, y);
    if (p.has_dcol) tma_store_2d_evict_first(&p.tmap_dcol, stg, x, y);
  }

  __device__ __forceinline__ void staging_flush(uint32_t stg, int lane, int x, int y) const {
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
      store_box(stg, x, y);
      bulk_commit_group();
    }
  }

  // Largest |v| of 32 values, folded into a running maximum.
  static __device__ __forceinline__ float absmax32(const float (&v)[32], float m) {
#pragma unroll
    for (int k = 0; k < 32; ++k) m = fmaxf(m, fabsf(v[k]));
    return m;
  }

  // The warp's running |D| maxima of one tile into the expert's amax (non-negative floats order
  // like their bit patterns as signed integers).
  __device__ __forceinline__ void amax_flush(int g, int slot, float m) const {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if ((threadIdx.x & 31) == 0 && m > 0.f &&
        MGG_IN_BOUNDS(p.status, slot >= 0 && slot < (OP == kOpGlu ? 2 : 1) * p.L, 104, slot))
      atomicMax(reinterpret_cast<int*>(p.amax) + slot, __float_as_int(m));
    (void)g;
  }

  // dGLU math on 32 columns of one row.  On entry gv / iv hold the C values of the gate and the
  // input block, on exit dgate / dinput; returns this row's partial of sum_j R * act.
  // One activation over a 32-column chunk; the activation is fixed per launch, so the branch is
  // taken once per chunk and only that activation's unrolled loop runs.
  // sigmoid of two values: 1/2 + tanh(x/2)/2, one SFU tanh.approx each (relative error about
  // 2^-11, far inside the fp32 / bf16 tolerances of the results it feeds).
  static __device__ __forceinline__ float2 sigmoid2(float2 x) {
    const float2 h = __fmul2_rn(x, make_float2(0.5f, 0.5f));
    return __ffma2_rn(make_float2(tanh_approx(h.x), tanh_approx(h.y)), make_float2(0.5f, 0.5f), make_float2(0.5f, 0.5f));
  }

  // dSiTU-GLU on element pairs with the packed fp32 instructions, like dSwiGLU / dGeGLU below:
  //   s = sigmoid(x_g), tg = tanh(x_g / b1), tu = tanh(x_i / b2), Tg = b1 tg s, Tu = b2 tu,
  //   dTg = (1 - tg^2) s + Tg (1 - s), dTu = 1 - tu^2,
  //   dgate = R p Tu dTg, dinput = R p Tg dTu, dprob += R Tg Tu,
  // with tanh on the SFU (tanh.approx) and the sigmoid as below.
  template <int NV>
  __device__ __forceinline__ float dsitu_math(const uint32_t* r, float* gv, float* iv, float alpha2, float beta_g,
                                              float pr) const {
    static_assert(NV % 2 == 0, "pairs of elements");
    const float2 one2 = make_float2(1.0f, 1.0f);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    const float2 b2 = make_float2(beta_g, beta_g);
    const float ap = alpha2 * pr;
    const float2 ap2 = make_float2(ap, ap);
    const float2 kg2 = make_float2(p.situ_inv_b1, p.situ_inv_b1), ku2 = make_float2(p.situ_inv_b2, p.situ_inv_b2);
    const float2 sb1 = make_float2(p.situ_b1, p.situ_b1), sb2 = make_float2(p.situ_b2, p.situ_b2);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NV; k += 2) {
      const float2 acc_v = make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1]));
      const float2 xg = __fmul2_rn(b2, make_float2(gv[k], gv[k + 1]));  // one fp32 product each
      const float2 xi = __fmul2_rn(b2, make_float2(iv[k], iv[k + 1]));
      const float2 Rp = __fmul2_rn(acc_v, ap2);
      const float2 s = sigmoid2(xg);
      const float2 zg = __fmul2_rn(xg, kg2);
      const float2 tg = make_float2(tanh_approx(zg.x), tanh_approx(zg.y));
      const float2 zu = __fmul2_rn(xi, ku2);
      const float2 tu = make_float2(tanh_approx(zu.x), tanh_approx(zu.y));
      const float2 Tg = __fmul2_rn(sb1, __fmul2_rn(tg, s));
      const float2 Tu = __fmul2_rn(sb2, tu);
      const float2 oms = __ffma2_rn(s, neg1, one2);                                   // 1 - s
      const float2 omg = __ffma2_rn(__fmul2_rn(tg, tg), neg1, one2);                  // 1 - tg^2
      const float2 dTg = __ffma2_rn(Tg, oms, __fmul2_rn(omg, s));
      const float2 dTu = __ffma2_rn(__fmul2_rn(tu, tu), neg1, one2);                  // 1 - tu^2
      const float2 dg = __fmul2_rn(__fmul2_rn(Rp, Tu), dTg);
      const float2 di = __fmul2_rn(__fmul2_rn(Rp, Tg), dTu);
      acc = __ffma2_rn(acc_v, __fmul2_rn(Tg, Tu), acc);
      gv[k] = dg.x;
      gv[k + 1] = dg.y;
      iv[k] = di.x;
      iv[k + 1] = di.y;
    }
    return alpha2 * (acc.x + acc.y);
  }

  // dSwiGLU / dGeGLU on element pairs with the packed fp32 instructions (add/mul/fma.f32x2): the
  // epilogue is bound by instruction latency and issue, and each packed instruction does two
  // lanes' worth.  Every product and sum is one IEEE round-to-nearest fp32 operation per element;
  // the dSwiGLU sigmoid is 1/2 + tanh(z/2)/2 (one SFU tanh.approx each), the dGeGLU one
  // 1 / (1 + 2^(-z log2 e)) (SFU ex2 and rcp).  x_g and x_i stay single products
  // (the clamp and filter decisions are taken on them in fp32).  R p = acc (alpha^2 p) and the
  // dprob sum is alpha^2 sum acc * act, the factor applied once at the end.
  template <int ACT, int NV, bool IND = false>
  __device__ __forceinline__ float dglu_math_act(const uint32_t* r, float* gv, float* iv, float alpha2, float beta_g,
                                                 float pr) const {
    static_assert(NV % 2 == 0, "pairs of elements");
    const float2 one2 = make_float2(1.0f, 1.0f);
    const float2 b2 = make_float2(beta_g, beta_g);
    const float ap = alpha2 * pr;
    const float2 ap2 = make_float2(ap, ap);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NV; k += 2) {
      const float2 acc_v = make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1]));
      const float2 xg = __fmul2_rn(b2, make_float2(gv[k], gv[k + 1]));
      const float2 xi = __fmul2_rn(b2, make_float2(iv[k], iv[k + 1]));
      const float2 Rp = __fmul2_rn(acc_v, ap2);
      float2 dg, di, act;
      if constexpr (ACT == MGG_ACT_DSWIGLU) {
        const float2 s = sigmoid2(xg);
        const float2 xs = __fmul2_rn(xg, s);                                        // x_g s
        const float2 oms = __ffma2_rn(s, make_float2(-1.0f, -1.0f), one2);          // 1 - s
        const float2 inner = __ffma2_rn(xg, oms, one2);                             // 1 + x_g (1 - s)
        di = __fmul2_rn(Rp, xs);
        dg = __fmul2_rn(__fmul2_rn(Rp, __fmul2_rn(xi, s)), inner);
        act = __fmul2_rn(xs, xi);
      } else {
        static_assert(ACT == MGG_ACT_DGEGLU, "dSiTU-GLU has its own path");
        const float2 cgt = make_float2(fminf(xg.x, 7.0f), fminf(xg.y, 7.0f));
        const float2 cit = make_float2(fminf(fmaxf(xi.x, -7.0f), 7.0f), fminf(fmaxf(xi.y, -7.0f), 7.0f));
        // filters: the indicator (1 inside the clamp range) or the value itself (IND = false)
        const float2 gf = make_float2(xg.x <= 7.0f ? (IND ? 1.0f : xg.x) : 0.0f,
                                      xg.y <= 7.0f ? (IND ? 1.0f : xg.y) : 0.0f);
        const float2 inf_ = make_float2(fabsf(xi.x) <= 7.0f ? (IND ? 1.0f : xi.x) : 0.0f,
                                        fabsf(xi.y) <= 7.0f ? (IND ? 1.0f : xi.y) : 0.0f);
        constexpr float kA = 1.702f;
        // sigmoid(1.702 cgt) as 1 / (1 + 2^(-1.702 cgt log2 e)) on the SFU's ex2 / rcp: measured 1.5%
        // faster than the tanh form on the fp32-D dGeGLU layer, whose epilogue this path bounds
        constexpr float kLog2e = 1.4426950408889634f;
        const float2 z = __fmul2_rn(cgt, make_float2(-kA * kLog2e, -kA * kLog2e));
        const float2 den = __fadd2_rn(make_float2(ex2_approx(z.x), ex2_approx(z.y)), one2);
        const float2 s = make_float2(rcp_approx(den.x), rcp_approx(den.y));
        const float2 ci1 = __fadd2_rn(cit, one2);
        const float2 aoms = __ffma2_rn(s, make_float2(-kA, -kA), make_float2(kA, kA));  // 1.702 (1 - s)
        const float2 inner = __ffma2_rn(cgt, aoms, one2);                               // 1 + 1.702 cgt (1 - s)
        const float2 gs = __fmul2_rn(cgt, s);
        dg = __fmul2_rn(__fmul2_rn(__fmul2_rn(Rp, __fmul2_rn(ci1, s)), inner), gf);
        di = __fmul2_rn(__fmul2_rn(Rp, gs), inf_);
        act = __fmul2_rn(gs, ci1);
      }
      acc = __ffma2_rn(acc_v, act, acc);
      gv[k] = dg.x;
      gv[k + 1] = dg.y;
      iv[k] = di.x;
      iv[k + 1] = di.y;
    }
    return alpha2 * (acc.x + acc.y);
  }

  // NV values per call: r points at the NV accumulator words, gv / iv at NV gate / input values.
  template <int NV>
  __device__ __forceinline__ float dglu_math(const uint32_t* r, float* gv, float* iv, float alpha2, float beta_g,
                                             float pr) const {
    if (p.act == MGG_ACT_DSWIGLU) return dglu_math_act<MGG_ACT_DSWIGLU, NV>(r, gv, iv, alpha2, beta_g, pr);
    if (p.act == MGG_ACT_DSITUGLU) return dsitu_math<NV>(r, gv, iv, alpha2, beta_g, pr);
    if (p.indicator) return dglu_math_act<MGG_ACT_DGEGLU, NV, true>(r, gv, iv, alpha2, beta_g, pr);
    return dglu_math_act<MGG_ACT_DGEGLU, NV, false>(r, gv, iv, alpha2, beta_g, pr);
  }

  __device__ __forceinline__ void dbias_partials(const TileWork& w, int j0, int lane, float (&gv)[32],
                                                 float (&iv)[32]) const {
    const float sg = warp_column_sums(gv, lane), si = warp_column_sums(iv, lane);
    if (dbias_in_range(w, 2 * j0) && dbias_in_range(w, 2 * j0 + 32)) dbias_add(w, j0, lane, sg, si);
  }

  // Adds the column totals of a staged 32 x 32 fp32 box (128B-swizzled rows, as stage_block writes
  // them) into the 32 consecutive fp32 partials at ws.  Lane l reads 16-byte column group l & 7 of
  // rows 8 (l >> 3) .. 8 (l >> 3) + 7 (the eight lanes of a quarter-warp hit all 32 banks once),
  // two shuffle rounds add the four row quarters, and lanes 0..7 add their four columns with one
  // 16-byte reduction.
  static __device__ __forceinline__ void box_dbias_add(uint32_t box, int lane, float* ws) {
    const int cg = lane & 7, rq = lane >> 3;
    float2 s01 = make_float2(0.f, 0.f), s23 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 v = ld_shared_v4(box + swz128(rq * 8 + i, cg));
      s01 = __fadd2_rn(s01, make_float2(__uint_as_float(v.x), __uint_as_float(v.y)));
      s23 = __fadd2_rn(s23, make_float2(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
#pragma unroll
    for (int off = 8; off <= 16; off <<= 1) {
      s01 = __fadd2_rn(s01, make_float2(__shfl_xor_sync(0xffffffffu, s01.x, off),
                                        __shfl_xor_sync(0xffffffffu, s01.y, off)));
      s23 = __fadd2_rn(s23, make_float2(__shfl_xor_sync(0xffffffffu, s23.x, off),
                                        __shfl_xor_sync(0xffffffffu, s23.y, off)));
    }
    if (lane < 8) {
      const float v4[4] = {s01.x, s01.y, s23.x, s23.y};
      red_add_v4(ws + 4 * cg, v4);
    }
  }

  // The expert's fp32 dbias partials for the gate (second = 0) or input (second = 1) block of
  // compact chunk j0.
  __device__ __forceinline__ float* dbias_ws_at(const TileWork& w, int j0, int second) const {
    const int first_half = (p.gate_first != 0) == (second == 0) ? 0 : 32;
    return p.dbias_ws + (size_t)w.expert * 2 * (size_t)p.N + 2 * j0 + first_half;
  }

  // Checked build: the 32 fp32 dbias partials at column `col` of expert w.expert exist.
  __device__ __forceinline__ bool dbias_in_range(const TileWork& w, int col) const {
    return MGG_IN_BOUNDS(p.status, w.expert < p.L && col >= 0 && col + 32 <= 2 * p.N, 103, col);
  }

  // Adds this warp's column totals (lane l: gate column l in sg, input column l in si) of compact
  // chunk j0 into the expert's fp32 partials.
  __device__ __forceinline__ void dbias_add(const TileWork& w, int j0, int lane, float sg, float si) const {
    const int first = 2 * j0, second = 2 * j0 + 32;
    const int gcol = p.gate_first ? first : second;
    const int icol = p.gate_first ? second : first;
    float* ws = p.dbias_ws + (size_t)w.expert * 2 * (size_t)p.N;
    // lanes 4i gather columns 4i..4i+3 and add them with one 16-byte reduction (4x fewer atomics
    // on addresses that every CTA of the same expert and column panel updates)
    float g4[4], i4[4];
    g4[0] = sg;
    i4[0] = si;
#pragma unroll
    for (int d = 1; d < 4; ++d) {
      g4[d] = __shfl_down_sync(0xffffffffu, sg, d);
      i4[d] = __shfl_down_sync(0xffffffffu, si, d);
    }
    if ((lane & 3) == 0) {
      red_add_v4(ws + gcol + lane, g4);
      red_add_v4(ws + icol + lane, i4);
    }
  }

  // One entry per CTA tile of 128 rows (a pair's tile logs two).
  __device__ __forceinline__ void log_tile(const TileWork& w, long long t, int rank) const {
    const long long idx = PAIR ? 2 * t + rank : t;
    if (p.tile_log != nullptr && idx < p.tile_log_cap) {
      int32_t* e = p.tile_log + 4 * idx;
      e[0] = w.expert;
      e[1] = w.m0 + rank * BM;
      e[2] = w.n0;
      e[3] = (int32_t)blockIdx.x;
    }
  }

  // Epilogue uses of a tile: each covers a 32-row x 64-column box of C and D_row per warp.  A dGLU
  // use is 32 accumulator columns (gate and input block); a dsReLU use 64 accumulator columns
  // (rounded up: past N the accumulator and the C box hold zeros).
  __device__ __forceinline__ int num_chunks(const TileWork& w) const {
    const int cols = p.N - w.n0 < BN ? p.N - w.n0 : BN;
    return OP == kOpGlu ? cols / 32 : (cols + 63) / 64;
  }

  // First column of C / D_row of use c of tile w.
  __device__ __forceinline__ int use_col(const TileWork& w, int c) const {
    return OP == kOpGlu ? 2 * (w.n0 + 32 * c) : w.n0 + 64 * c;
  }

  // Chunks of this warp: half, half + kEpiHalves, ...
  __device__ __forceinline__ int own_chunks(int nchunks, int half) const {
    return nchunks > half ? (nchunks - half + kEpiHalves - 1) / kEpiHalves : 0;
  }

  // ---------------------------------------------------------------- TMA path for 16-bit C
  // Ring of kCRing 4 KB boxes per warp: box u % kCRing holds rows [row0, row0+32) x C columns
  // [2*j0, 2*j0+64) (the gate and the input block of compact chunk j0).  Use u + 2 is loaded when
  // use u is done; the results overwrite the consumed box and leave by bulk stores (16-bit D in
  // one group, fp32 D as two halves in two), so a box is reloaded only once those stores have
  // read it: with 2 boxes that is the use just finished, with 3 the one before it.
  __device__ __forceinline__ void c_issue(const EpiCtx& ctx, uint32_t use, int x, int row0) const {
    const uint32_t b = use % kCRing;
    mbar_arrive_expect_tx(&ctx.bars[b], 4096);
    // C is read once: evict-first keeps the reused A / B lines in L2
    tma_load_2d_evict_first(smem_u32(ctx.stg) + b * 4096, &p.tmap_c, smem_u32(&ctx.bars[b]), x, row0);
  }

  __device__ __forceinline__ void read_c_block(uint32_t box, int lane, int blk, float (&v)[32]) const {
    const bool bf = p.c_dtype == MGG_BF16;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 x = ld_shared_v4(box + swz128(lane, 4 * blk + i));
      const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (bf) {
          v[8 * i + 2 * j + 0] = bf16_bits_to_float(wv[j] & 0xffffu);
          v[8 * i + 2 * j + 1] = bf16_bits_to_float(wv[j] >> 16);
        } else {
          v[8 * i + 2 * j + 0] = __half2float(__ushort_as_half((unsigned short)(wv[j] & 0xffffu)));
          v[8 * i + 2 * j + 1] = __half2float(__ushort_as_half((unsigned short)(wv[j] >> 16)));
        }
      }
    }
  }

  // Every dgrad tile runs full-width MMAs.
  __device__ __forceinline__ bool narrow(const TileWork&) const { return false; }

  __device__ void prologue(const TileWork& w, long long, const EpiCtx& ctx) const {
    if constexpr (Cfg::kTmaC) {
      if (*ctx.wg.abort_flag) return;  // the CTA is stopping: start no copies that nobody would wait for
      const int nown = own_chunks(num_chunks(w), ctx.half);
      const int row0 = w.m0 + ctx.rank * BM + 32 * ctx.q;
      fence_async_shared();  // earlier generic reads of the ring before the async overwrite
      __syncwarp();
      if (ctx.lane == 0 && nown > 0) {
        // every store out of the ring has read its box (the tile's accumulator is still being
        // computed, so this wait costs nothing on the critical path)
        bulk_wait_read<0>();
        c_issue(ctx, c_uses, use_col(w, ctx.half), row0);
        if (nown > 1) {
          c_issue(ctx, c_uses + 1, use_col(w, ctx.half + kEpiHalves), row0);
        }
      }
      __syncwarp();
    }
  }

  __device__ void epilogue_tmac(const TileWork& w, long long t, uint32_t taddr, const EpiCtx& ctx,
                                AccRelease rel) const {
    const int lane = ctx.lane, half = ctx.half;
    const int g = MGG_IN_BOUNDS(p.status, w.expert < p.L, 101, w.expert) ? w.expert : 0;
    const float alpha_g = __ldg(p.alpha + g);
    const float alpha2 = alpha_g * alpha_g;
    const float beta_g = OP == kOpGlu ? __ldg(p.beta + g) : 1.0f;
    const int row0 = w.m0 + ctx.rank * BM + ctx.q * 32;
    const int row = row0 + lane;
    const bool row_ok = MGG_IN_BOUNDS(p.status, row < p.M, 102, row);
    const float pr = row_ok ? __ldg(p.prob + row) : 0.0f;
    const int nown = own_chunks(num_chunks(w), half);
    const uint32_t ring = smem_u32(ctx.stg);
    const int gblk = p.gate_first ? 0 : 1;
    const bool want_amax = p.amax != nullptr;
    float dprob_acc = 0.f;
    float amx0 = 0.f, amx1 = 0.f;  // running |D| maxima (dGLU: gate, input; dsReLU: amx0)
    bool released = false;
#pragma unroll 1
    for (int i = 0; i < nown; ++i) {
      const int c = half + i * kEpiHalves;
      const uint32_t u = c_uses + i;
      const uint32_t box = ring + (u % kCRing) * 4096;
      const int x = use_col(w, c);  // first C / D_row column of this use
      uint32_t r[32];
      const int tcol = (OP == kOpGlu ? 32 : 64) * c;  // this use's first accumulator column
      tmem_load_32cols(taddr + (MGG_IN_BOUNDS(p.status, tcol + (OP == kOpGlu ? 32 : 64) <= BN, 105, tcol) ? tcol : 0), r);
      if (OP == kOpGlu && i == nown - 1) {
        rel(lane);
        released = true;
      }
      if (!warp_wait(&ctx.bars[u % kCRing], (u / kCRing) & 1u, ctx.wg, 7)) {
        // stopping: let this warp's C copies still in flight (uses u and u + 1) land first
        if (lane == 0)
          for (uint32_t v = u; v < c_uses + (uint32_t)nown && v < u + 2; ++v)
            mbar_wait_drain(&ctx.bars[v % kCRing], (v / kCRing) & 1u);
        __syncwarp();
        break;
      }
      if constexpr (OP == kOpGlu) {
        const int j0 = w.n0 + c * 32;
        float gv[32], iv[32];
        read_c_block(box, lane, gblk, gv);
        read_c_block(box, lane, 1 - gblk, iv);
        dprob_acc += dglu_math<32>(r, gv, iv, alpha2, beta_g, pr);
        if (want_amax) {
          amx0 = absmax32(gv, amx0);
          amx1 = absmax32(iv, amx1);
        }
        if constexpr (DS == 2) {  // D_row written back over this lane's own row of the C box
          stage_block(box, lane, gblk, gv);
          stage_block(box, lane, 1 - gblk, iv);
          staging_flush(box, lane, x, row0);
        } else {  // fp32: the gate half, then the input half, each a 32 x 32 box through the C box
          const bool db = p.dbias_ws != nullptr;
          stage_block(box, lane, 0, gv);
          staging_flush(box, lane, p.gate_first ? x : x + 32, row0);
          // dbias column totals straight from the staged fp32 values (the exact D_row values)
          if (db && dbias_in_range(w, 2 * j0)) box_dbias_add(box, lane, dbias_ws_at(w, j0, 0));
          if (lane == 0) bulk_wait_read<0>();  // the gate half has left the box
          __syncwarp();
          stage_block(box, lane, 0, iv);
          staging_flush(box, lane, p.gate_first ? x + 32 : x, row0);
          if (db && dbias_in_range(w, 2 * j0 + 32)) box_dbias_add(box, lane, dbias_ws_at(w, j0, 1));
        }
        if (DS == 2 && p.dbias_ws != nullptr) dbias_partials(w, j0, lane, gv, iv);
      } else {
        // dsReLU on the box's two 32-column blocks: G = alpha acc, D = prob 2 C relu(G),
        // dprob += C relu(G)^2.  Both blocks of C are read before any result is staged (fp32
        // results fill the whole box).
        float c0[32], c1[32];
        read_c_block(box, lane, 0, c0);
        read_c_block(box, lane, 1, c1);
        const float p2 = 2.0f * pr;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float rr = fmaxf(alpha_g * __uint_as_float(r[k]), 0.0f);
          dprob_acc += c0[k] * rr * rr;
          c0[k] = p2 * c0[k] * rr;
        }
        tmem_load_32cols(taddr + 64 * c + 32, r);
        if (i == nown - 1) {
          rel(lane);
          released = true;
        }
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float rr = fmaxf(alpha_g * __uint_as_float(r[k]), 0.0f);
          dprob_acc += c1[k] * rr * rr;
          c1[k] = p2 * c1[k] * rr;
        }
        if (want_amax) amx0 = absmax32(c1, absmax32(c0, amx0));
        if constexpr (DS == 2) {
          stage_block(box, lane, 0, c0);
          stage_block(box, lane, 1, c1);
          staging_flush(box, lane, x, row0);
        } else {
          stage_block(box, lane, 0, c0);
          staging_flush(box, lane, x, row0);
          if (x + 32 < p.N) {  // a use may end at N after its first half
            if (lane == 0) bulk_wait_read<0>();  // the first half has left the box
            __syncwarp();
            stage_block(box, lane, 0, c1);
            staging_flush(box, lane, x + 32, row0);
          } else if (lane == 0) {
            bulk_commit_group();  // an empty group keeps kGroups groups per use
          }
        }
      }
      if (i + 2 < nown) {  // refill with this warp's use u + 2 the box last used kCRing - 2 uses ago
        __syncwarp();
        if (lane == 0) {
          // the stores out of that box have read it (at most the later uses' groups still read)
          bulk_wait_read<(kCRing - 2) * Cfg::kGroups>();
          c_issue(ctx, u + 2, use_col(w, c + 2 * kEpiHalves), row0);
        }
      }
    }
    if (!released) rel(lane);
    c_uses += (uint32_t)nown;
    if (nown > 0 && row_ok) atomicAdd(p.dprob + row, dprob_acc);
    if (want_amax && nown > 0) {
      if constexpr (OP == kOpGlu) {
        amax_flush(g, 2 * g, amx0);
        amax_flush(g, 2 * g + 1, amx1);
      } else {
        amax_flush(g, g, amx0);
      }
    }
    if (ctx.q == 0 && half == 0 && lane == 0) log_tile(w, t, ctx.rank);
  }

  __device__ void epilogue_regc(const TileWork& w, long long t, uint32_t taddr, const EpiCtx& ctx,
                                AccRelease rel) const {
    const int lane = ctx.lane, half = ctx.half;
    const int g = MGG_IN_BOUNDS(p.status, w.expert < p.L, 101, w.expert) ? w.expert : 0;
    const float alpha_g = __ldg(p.alpha + g);
    const float alpha2 = alpha_g * alpha_g;
    const float beta_g = __ldg(p.beta + g);
    const int row0 = w.m0 + ctx.rank * BM + ctx.q * 32;
    const bool row_ok = MGG_IN_BOUNDS(p.status, row0 + ctx.lane < p.M, 102, row0 + ctx.lane);
    const int row = row_ok ? row0 + lane : 0;  // checked build: a bad row reads row 0 and adds nothing
    const float pr = row_ok ? __ldg(p.prob + row) : 0.0f;
    const size_t row_off = (size_t)row * 2 * (size_t)p.N;
    const uint32_t stg = smem_u32(ctx.stg);
    const int nchunks = num_chunks(w);
    const bool want_amax = p.amax != nullptr;
    float dprob_acc = 0.f;
    float amx0 = 0.f, amx1 = 0.f;
    bool released = false;

    uint4 cg[CV], ci[CV];
    if (half < nchunks) load_c(row_off, w.n0 + 32 * half, cg, ci);
#pragma unroll 1
    for (int c = half; c < nchunks; c += kEpiHalves) {
      const int j0 = w.n0 + c * 32;
      uint32_t r[32];
      tmem_load_32cols(taddr + (MGG_IN_BOUNDS(p.status, c * 32 + 32 <= BN, 105, c) ? c * 32 : 0), r);
      if (c + kEpiHalves >= nchunks) {  // this warp's last read: the MMA warp may reuse the accumulator
        rel(lane);
        released = true;
      }
      uint4 ng[CV], ni[CV];
      if (c + kEpiHalves < nchunks) load_c(row_off, j0 + 32 * kEpiHalves, ng, ni);
      float gv[32], iv[32];
      unpack_c(cg, gv);
      unpack_c(ci, iv);
      dprob_acc += dglu_math<32>(r, gv, iv, alpha2, beta_g, pr);
      if (want_amax) {
        amx0 = absmax32(gv, amx0);
        amx1 = absmax32(iv, amx1);
      }
      if constexpr (DS == 2) {  // both 32-column blocks in one 64-column box
        staging_free(lane);
        stage_block(stg, lane, p.gate_first ? 0 : 1, gv);
        stage_block(stg, lane, p.gate_first ? 1 : 0, iv);
        staging_flush(stg, lane, 2 * j0, row0);
      } else {  // fp32: one 32-column box per block
        const int first = 2 * j0, second = 2 * j0 + 32;
        staging_free(lane);
        stage_block(stg, lane, 0, gv);
        stage_block(stg + 4096, lane, 0, iv);
        fence_async_shared();
        __syncwarp();
        if (lane == 0) {
          store_box(stg, p.gate_first ? first : second, row0);
          store_box(stg + 4096, p.gate_first ? second : first, row0);
          bulk_commit_group();
        }
      }
      if (p.dbias_ws != nullptr) dbias_partials(w, j0, lane, gv, iv);
#pragma unroll
      for (int i = 0; i < CV; ++i) {
        cg[i] = ng[i];
        ci[i] = ni[i];
      }
    }
    if (!released) rel(lane);
    if (half < nchunks && row_ok) atomicAdd(p.dprob + row, dprob_acc);
    if (want_amax && half < nchunks) {
      amax_flush(g, 2 * g, amx0);
      amax_flush(g, 2 * g + 1, amx1);
    }
    if (ctx.q == 0 && half == 0 && lane == 0) log_tile(w, t, ctx.rank);
  }

  __device__ void epilogue(const TileWork& w, long long t, uint32_t taddr, bool, const EpiCtx& ctx,
                           AccRelease rel) const {
    static_assert(OP == kOpGlu || Cfg::kTmaC, "the dsReLU epilogue reads C through the TMA ring");
    if constexpr (Cfg::kTmaC) epilogue_tmac(w, t, taddr, ctx, rel);
    else epilogue_regc(w, t, taddr, ctx, rel);
  }
};

template <int BN, int CS, int DS, bool TMAC, bool PAIR, int OP, int EPI>
__global__ void __launch_bounds__(cta_threads(DgluCfg<CS, DS, TMAC, PAIR, EPI>::kEpiWarps), 1)
    dglu_bwd_kernel(const __grid_constant__ DgluParams prm) {
  DgluPolicy<BN, CS, DS, TMAC, PAIR, OP, EPI> pol(prm);
  persistent_gemm<BN, DgluCfg<CS, DS, TMAC, PAIR, EPI>::kStages, PAIR>(pol);
}

template <int BN, int CS, int DS, bool TMAC, bool PAIR, int OP = kOpGlu, int EPI = 8>
static cudaError_t launch_dglu_variant(const DgluParams& prm, int num_sms, int device, cudaStream_t stream) {
  using C = DgluCfg<CS, DS, TMAC, PAIR, EPI>;
  constexpr int smem = SmemLayout<PAIR ? BN / 2 : BN, C::kStages, C::kEpiWarps, C::kStgBytes, num_acc(BN)>::DYN_BYTES;
  auto kern = dglu_bwd_kernel<BN, CS, DS, TMAC, PAIR, OP, EPI>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  static UnitCache cache;  // co-resident CTAs (pairs) of this variant, asked once per device
  return launch_persistent(kern, prm, prm.total_tiles, num_sms, PAIR, cta_threads(C::kEpiWarps), smem,
                           cache.slot(device), stream);
}

// Checks the device-resident arguments, builds the per-expert weight maps and zeroes amax.
__global__ void dglu_prep_kernel(const int32_t* offsets, int L, long long M, const int64_t* b_ptrs,
                                 const __grid_constant__ CUtensorMap tmpl, CUtensorMap* maps, int* status,
                                 float* amax, int n_amax) {
  griddep_launch_dependents();  // the GEMM kernel may launch now; it waits for this kernel's results
  bool bad_off = false, bad_ptr = false;
  for (int e = threadIdx.x; e < L; e += blockDim.x) {
    const int prev = e ? offsets[e - 1] : 0;
    const int cur = offsets[e];
    if (cur < prev || ((cur - prev) & 255) != 0) bad_off = true;
    if (e == L - 1 && (long long)cur != M) bad_off = true;
    if (b_ptrs != nullptr) {
      const long long ptr = b_ptrs[e];
      if (ptr == 0 || (ptr & 15) != 0) bad_ptr = true;
    }
  }
  const int any_off = __syncthreads_or(bad_off);
  const int any_ptr = __syncthreads_or(bad_ptr);
  if (threadIdx.x == 0) {
    status[0] = any_off ? (int)MGG_ERR_DEVICE_OFFSETS : any_ptr ? (int)MGG_ERR_DEVICE_POINTER : 0;
    status[1] = 0;
    status[2] = 0;
    status[3] = 0;
  }
  if (any_off || any_ptr) return;  // outputs stay untouched
  if (amax != nullptr)
    for (int i = threadIdx.x; i < n_amax; i += blockDim.x) amax[i] = 0.0f;
  if (b_ptrs == nullptr) return;
  const uint4* src = reinterpret_cast<const uint4*>(&tmpl);
  for (int e = threadIdx.x; e < L; e += blockDim.x) {
    uint4* dst = reinterpret_cast<uint4*>(maps + e);
#pragma unroll
    for (int i = 0; i < 8; ++i) dst[i] = src[i];
    tmap_replace_address(maps + e, reinterpret_cast<const void*>(b_ptrs[e]));
  }
  tmap_release();
}

// dbias (bf16) = bf16(dbias + fp32 partial sums): a single rounding of old + sum.
__global__ void dbias_finalize_kernel(const float* ws, __nv_bfloat16* dbias, long long n, const int* status) {
  griddep_wait();  // launched to overlap the GEMM kernel's tail: its partial sums are complete from here
  if (*status != 0) return;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    dbias[i] = __float2bfloat16_rn(__bfloat162float(dbias[i]) + ws[i]);
}

// What both grouped-GEMM epilogue calls pass to the launch (from mgg_dglu_bwd_args or
// mgg_dsrelu_bwd_args).
struct EpiCall {
  int64_t M, K, N, L;            // N: compact width (dGLU) or columns of C / D_row (dsReLU)
  const int64_t* b_ptrs;
  int b_major;
  const int32_t* offsets;
  const float* alpha;
  const float* beta;             // dGLU only
  const float* prob;
  const void* c;
  float* dprob;
  void* dbias;                   // dGLU only
  float* amax;
  bool d_col;
  void* workspace;
  int32_t* tile_log;
  int64_t tile_log_capacity;
  int sched, c_dtype, d_dtype;
  int act, geglu_filter, gate_first;
  float situ_beta1, situ_beta2;
};

template <int OP>
static cudaError_t launch_epi_gemm(const DgluLaunch& Lc, const EpiCall& a, cudaStream_t stream) {
  constexpr int BN = kDgluTileN;

  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  int* status = reinterpret_cast<int*>(ws);
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(ws + kWsHeaderBytes);
  float* dbias_ws = reinterpret_cast<float*>(ws + kWsHeaderBytes + kTmapBytes * (size_t)a.L);

  // stream order: the fills, the preparation kernel, then the GEMM kernel, which may launch while
  // the preparation kernel runs, then the dbias finalisation
  cudaError_t err;
  if (a.dbias != nullptr) {
    err = cudaMemsetAsync(dbias_ws, 0, sizeof(float) * (size_t)a.L * 2 * (size_t)a.N, stream);
    if (err != cudaSuccess) return err;
  }
  if (a.tile_log != nullptr && a.tile_log_capacity > 0) {
    err = cudaMemsetAsync(a.tile_log, 0xff, sizeof(int32_t) * 4 * (size_t)a.tile_log_capacity, stream);
    if (err != cudaSuccess) return err;
  }
  dglu_prep_kernel<<<1, 1024, 0, stream>>>(a.offsets, (int)a.L, (long long)a.M, a.b_ptrs, Lc.tmap_b, maps, status,
                                          a.amax, (int)(a.L * (OP == kOpGlu ? 2 : 1)));
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const long long num_n = (a.N + BN - 1) / BN;
  const long long total = (a.M / (Lc.pair ? 2 * BM : BM)) * num_n;  // M is a multiple of 256
  if (total > 0) {
    DgluParams prm;
    prm.tmap_a = Lc.tmap_a;
    prm.tmap_b = Lc.tmap_b;
    prm.tmap_d = Lc.tmap_d;
    prm.tmap_c = Lc.tmap_c;
    prm.tmap_dcol = Lc.tmap_dcol;
    prm.has_dcol = a.d_col ? 1 : 0;
    prm.amax = a.amax;
    prm.b_maps = a.b_ptrs != nullptr ? maps : nullptr;
    prm.offsets = a.offsets;
    prm.alpha = a.alpha;
    prm.beta = a.beta;
    prm.prob = a.prob;
    prm.c = a.c;
    prm.dprob = a.dprob;
    prm.dbias_ws = a.dbias != nullptr ? dbias_ws : nullptr;
    prm.status = status;
    prm.tile_log = a.tile_log;
    prm.tile_log_cap = a.tile_log != nullptr ? a.tile_log_capacity : 0;
    prm.total_tiles = total;
    prm.dynamic = a.sched == MGG_SCHED_DYNAMIC;
    prm.M = (int)a.M;
    prm.K = (int)a.K;
    prm.N = (int)a.N;
    prm.L = (int)a.L;
    prm.num_n = (int)num_n;
    prm.num_kb = (int)((a.K + BK - 1) / BK);
    prm.a_mn = 0;
    prm.b_mn = (a.b_ptrs != nullptr && a.b_major == MGG_MAJOR_MN) ? 1 : 0;
    prm.b_blocked = Lc.b_blocked ? 1 : 0;
    prm.c_dtype = a.c_dtype;
    prm.d_dtype = a.d_dtype;
    prm.act = a.act;
    prm.indicator = a.geglu_filter == MGG_FILTER_INDICATOR;
    prm.gate_first = a.gate_first != 0;
    prm.situ_b1 = a.situ_beta1 != 0.0f ? a.situ_beta1 : 4.0f;
    prm.situ_b2 = a.situ_beta2 != 0.0f ? a.situ_beta2 : 25.0f;
    prm.situ_inv_b1 = 1.0f / prm.situ_b1;
    prm.situ_inv_b2 = 1.0f / prm.situ_b2;

    const int cs = a.c_dtype == MGG_FP32 ? 4 : 2, ds = a.d_dtype == MGG_FP32 ? 4 : 2;
    const int n = Lc.num_sms, dev = Lc.device;
    // four epilogue warps (and one more operand stage) where the per-element work is light: the
    // C ring with 16-bit D_row and the dsReLU, dSwiGLU or (packed) dSiTU-GLU math
    const bool light = ds == 2 && (OP == kOpSrelu || a.act == MGG_ACT_DSWIGLU || a.act == MGG_ACT_DSITUGLU);
    if constexpr (OP == kOpSrelu) {  // 16-bit C through the TMA ring (the host checked C's dtype)
      if (Lc.pair) err = light ? launch_dglu_variant<BN, 2, 2, true, true, OP, 4>(prm, n, dev, stream)
                               : launch_dglu_variant<BN, 2, 4, true, true, OP>(prm, n, dev, stream);
      else err = light ? launch_dglu_variant<BN, 2, 2, true, false, OP, 4>(prm, n, dev, stream)
                       : launch_dglu_variant<BN, 2, 4, true, false, OP>(prm, n, dev, stream);
    } else if (Lc.pair) {  // pairs take the C ring whenever C is 16-bit
      if (cs == 2 && light) err = launch_dglu_variant<BN, 2, 2, true, true, kOpGlu, 4>(prm, n, dev, stream);
      else if (cs == 2) err = ds == 2 ? launch_dglu_variant<BN, 2, 2, true, true>(prm, n, dev, stream)
                                      : launch_dglu_variant<BN, 2, 4, true, true>(prm, n, dev, stream);
      else err = ds == 2 ? launch_dglu_variant<BN, 4, 2, false, true>(prm, n, dev, stream)
                         : launch_dglu_variant<BN, 4, 4, false, true>(prm, n, dev, stream);
    } else if (cs == 2 && a.K <= kTmaCMaxK) {
      if (light) err = launch_dglu_variant<BN, 2, 2, true, false, kOpGlu, 4>(prm, n, dev, stream);
      else err = ds == 2 ? launch_dglu_variant<BN, 2, 2, true, false>(prm, n, dev, stream)
                         : launch_dglu_variant<BN, 2, 4, true, false>(prm, n, dev, stream);
    } else if (cs == 2) {  // 16-bit C in registers one chunk ahead (single CTAs, K > kTmaCMaxK)
      if (light) err = launch_dglu_variant<BN, 2, 2, false, false, kOpGlu, 4>(prm, n, dev, stream);
      else err = ds == 2 ? launch_dglu_variant<BN, 2, 2, false, false>(prm, n, dev, stream)
                         : launch_dglu_variant<BN, 2, 4, false, false>(prm, n, dev, stream);
    } else {
      err = ds == 2 ? launch_dglu_variant<BN, 4, 2, false, false>(prm, n, dev, stream)
                    : launch_dglu_variant<BN, 4, 4, false, false>(prm, n, dev, stream);
    }
    if (err != cudaSuccess) return err;
  }
  if (a.dbias != nullptr) {
    const long long n = a.L * 2 * a.N;
    const int blocks = (int)((n + 255) / 256 < 1024 ? (n + 255) / 256 : 1024);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)(blocks > 0 ? blocks : 1), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, dbias_finalize_kernel, (const float*)dbias_ws,
                             static_cast<__nv_bfloat16*>(a.dbias), n, (const int*)status);
  }
  return err;
}

cudaError_t launch_dglu_bwd(const DgluLaunch& Lc, cudaStream_t stream) {
  const mgg_dglu_bwd_args& a = *Lc.args;
  EpiCall e{a.M, a.K, a.N, a.L, a.b_ptrs, a.b_major, a.padded_offsets, a.alpha, a.beta, a.prob, a.c, a.dprob,
            a.dbias, a.amax, a.d_col != nullptr, a.workspace, a.tile_log, a.tile_log_capacity, a.sched, a.c_dtype,
            a.d_dtype, a.act, a.geglu_filter, a.gate_first, a.situ_beta1, a.situ_beta2};
  return launch_epi_gemm<kOpGlu>(Lc, e, stream);
}

cudaError_t launch_dsrelu_bwd(const DgluLaunch& Lc, const mgg_dsrelu_bwd_args& a, cudaStream_t stream) {
  EpiCall e{a.M, a.K, a.N, a.L, a.b_ptrs, a.b_major, a.padded_offsets, a.alpha, nullptr, a.prob, a.c, a.dprob,
            nullptr, a.amax, a.d_col != nullptr, a.workspace, a.tile_log, a.tile_log_capacity, a.sched, a.c_dtype,
            a.d_dtype, MGG_ACT_DSWIGLU, MGG_FILTER_VALUE, 1, 0.0f, 0.0f};
  return launch_epi_gemm<kOpSrelu>(Lc, e, stream);
}

// ------------------------------------------------------------------------------------
// tensormap.replace probe (test hook)
// ------------------------------------------------------------------------------------
__global__ void tmap_replace_probe_kernel(const __grid_constant__ CUtensorMap tmpl, CUtensorMap* out,
                                          const void* addr, uint32_t dim0, uint64_t stride1, int fields) {
  if (threadIdx.x != 0) return;
  const uint4* src = reinterpret_cast<const uint4*>(&tmpl);
  uint4* dst = reinterpret_cast<uint4*>(out);
#pragma unroll
  for (int i = 0; i < 8; ++i) dst[i] = src[i];
  if (fields & 1) tmap_replace_address(out, addr);
  if (fields & 2) tmap_replace_dim(out, 0, dim0);
  if (fields & 4) tmap_replace_stride0(out, stride1);
  tmap_release();
}

cudaError_t launch_tmap_replace_probe(const CUtensorMap& tmpl, void* out, const void* addr, uint32_t dim0,
                                      uint64_t stride1, int fields, cudaStream_t stream) {
  tmap_replace_probe_kernel<<<1, 32, 0, stream>>>(tmpl, static_cast<CUtensorMap*>(out), addr, dim0, stride1, fields);
  return cudaGetLastError();
}

}  // namespace mgg
