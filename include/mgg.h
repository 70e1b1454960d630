/*
 * mgg.h - C ABI of the GB300 (sm_103a) BF16 MoE grouped GEMM backward.
 *
 * Two operations, restated from the cuDNN-frontend pages they come from:
 *
 *   mgg_dglu_bwd  "Grouped GEMM + dGLU (SM100)", BF16 contract, section
 *                 "Tensors, layouts, and equation": for expert g with rows
 *                 [padded_offsets[g-1], padded_offsets[g]),
 *                     R_g = alpha_g^2 * A_g * B_g^T,   X_g = beta_g * C_g,
 *                 X split into alternating 32-wide gate/input blocks, the dSwiGLU
 *                 or dGeGLU backward written to the interleaved D_row, dprob
 *                 accumulating the row sum of R times the unscaled activation and
 *                 the optional dbias accumulating the per-expert column sum of D_row.
 *
 *   mgg_wgrad     "Grouped GEMM + WGrad (Unified)", section "Operation":
 *                     Wgrad[e] = A[:, begin:end] @ B[begin:end, :],
 *                 begin = 0 for e = 0 else offsets[e-1], end = offsets[e];
 *                 overwrite (an empty expert produces zeros) or accumulate_on_output.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller and must stay
 *   valid until the work queued on `stream` has completed.  The library keeps no
 *   pointer after a call returns and allocates no device memory; scratch space is
 *   the caller's `workspace` (size from the *_workspace_size functions).
 *   Required pointers are non-NULL, except the per-row tensors of a call without
 *   rows (M == 0: a, c, prob, dprob, d_row) or tokens (tokens_sum == 0: a, b),
 *   which may be NULL: nothing is read from or written to them.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work of a
 *   call is queued on it; the call does not synchronise.  Inside a call the GEMM
 *   kernel may start while the call's preparation kernel still runs (programmatic
 *   dependent launch) and waits for its results.  The GEMM kernel also lets a
 *   kernel that the caller queues after it WITH programmatic stream serialization
 *   start launching as its tiles finish: such a kernel must wait for its
 *   prerequisites (griddepcontrol.wait / cudaGridDependencySynchronize) before it
 *   reads this call's outputs.  Ordinary launches, copies and events see the call's
 *   outputs complete, as with any stream-ordered work.
 * - Arguments are validated on the host before anything is queued.  A violation
 *   returns a status != MGG_OK, queues nothing and leaves every output untouched
 *   (mgg_last_error() holds a message).  Offsets and pointer-array CONTENTS live on
 *   the device: they are checked by the first kernel of the call, which writes a
 *   status word into the workspace and turns the rest of the call into no-ops
 *   (outputs untouched); read it with mgg_read_device_status().
 * - A workspace must not be shared by calls that may run concurrently.
 * - Calls are thread-safe; the error message is thread-local.
 */
#ifndef MGG_H_
#define MGG_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MGG_ABI_VERSION 5

typedef enum mgg_status {
  MGG_OK = 0,
  MGG_ERR_VALUE = 1,          /* bad shape, stride, dtype, alignment, mode or pointer (ValueError) */
  MGG_ERR_UNSUPPORTED = 2,    /* allowed by the pages but not provided by this library */
  MGG_ERR_RUNTIME = 3,        /* CUDA runtime/driver error while preparing or launching */
  MGG_ERR_ARCH = 4,           /* no usable device, or the device is not sm_103 */
  MGG_ERR_DEVICE_OFFSETS = 5, /* device check: offsets not non-decreasing / not 256-multiples / wrong end */
  MGG_ERR_DEVICE_POINTER = 6, /* device check: a pointer-array entry is null or not 16-byte aligned */
  MGG_ERR_DEVICE_TIMEOUT = 7, /* a pipeline wait inside a kernel exceeded its time limit */
  MGG_ERR_DEVICE_BOUNDS = 8   /* bounds-checked build only: a computed global index or TMEM column
                                 fell outside the call's extents; the access was skipped */
} mgg_status;

typedef enum mgg_dtype { MGG_BF16 = 0, MGG_FP16 = 1, MGG_FP32 = 2 } mgg_dtype;

/* dGLU page, "Common Parameters": act_func "dswiglu" (default), "dgeglu", or "dsituglu" (whose
 * equations the page gives under "Block-scaled contract", "Equations": T_g = beta1 tanh(G/beta1)
 * sigmoid(G), T_u = beta2 tanh(U/beta2); here it runs in the BF16 path). */
typedef enum mgg_act { MGG_ACT_DSWIGLU = 0, MGG_ACT_DGEGLU = 1, MGG_ACT_DSITUGLU = 2 } mgg_act;

/* dGeGLU filters.  VALUE: as printed on the dGLU page (gate_filter = raw_gate when
 * raw_gate <= 7 else 0; input_filter = raw_input when -7 <= raw_input <= 7 else 0).
 * INDICATOR: 1 in place of the raw value (the analytic derivative of the clamped GeGLU). */
typedef enum mgg_geglu_filter { MGG_FILTER_VALUE = 0, MGG_FILTER_INDICATOR = 1 } mgg_geglu_filter;

/* Storage major of a matrix operand: K = the reduction axis has unit stride;
 * MN = the row/column (M or N) axis has unit stride. */
typedef enum mgg_major { MGG_MAJOR_K = 0, MGG_MAJOR_MN = 1 } mgg_major;

/* Persistent tile scheduling (dGLU page, class API: use_dynamic_sched; wgrad page,
 * "Scheduling, cache, and errors": dynamic persistent scheduling). */
typedef enum mgg_sched { MGG_SCHED_STATIC = 0, MGG_SCHED_DYNAMIC = 1 } mgg_sched;

/* How output tiles map to SMs.  SINGLE: one CTA per SM computes 128-row tiles (cta_group::1).
 * PAIR: a cluster of two CTAs on two SMs computes 256-row tiles with cta_group::2 MMAs, each CTA
 * loading its own 128 rows of A and half of the tile's B columns (half the B traffic per SM);
 * wgrad accepts PAIR only when hidden is a multiple of 256.  AUTO: the library picks per call.
 * The result and the tile log (one entry per 128-row CTA tile) do not depend on the mode. */
typedef enum mgg_cta_mode { MGG_CTA_AUTO = 0, MGG_CTA_SINGLE = 1, MGG_CTA_PAIR = 2 } mgg_cta_mode;

/* wgrad page, "BF16 contract": input_order "tensor2d" (declared strides) or
 * "tensor_ragged" (per-expert K-contiguous blocks concatenated in memory). */
typedef enum mgg_input_order { MGG_ORDER_TENSOR2D = 0, MGG_ORDER_TENSOR_RAGGED = 1 } mgg_input_order;

/*
 * Arguments of mgg_dglu_bwd (dGLU page, BF16 contract).  M = valid rows =
 * padded_offsets[L-1]; K = reduction dimension; N = compact gradient width; L = experts.
 *
 *   a              bf16 (M, K), stride (K, 1)                           [read]
 *   b              dense weights: bf16 (N, K, L), stride (K, 1, N*K),   [read]
 *                  i.e. L consecutive K-major (N, K) matrices; or NULL
 *   b_ptrs         discrete weights: device int64[L], entry g = address of expert g's
 *                  bf16 (N, K) matrix, K-major (stride (K, 1)) when b_major = MGG_MAJOR_K
 *                  or N-major (stride (1, N)) when MGG_MAJOR_MN; or NULL.
 *                  Exactly one of b / b_ptrs must be given.
 *   c              (M, 2N), stride (2N, 1), dtype c_dtype                [read]
 *   padded_offsets int32[L], cumulative 256-aligned group ends           [read]
 *   alpha, beta    fp32[L]; prob fp32[M]                                 [read]
 *   dprob          fp32[M], caller-initialised (normally zero); the row sums are ADDED
 *   d_row          (M, 2N), stride (2N, 1), dtype d_dtype               [write]
 *   dbias          bf16 (L, 2N), caller-initialised; column sums are ADDED
 *                  (one bf16 rounding of old + sum); NULL = no dbias
 *   d_col          optional second copy of D_row, same shape, stride and dtype (the dGLU
 *                  page's column output; without quantisation it holds the D_row values);
 *                  NULL = off                                            [write]
 *   amax           optional fp32 (L, 2): per expert the largest |dgate| and |dinput| over
 *                  its rows (the page's per-group amax of 16-bit D_row; the two entries are
 *                  the gate and the input block), before output rounding; 0 for an empty
 *                  expert.  Overwritten (the call zeroes it first).  NULL = off  [write]
 *   workspace      device scratch of at least mgg_dglu_bwd_workspace_size(L, N) bytes,
 *                  256-byte aligned
 *   tile_log       optional int32[4 * tile_log_capacity]: for every output tile the
 *                  kernel writes (expert, m0, n0, cta); unused entries are -1.  NULL = off.
 * Requirements checked on the host: 1 <= L <= 1024; M, K, N >= 0 with M % 256 == 0,
 * K % 8 == 0 and N % 32 == 0; every pointer 16-byte aligned; dtypes in range.
 */
typedef struct mgg_dglu_bwd_args {
  int64_t M, K, N, L;
  const void* a;
  const void* b;
  const int64_t* b_ptrs;
  const void* c;
  const int32_t* padded_offsets;
  const float* alpha;
  const float* beta;
  const float* prob;
  float* dprob;
  void* d_row;
  void* dbias;
  void* d_col;
  float* amax;
  void* workspace;
  int32_t* tile_log;
  int64_t workspace_bytes;
  int64_t tile_log_capacity;
  int32_t b_major;        /* mgg_major, discrete weights only (dense weights are K-major) */
  int32_t c_dtype;        /* mgg_dtype */
  int32_t d_dtype;        /* mgg_dtype */
  int32_t act;            /* mgg_act */
  int32_t geglu_filter;   /* mgg_geglu_filter */
  int32_t gate_first;     /* 1: the gate block precedes the input block in every 64 columns */
  int32_t sched;          /* mgg_sched */
  int32_t cta_mode;       /* mgg_cta_mode */
  float situ_beta1;       /* dSiTU-GLU gate tanh scale, positive finite; 0 = the default 4.0 */
  float situ_beta2;       /* dSiTU-GLU input tanh scale, positive finite; 0 = the default 25.0 */
} mgg_dglu_bwd_args;

/*
 * Arguments of mgg_dsrelu_bwd: the dsReLU page's epilogue ("Equations") on the BF16 grouped
 * GEMM of the dGLU page's layouts.  M = valid rows = padded_offsets[L-1]; N = columns of C,
 * D_row and the GEMM result G.
 *
 *   a, b, b_ptrs, b_major, padded_offsets, prob, dprob, workspace, tile_log: as for
 *                  mgg_dglu_bwd (dprob: the row sums are ADDED)
 *   c              (M, N), stride (N, 1), 16-bit (bf16 or fp16)           [read]
 *   alpha          fp32[L]: G = alpha_g * A_g B_g^T (alpha, not squared)  [read]
 *   d_row          (M, N), stride (N, 1), dtype d_dtype:
 *                  D_row = prob * 2 * C * relu(G)                         [write]
 *   dprob          dprob[m] += sum_n C[m, n] * relu(G[m, n])^2
 *   d_col          optional copy of D_row (same shape, stride, dtype); NULL = off [write]
 *   amax           optional fp32 (L): per expert the largest |D_row| before output rounding,
 *                  0 for an empty expert; overwritten.  NULL = off            [write]
 *   workspace      at least mgg_dsrelu_bwd_workspace_size(L) bytes, 256-byte aligned
 * Requirements checked on the host: as for mgg_dglu_bwd with C (M, N); C is 16-bit.
 */
typedef struct mgg_dsrelu_bwd_args {
  int64_t M, K, N, L;
  const void* a;
  const void* b;
  const int64_t* b_ptrs;
  const void* c;
  const int32_t* padded_offsets;
  const float* alpha;
  const float* prob;
  float* dprob;
  void* d_row;
  void* d_col;
  float* amax;
  void* workspace;
  int32_t* tile_log;
  int64_t workspace_bytes;
  int64_t tile_log_capacity;
  int32_t b_major;        /* mgg_major, discrete weights only */
  int32_t c_dtype;        /* mgg_dtype: MGG_BF16 or MGG_FP16 */
  int32_t d_dtype;        /* mgg_dtype */
  int32_t sched;          /* mgg_sched */
  int32_t cta_mode;       /* mgg_cta_mode */
  int32_t reserved;       /* must be 0 */
} mgg_dsrelu_bwd_args;

/*
 * Arguments of mgg_wgrad (wgrad page, BF16 contract).  T = tokens_sum = offsets[L-1].
 *
 *   a        bf16 A (hidden, T): K-major stride (T, 1) when a_major = MGG_MAJOR_K, or
 *            M-major stride (1, hidden) when MGG_MAJOR_MN                         [read]
 *   b        bf16 B (T, inter): N-major stride (inter, 1) when b_major = MGG_MAJOR_MN,
 *            or K-major stride (1, T) when MGG_MAJOR_K                             [read]
 *            input_order TENSOR_RAGGED: a K-major operand is stored as per-expert
 *            K-contiguous blocks, expert e's block at element begin*hidden (A:
 *            (hidden, K_e), row length K_e) or begin*inter (B: (inter, K_e)); an MN-major
 *            operand is unaffected.
 *   offsets  int32[L], non-decreasing cumulative token ends, counts multiples of 256
 *   out      dense output (L, hidden, inter), stride (hidden*inter, inter, 1); or NULL
 *   out_ptrs discrete outputs: device int64[L] of (hidden, inter) row-major matrices,
 *            each non-null and 16-byte aligned; or NULL.  Exactly one of out / out_ptrs.
 *   out_dtype bf16 / fp16 / fp32; accumulate != 0: out = old + Wgrad (one rounding)
 *            and empty experts are left untouched; accumulate == 0: out = Wgrad, zeros
 *            for an empty expert.
 * Requirements checked on the host: 1 <= L <= 1024; hidden, inter >= 8, multiples of 8;
 * tokens_sum % 256 == 0; every pointer 16-byte aligned.
 */
typedef struct mgg_wgrad_args {
  int64_t hidden, inter, L, tokens_sum;
  const void* a;
  const void* b;
  const int32_t* offsets;
  void* out;
  const int64_t* out_ptrs;
  void* workspace;
  int32_t* tile_log;
  int64_t workspace_bytes;
  int64_t tile_log_capacity;
  int32_t a_major;        /* mgg_major */
  int32_t b_major;        /* mgg_major */
  int32_t input_order;    /* mgg_input_order */
  int32_t out_dtype;      /* mgg_dtype */
  int32_t accumulate;     /* accumulate_on_output */
  int32_t sched;          /* mgg_sched */
  int32_t cta_mode;       /* mgg_cta_mode */
  int32_t reserved1;      /* must be 0 */
} mgg_wgrad_args;

/* Library ABI version (MGG_ABI_VERSION of the build). */
int mgg_abi_version(void);

/* sizeof the argument structs as compiled into the library (binding layout checks). */
size_t mgg_sizeof_dglu_bwd_args(void);
size_t mgg_sizeof_dsrelu_bwd_args(void);
size_t mgg_sizeof_wgrad_args(void);

/* Byte offset of every field of one argument struct as compiled into the library, in declaration
 * order (which = 0: mgg_dglu_bwd_args, 1: mgg_dsrelu_bwd_args, 2: mgg_wgrad_args).  Writes at most
 * `cap` offsets into `out` (host memory; may be NULL when cap = 0) and returns the struct's number of
 * fields, or -1 for an unknown `which`.  Lets a binding check its mirror of the structs field by
 * field, not only by size. */
int mgg_args_field_offsets(int which, size_t* out, int cap);

/* Last error message of the calling thread ("" after a successful call). */
const char* mgg_last_error(void);

/* Name of a status code. */
const char* mgg_status_string(int status);

/* Workspace bytes for mgg_dglu_bwd with L experts and compact width N
 * (status word, per-expert tensor-map slots, fp32 dbias partial sums). */
size_t mgg_dglu_bwd_workspace_size(int64_t L, int64_t N);

/* Workspace bytes for mgg_dsrelu_bwd with L experts (status word, per-expert tensor-map slots). */
size_t mgg_dsrelu_bwd_workspace_size(int64_t L);

/* Workspace bytes for mgg_wgrad with L experts (status word, per-expert tensor-map
 * slots for ragged inputs and discrete outputs, the expert order of the scheduler). */
size_t mgg_wgrad_workspace_size(int64_t L);

/* Number of output tiles mgg_dglu_bwd / mgg_wgrad enumerate (tile_log capacity); mgg_dsrelu_bwd
 * enumerates mgg_dglu_bwd_num_tiles(M, N) tiles of the same shape. */
int64_t mgg_dglu_bwd_num_tiles(int64_t M, int64_t N);
int64_t mgg_wgrad_num_tiles(int64_t L, int64_t hidden, int64_t inter);
/* Tile shape (rows, columns) of the output tiles each operation logs. */
void mgg_dglu_bwd_tile_shape(int32_t* tile_m, int32_t* tile_n);
void mgg_wgrad_tile_shape(int64_t inter, int32_t* tile_m, int32_t* tile_n);

/* Grouped GEMM + dGLU backward.  Queues its kernels on `stream` (a cudaStream_t). */
mgg_status mgg_dglu_bwd(const mgg_dglu_bwd_args* args, void* stream);

/* Grouped GEMM + dsReLU backward.  Queues its kernels on `stream` (a cudaStream_t). */
mgg_status mgg_dsrelu_bwd(const mgg_dsrelu_bwd_args* args, void* stream);

/* Grouped wgrad.  Queues its kernels on `stream` (a cudaStream_t). */
mgg_status mgg_wgrad(const mgg_wgrad_args* args, void* stream);

/* Grouped wgrad for callers that cannot allocate device memory (no counterpart on the
 * pages).  Same arguments and results as mgg_wgrad, except that `workspace` and
 * `workspace_bytes` are ignored: the scratch lives in a fixed array inside the library's
 * device memory, sized for at most 1024 experts (397,568 bytes, held on every GPU that loads
 * the library until the process exits); L above that returns MGG_ERR_VALUE.  Nothing is
 * allocated.  The first call on a device (and the first after its context was reset) looks
 * the array's address up with that device current: make it before any stream capture.
 * Every call shares the array and it keeps the last call's contents; calls that may overlap
 * on the GPU race on it and must be ordered.
 * The device-side status word of these calls is not exposed: when the offsets or out_ptrs
 * contents fail the device check (see mgg_wgrad), the call still returns MGG_OK and leaves
 * every output untouched.  Callers of this entry point must therefore check their offsets
 * (non-decreasing, counts multiples of 256, last == tokens_sum) and output pointers (non-null,
 * 16-byte aligned) on the host before the call. */
mgg_status mgg_wgrad_noalloc(const mgg_wgrad_args* args, void* stream);

/* Waits for `stream`, then returns the device-side status word of the last call that
 * used `workspace` (MGG_OK, MGG_ERR_DEVICE_OFFSETS, MGG_ERR_DEVICE_POINTER or
 * MGG_ERR_DEVICE_TIMEOUT).  Synchronising; not for use inside stream capture. */
mgg_status mgg_read_device_status(const void* workspace, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MGG_H_ */
