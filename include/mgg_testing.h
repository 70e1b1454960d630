/*
 * mgg_testing.h - test hooks of libmgg (not part of the operation's interface).
 *
 * They let the test suite check, without issuing any TMA copy, that the device-side
 * tensor-map rewriting used for per-expert operands (discrete weight pointers,
 * tensor_ragged inputs) produces exactly the descriptor the driver would encode, and
 * that a pipeline wait that never completes ends with MGG_ERR_DEVICE_TIMEOUT.
 */
#ifndef MGG_TESTING_H_
#define MGG_TESTING_H_

#include <stddef.h>
#include <stdint.h>

#include "mgg.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Encodes on the host a 2-D bf16 tiled tensor map (128-byte swizzle) into out128 (128 bytes,
 * host memory, 64-byte aligned): dims {dim0, dim1}, byte stride of dim 1, box {box0, box1}.
 * Needs the CUDA driver; returns MGG_ERR_RUNTIME when the driver rejects the arguments. */
mgg_status mgg_test_encode_tmap_2d(void* out128, const void* addr, uint64_t dim0, uint64_t dim1,
                                   uint64_t stride1_bytes, uint32_t box0, uint32_t box1);

/* Copies the host descriptor tmpl128 into device memory out_dev128 (128 bytes, 128-byte
 * aligned) and rewrites there, with tensormap.replace, the fields selected by `fields`:
 * bit 0 global address = addr, bit 1 dim0 = dim0, bit 2 byte stride of dim 1 = stride1.
 * Queued on `stream`; the result is read back by the caller. */
mgg_status mgg_test_tmap_replace(const void* tmpl128, void* out_dev128, const void* addr, uint32_t dim0,
                                 uint64_t stride1_bytes, int fields, void* stream);

/* Launches one CTA (two as a cluster when cluster = 1) whose first thread waits on a shared-memory
 * mbarrier that nothing ever arrives on, through the same bounded wait the grouped GEMM kernels use
 * (acquire at cluster scope when cluster = 1), with the limit limit_ns (0 < limit_ns <= 1e8) in
 * place of their 1 s.  The wait gives up after the limit and records, in status_dev (device int32[4],
 * 16-byte aligned): [0] = MGG_ERR_DEVICE_TIMEOUT, [1] = where, [2] = the CTA; then a second wait of
 * the same CTA must return at once because the abort flag is up, without overwriting [1]; [3] holds
 * bit 0 (first wait failed), bit 1 (second wait returned early) and bit 2 ([1] kept).  The kernel
 * issues no TMA copy and no MMA.  Queued on `stream`; read the word with mgg_read_device_status. */
mgg_status mgg_test_wait_timeout(void* status_dev, int64_t limit_ns, int32_t where, int32_t cluster, void* stream);

/* Runs, in one thread, the index check the kernels make on a computed index: `value` against
 * [0, limit).  In the bounds-checked build a value outside records MGG_ERR_DEVICE_BOUNDS in
 * status_dev (device int32[4], 16-byte aligned, zeroed by the caller): [0] = 8, [1] = 501,
 * [2] = the value; and the guarded write of [3] = 1 is skipped.  In the normal build the check
 * compiles away and [3] = 1 is always written.  Queued on `stream`. */
mgg_status mgg_test_bounds_check(void* status_dev, int64_t value, int64_t limit, void* stream);

/* Build flags of the loaded library: bit 0 set for the bounds-checked build (-DMGG_CHECKED), whose
 * kernels test every computed global index, tensor-map slot and TMEM column against the call's
 * extents and record MGG_ERR_DEVICE_BOUNDS (where, value) instead of making the access. */
int mgg_test_build_flags(void);

#ifdef __cplusplus
}
#endif

#endif /* MGG_TESTING_H_ */
