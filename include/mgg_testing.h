/*
 * mgg_testing.h - test hooks of libmgg (not part of the operation's interface).
 *
 * They let the test suite check, without issuing any TMA copy, that the device-side
 * tensor-map rewriting used for per-expert operands (discrete weight pointers,
 * tensor_ragged inputs) produces exactly the descriptor the driver would encode.
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

#ifdef __cplusplus
}
#endif

#endif /* MGG_TESTING_H_ */
