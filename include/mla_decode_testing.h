/*
 * mla_decode_testing.h -- test and benchmark hooks of the MLA decode library.
 * Not part of the decode operation: one exercises its failure detection, the
 * other measures the memory ceiling of its access pattern.
 *
 * Every wait inside the tensor-core decode kernel is bounded (2 s).  When a
 * wait runs out, the kernel records MLA device error 1 (wait timeout, read
 * with mla_device_error), stops its other roles, drains what it has in
 * flight, frees its tensor memory and returns; the CUDA context stays usable.
 */
#ifndef MLA_DECODE_TESTING_H_
#define MLA_DECODE_TESTING_H_

#include <stdint.h>

#include "mla_decode.h" /* MLA_API */

#ifdef __cplusplus
extern "C" {
#endif

/* on != 0: every later tensor-core decode launch made from the CALLING
 * THREAD (other threads are unaffected) issues no page copies, so each of its
 * waits for a page runs out after 2 s and the launch ends with device error
 * 1; its outputs are undefined.  on == 0 restores normal operation.  Returns
 * the previous setting of this thread.  Host-side only: nothing on the GPU
 * faults, traps or hangs. */
MLA_API int mla_test_stall_copies(int on);

/* Instrumentation of the tensor-core kernels' online softmax: the next decode
 * call (mla_decode_paged or mla_decode_paged_noalloc) made by the calling
 * thread adds, with device atomics, to device_counts[0] the number of times an
 * attention warpgroup rescaled its accumulated output tile in tensor memory
 * because a row's reference maximum moved after that warpgroup's first page,
 * and to device_counts[1] the number of reference moves of any kind
 * (including the first page's).  device_counts: device int32[2], zeroed by the
 * caller.  One-shot and thread-local; the CUDA-core kernel counts nothing.
 * Returns 0. */
MLA_API int mla_test_count_rescales(int32_t *device_counts);

/* Benchmark instrumentation: the HBM ceiling of the decode's access pattern.
 * Launches `ctas` CTAs; CTA c copies the pages page_ids[c * pages_per_cta + i]
 * (i < pages_per_cta) of the cache, whole 36,864-byte pages, through TMA into
 * a 4-deep shared-memory ring, exactly as the tensor-core decode kernel
 * stages them, and discards them.  No arithmetic, no output: the time of one
 * launch is the floor for any kernel that reads those pages that way.
 *
 *   kv_cache       device, [num_pages, 64, 576] bytes, 16-byte aligned.
 *   num_pages      >= 1, num_pages * 64 < 2^31.
 *   page_ids       device int32 [ctas * pages_per_cta]; an id outside
 *                  [0, num_pages) reads page 0 and sets device error 2.
 *   ctas           1 .. 65535; pages_per_cta >= 1.
 *   stream         cudaStream_t as void*.
 * Asynchronous on `stream`; returns an mla_status_t (0 = MLA_OK; nothing is
 * launched on error).  Waits are bounded like the decode kernel's (2 s,
 * device error 1). */
MLA_API int mla_bench_stream_pages(const void *kv_cache, int64_t num_pages, const int32_t *page_ids,
                           int32_t ctas, int32_t pages_per_cta, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_TESTING_H_ */
