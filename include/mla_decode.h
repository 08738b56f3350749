/*
 * mla_decode.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * One operation and its merge step, from the blog post "Kimi K3 on AMD
 * Instinct MI355X: vLLM serving ..." (three language editions):
 *
 *   - Model section: every MLA layer keeps a compressed KV history that grows
 *     with the conversation; each new query attends over all of it.
 *   - Section 1 "Cache", DCP paragraph: a history can be cut into shards; each
 *     partial answer carries normalisation information (its log-sum-exp) and
 *     the partial answers are merged with softmax weights.  The worked figure
 *     24 layers x 142,000 positions x 576 FP8 bytes fixes one byte per latent
 *     element and no per-position scale bytes.
 *   - Section 4 "MLA": query heads attend independently; the history is split
 *     into parallel partitions inside one GPU and the results are combined,
 *     with the KV storage unchanged.
 *   - Benchmark configuration section: FP8 KV cache.
 *
 * Conventions this library fixes where the post is silent:
 *   - a cached position is 576 OCP E4M3FN codes; codes [0, 512) are the latent
 *     (also the value vector), codes [512, 576) the rotated positional part;
 *   - one fp32 scale for the whole cache: x = e4m3fn(code) * (*kv_scale);
 *   - pages of 64 positions, addressed through a block table;
 *   - seq_lens[b] counts the T new positions; query t sees positions
 *     p < seq_lens[b] - T + 1 + t;
 *   - lse is the natural log of sum_p exp(score_p), score_p including sm_scale.
 *
 * Threading and ownership: every call is asynchronous on the given CUDA
 * stream (a cudaStream_t passed as void*; NULL is the legacy default stream)
 * and never synchronises with the host.  The caller owns every tensor; the
 * library never frees or retains caller pointers beyond the call.  Scratch
 * memory for split partials is owned by the library, kept per (device,
 * stream) and grown with stream-ordered allocation on first need.  Calls on
 * one stream are ordered; calls on different streams use different scratch.
 * CUDA graphs: a call may be captured once an uncaptured call of at least
 * the same scratch size has run on that stream; a captured call that would
 * have to grow the scratch returns MLA_ERR_UNSUPPORTED and records nothing.
 * Scratch that a captured call used is not freed when the stream's scratch
 * grows, so the graph stays valid after later, larger calls on the stream; a
 * graph replayed on another stream still uses the scratch of the stream it was
 * captured on.  mla_release_graph_scratch() frees such scratch once the graphs
 * that used it are gone.
 *
 * Errors: every entry point validates its arguments on the host before any
 * launch and returns a status; mla_last_error() gives a message for the last
 * failing call of the calling thread.  Device kernels never trap: bounded
 * waits and the checks of device-resident indices (page ids, sequence
 * lengths, append positions) write a device error word that
 * mla_device_error() reads.
 */
#ifndef MLA_DECODE_H_
#define MLA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

/* Every entry point carries MLA_API: the library is built with hidden symbol
 * visibility, so these declarations are its only exported names. */
#if defined(__GNUC__) || defined(__clang__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,  /* null pointer, wrong rank/shape/dtype/stride   */
    MLA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dims != 576)   */
    MLA_ERR_CUDA = 3,         /* a CUDA runtime call failed; see mla_last_error */
    MLA_ERR_NO_MEMORY = 4,    /* scratch allocation failed                      */
    MLA_ERR_DEVICE = 5        /* a kernel reported an error (mla_device_error)  */
} mla_status_t;

typedef enum {
    MLA_DTYPE_BF16 = 1,
    MLA_DTYPE_F32 = 2,
    MLA_DTYPE_E4M3FN = 3,     /* raw OCP E4M3FN codes, one byte each */
    MLA_DTYPE_I32 = 4
} mla_dtype_t;

/* A strided view of device memory.  Strides are in elements.  This is the
 * library's own descriptor (not DLPack); unused trailing dims are ignored. */
typedef struct {
    void *data;
    int64_t shape[5];
    int64_t stride[5];
    int32_t ndim;
    int32_t dtype;            /* an mla_dtype_t */
} mla_tensor_t;

/* Kernel families behind mla_decode_paged (see mla_set_impl). */
typedef enum {
    MLA_IMPL_AUTO = 0,        /* tensor-core kernel where supported, else CUDA-core */
    MLA_IMPL_SIMT = 1,        /* CUDA-core split-KV kernel (FMA + shuffles)          */
    MLA_IMPL_TCGEN05 = 2      /* tcgen05 tensor-core split-KV kernel                  */
} mla_impl_t;

/*
 * mla_decode_paged -- MLA decode attention over a paged FP8 latent cache,
 * split into n_splits parallel partitions of the history and merged by LSE.
 *
 *   q           bf16  [B, T, H, 576], device, fully contiguous, base address
 *               16-byte aligned; the absorbed, already-rotated query of each
 *               head.
 *   kv_cache    e4m3fn [num_pages, 64, 576], device, fully contiguous; base
 *               address 16-byte aligned.
 *   kv_scale    device pointer to one fp32, the per-tensor dequantisation
 *               scale (read on the device, so the call can be captured in a
 *               CUDA graph while the scale changes).
 *   block_table i32 [B, max_pages], device, innermost dim contiguous; entry
 *               [b][j] is the physical page of positions 64j..64j+63 of
 *               request b.  Only the first ceil(seq_lens[b] / 64) entries are
 *               read; each must be in [0, num_pages).
 *   seq_lens    i32 [B], device; history length of request b including its T
 *               new positions; 0 (empty history) gives out = 0, lse = -inf;
 *               must be <= 64 * max_pages, and >= T unless 0.
 *   n_splits    > 0: use exactly this many history partitions per request;
 *               0: choose automatically to fill every SM (mla_auto_splits);
 *               a caller that knows the lengths on the host can pass
 *               mla_plan_splits(...) instead.
 *   sm_scale    softmax scale applied to q . x (e.g. 1/sqrt(192)).
 *   out         bf16 [B, T, H, 512], device, contiguous, caller-allocated;
 *               out = sum_p softmax_p * x_p[0:512], rounded to nearest even.
 *   lse         fp32 [B, T, H], device, contiguous, or NULL; natural log of
 *               the softmax normaliser (the merge weight of this answer).
 *   stream      cudaStream_t as void*.
 *
 * Limits: H * T <= 128; dims fixed at 576 / 512; page size fixed at 64.
 * Returns MLA_OK or an error status (nothing is launched on error).
 * Page ids and seq_lens live on the device, so the host cannot check them
 * without a synchronisation; the kernels do: a page id outside
 * [0, num_pages) is not read (its 64 positions contribute nothing) and sets
 * device error 2; a seq_len outside [0, 64 * max_pages], or in (0, T), is
 * treated as 0 and sets device error 3 (see mla_device_error).
 */
MLA_API mla_status_t mla_decode_paged(const mla_tensor_t *q, const mla_tensor_t *kv_cache,
                              const float *kv_scale, const mla_tensor_t *block_table,
                              const mla_tensor_t *seq_lens, int32_t n_splits, float sm_scale,
                              const mla_tensor_t *out, const mla_tensor_t *lse, void *stream);

/*
 * mla_merge_partials -- combine n_shards partial answers of the same rows by
 * their normalisers (section 1, DCP merge):
 *     lse = M + ln sum_s exp(lse_s - M),  M = max_s lse_s,
 *     out = sum_s exp(lse_s - lse) * partial_out_s.
 * Shards with lse_s = -inf weigh 0 and their partial_out values are ignored
 * (whatever bits they hold, NaN included); rows whose every shard is -inf get
 * out = 0, lse = -inf.
 *
 *   partial_out bf16 or fp32 [S, B, T, H, 512] (any rank >= 2 whose first dim
 *               is S and last dim 512), device, contiguous.
 *   partial_lse fp32 [S, B, T, H] (the same shape without the last dim).
 *   n_shards    S (must equal partial_out->shape[0]); 1 <= S <= 4096.
 *   out         bf16 [B, T, H, 512], device, contiguous.
 *   lse         fp32 [B, T, H], device, contiguous, or NULL.
 */
MLA_API mla_status_t mla_merge_partials(const mla_tensor_t *partial_out, const mla_tensor_t *partial_lse,
                                int32_t n_shards, const mla_tensor_t *out,
                                const mla_tensor_t *lse, void *stream);

/*
 * mla_decode_paged_noalloc -- the same operation as mla_decode_paged, with the
 * same arguments and results, for callers that must not have the library
 * allocate device memory: for example a serving engine that reserves nearly
 * all of the GPU's memory for its own page pool and accounts for every byte,
 * or a latency-critical decode step that must not pay for a first-use
 * allocation.  (The post has no counterpart; this is a property of the
 * library, not of the method.)
 *
 * The split partials live in one fixed device array of 8 MiB inside the
 * library (every GPU that loads the library holds it until the process
 * exits); this call never calls cudaMalloc, cudaMallocAsync or cudaFree.
 * With n_splits = 0 the automatic count (mla_auto_splits) is capped at the
 * largest count whose partials fit 8 MiB, down to 1 (no split, no scratch),
 * so the automatic mode always runs.  An explicit n_splits whose partials need
 * more than 8 MiB (see mla_decode_workspace_bytes) returns
 * MLA_ERR_UNSUPPORTED with a message and launches nothing.  Kernel family,
 * profile events and test hooks apply as for mla_decode_paged.  The library
 * does not survive cudaDeviceReset (the array's cached address would be
 * stale).  The first call on each device
 * looks up the array's device address with that device current; make that
 * first call before any stream capture.  All calls share the one array and
 * it keeps the previous call's contents (nothing in it needs to start at
 * zero): calls that overlap on the GPU, on any streams, race with each other.
 */
MLA_API mla_status_t mla_decode_paged_noalloc(const mla_tensor_t *q, const mla_tensor_t *kv_cache,
                                      const float *kv_scale, const mla_tensor_t *block_table,
                                      const mla_tensor_t *seq_lens, int32_t n_splits,
                                      float sm_scale, const mla_tensor_t *out,
                                      const mla_tensor_t *lse, void *stream);

/*
 * mla_append_latent -- write the new positions of a decode step into the
 * paged FP8 cache (the post's model section: each layer's compressed history
 * grows by one latent per new position; section 1: 576 FP8 bytes per
 * position, no per-position scale).
 *
 *   latent      bf16 [B, T, 576], device, contiguous, 16-byte aligned; the new
 *               latents (512 latent dims, then the 64 rotated positional dims)
 *               of T new positions per request.
 *   kv_scale    device pointer to the fp32 per-tensor scale of the cache.
 *   block_table i32 [B, max_pages], device, rows contiguous (as for decode).
 *   start_pos   i32 [B], device: position of latent[b, 0] in request b's
 *               history (its length before the append).
 *   kv_cache    e4m3fn [num_pages, 64, 576], device, contiguous, 16-byte
 *               aligned; written in place.
 *   stream      cudaStream_t as void*.
 *
 * Position p = start_pos[b] + t receives code[d] = e4m3fn(latent[b,t,d] /
 * kv_scale) -- one correctly rounded fp32 division, round to nearest even,
 * magnitudes beyond 448 saturate to +-448 (NaN stays NaN) -- in page
 * block_table[b][p / 64], row p % 64.  No other cache byte changes.  A decode
 * that follows on the same stream with seq_lens[b] = start_pos[b] + T sees
 * the new positions.  Rows whose position lies outside [0, max_pages * 64)
 * or whose page id lies outside [0, num_pages) are not written and set the
 * device error word (3 or 2; see mla_device_error).
 * Returns MLA_OK or an error status (nothing is launched on error); B*T = 0
 * is a no-op.  The call allocates nothing and never synchronises.
 */
MLA_API mla_status_t mla_append_latent(const mla_tensor_t *latent, const float *kv_scale,
                               const mla_tensor_t *block_table, const mla_tensor_t *start_pos,
                               const mla_tensor_t *kv_cache, void *stream);

/* The automatic split count used when n_splits == 0, from max_pages alone
 * (every request taken as max_pages long): the count that minimises the number
 * of waves of CTAs times (the partition length + a fixed 8 pages per CTA),
 * with at least 2 pages (128 positions) per partition.  A (request,
 * partition) unit takes one CTA of the 12-head tensor-core kernel for up to 16
 * rows, and ceil(H * T / 32) CTAs of the 32-row kernel beyond.  Partitions
 * never exceed 160 pages (10,240 positions), so that in a batch of mixed
 * lengths the longest request does not bound the call.
 * Pure host function; sm_count <= 0 means "query the current device". */
MLA_API int32_t mla_auto_splits(int32_t B, int32_t T, int32_t H, int32_t max_pages, int32_t sm_count);

/* The split count for a batch whose lengths the caller knows on the host (a
 * serving engine schedules them): pass the result as n_splits.  It replays
 * the launch on the host -- each CTA on the SM that frees first, one per SM,
 * a partition costing its pages at a fixed per-page time plus a fixed 8 pages
 * of set-up and epilogue -- and returns the count with the shortest finish
 * (ties: fewer partitions).  A unit of more than 16 rows takes ceil(H * T / 32)
 * CTAs of the 32-row tensor-core kernel, one after another; a unit of up to
 * 16 rows one CTA.  The CTAs run in launch order while they fit the SMs, and
 * otherwise (up to 1,024 requests) longest first -- full partitions, then the
 * partial ones by length, then those past each request's history at ~3/4
 * page each -- as the decode launches them.  Counts are tried up to 8
 * waves of full-length CTAs, and for units of up to 16 rows down to
 * partitions of 64 pages.  When host_seq_lens is NULL (or B is 0) it returns
 * mla_auto_splits(B, T, H, max_pages, sm_count).  A plan takes ~0.1-8 ms on
 * one host core (8 ms for 4,096 requests), so an engine plans once per batch.
 *   host_seq_lens  host pointer to the B lengths the decode will read from
 *                  seq_lens (values outside [0, 64 * max_pages] are clamped).
 *   max_pages      the block table's width, as passed to the decode.
 * Pure host function; sm_count <= 0 means "query the current device". */
MLA_API int32_t mla_plan_splits(int32_t B, int32_t T, int32_t H, const int32_t *host_seq_lens,
                        int32_t max_pages, int32_t sm_count);

/* Pages per partition for a given split count: ceil(max_pages / n_splits),
 * so that the partitions of a full-length request differ by at most one
 * page, except the last, which takes the remainder. */
MLA_API int32_t mla_split_chunk_pages(int32_t max_pages, int32_t n_splits);

/* Bytes of library scratch one mla_decode_paged call with these sizes uses
 * (0 when n_splits resolves to 1). */
MLA_API size_t mla_decode_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t n_splits);

/* Free the split scratch that calls captured in CUDA graphs used (on the
 * current device): the buffers kept when a stream's scratch grew, and the
 * live buffers of streams whose calls were captured (their next uncaptured
 * call allocates anew).  Call it only when no graph that captured a library
 * call on this device will be replayed again (e.g. after destroying them).
 * Synchronises the device (cudaFree). */
MLA_API mla_status_t mla_release_graph_scratch(void);

/* Select the kernel family for subsequent mla_decode_paged calls in this
 * process (all threads).  Returns the previous setting. */
MLA_API int32_t mla_set_impl(int32_t impl);

/* Kernel family (MLA_IMPL_SIMT or MLA_IMPL_TCGEN05) that the calling thread's
 * last successful mla_decode_paged call launched; 0 before any call. */
MLA_API int32_t mla_last_decode_impl(void);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device: 0 means no kernel reported an error.  Codes: 1 a bounded
 * wait timed out, 2 a page id out of range, 3 a seq_len out of range. */
MLA_API mla_status_t mla_device_error(int32_t *code, void *stream);

/* Benchmark instrumentation: the next mla_decode_paged call made by the
 * calling thread records ev_begin on its stream just before its split-KV
 * kernel and ev_end just after that kernel (before the split combine).  The
 * events are cudaEvent_t handles passed as void*; either may be NULL.  The
 * request is one-shot and thread-local; it changes nothing else. */
MLA_API mla_status_t mla_profile_next_decode(void *ev_begin, void *ev_end);

MLA_API const char *mla_status_string(mla_status_t status);
MLA_API const char *mla_last_error(void);   /* thread-local; "" when none */

#ifdef __cplusplus
}
#endif

#endif /* MLA_DECODE_H_ */
