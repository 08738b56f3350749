// mla_internal.cuh -- parameter blocks and launchers shared by the kernels and
// the host API of the MLA decode library (internal; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

constexpr int kPage = 64;        // positions per page
constexpr int kDqk = 576;        // latent + positional dims per position
constexpr int kDv = 512;         // value dims (the latent)
constexpr int kMaxRows = 128;    // H * T rows per request handled by one call
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Device error codes (written to the library's device error word).
enum DeviceError : int {
    kErrNone = 0,
    kErrWaitTimeout = 1,
    kErrPageRange = 2,
    kErrSeqRange = 3,
};

// One decode call, as seen by every decode kernel.
struct DecodeParams {
    const uint16_t* q;          // bf16 bits [B][T][H][576]
    const uint8_t* kv;          // e4m3fn codes [num_pages][64][576]
    const float* kv_scale;      // device scalar
    const int32_t* block_table; // [B][bt_stride]
    const int32_t* seq_lens;    // [B]
    int64_t bt_stride;
    int64_t num_pages;
    int B, T, H;
    int max_pages;              // block_table width
    int n_splits;               // partitions per request (>= 1)
    int chunk_pages;            // pages per partition (even)
    float sm_scale_log2;        // sm_scale * log2(e)
    // n_splits == 1: final outputs
    uint16_t* out;              // bf16 [B][T][H][512]
    float* lse;                 // [B][T][H] or null
    // n_splits > 1: fp32 partials [n_splits][B][T][H][512] and [n_splits][B][T][H]
    float* part_out;
    float* part_lse;
    int* err;                   // device error word
    int test_stall_copies;      // failure-detection tests only: issue no page copies
    // tests only (null otherwise): [0] += 1 each time an attention warpgroup
    // rescales its accumulated output tile after a reference move past its
    // first page, [1] += 1 for every reference move
    int* test_counts;
    // tcgen05 kernel for more than 16 rows: CTAs per (partition, request) and
    // rows each (the last CTA may have fewer)
    int row_ctas;
    int rows_per_cta;
    // tcgen05 kernels: a moved reference maximum sits this far (log2 units)
    // below the page maximum (set per launch from the partition length)
    float ref_shift;
    // 12-head tcgen05 kernel, more units than SMs: the longest-first order of
    // the units, {b * n_splits + split, seq_len} per launch index (split scratch)
    int2* lpt_order;
};

struct MergeParams {
    const void* part_out;       // [S][rows][512], fp32 or bf16
    const float* part_lse;      // [S][rows]
    int S;
    int64_t rows;
    int in_bf16;                // 1: part_out is bf16
    uint16_t* out;              // bf16 [rows][512]
    float* lse;                 // [rows] or null
    int pdl;                    // launched as a programmatic dependent of the producer
    // The split combine of a decode call sets these (null seq_lens otherwise):
    // part s of request b's rows holds an answer only for the partitions its
    // history reaches, s < ceil(ceil(L_b / 64) / chunk_pages); the others were
    // not written by this call and count as empty, whatever the scratch holds.
    const int32_t* seq_lens;    // [rows / rows_per_req], device
    int rows_per_req;           // H * T
    int T;
    int chunk_pages;
    int max_pages;              // lengths beyond max_pages * 64 (or below T) count as 0
};

cudaError_t launch_simt_decode(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_tc_decode(const DecodeParams& p, cudaStream_t stream, bool* handled);
cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream);
cudaError_t launch_stream_probe(const uint8_t* kv, int64_t num_pages, const int32_t* page_ids, int ctas,
                                int pages_per_cta, int* err, cudaStream_t stream);

}  // namespace mla

// ---------------------------------------------------------------- host side
// Host-only declarations that need the driver API types.
#include <cuda.h>

namespace mla {

// The two TMA views of the cache that the tensor-core kernels copy pages
// through: map3 moves a whole 64-position page per copy, map2 one 64 x 64-byte
// box of it (both 64-byte swizzled).
cudaError_t encode_cache_maps(CUtensorMap* map3, CUtensorMap* map2, const uint8_t* kv, int64_t num_pages);

}  // namespace mla
