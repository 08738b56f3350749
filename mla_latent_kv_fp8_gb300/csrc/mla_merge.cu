// mla_merge.cu -- merge kernels for partial attention answers (the device
// code is in mla_merge_dev.cuh).
//
// "Kimi K3 on AMD Instinct MI355X" post, section 1 (DCP paragraph): each
// partial answer over a part of the history carries normalisation information
// so that the merge weighs the parts correctly.  With lse_s the natural-log
// normaliser of part s:
//     lse = M + ln sum_s exp(lse_s - M),   M = max_s lse_s
//     out = sum_s exp(lse_s - lse) * o_s
// Parts with lse_s = -inf weigh exactly 0; their values are never multiplied.
//
// Three kernels:
//   * many rows (>= 1,216; >= 256 for bf16 parts) and few parts (S <= 32):
//     one warp per whole row, 16 dims per lane, 16-byte loads of four parts
//     per round in flight, the first round issued with the normaliser loads --
//     the HBM-bound DCP merge and the split combine of large batches;
//   * few parts (S <= 32), fewer rows: one warp per (row, 64 value dims); lane s holds
//     lse_s, the normaliser is a shuffle reduction, each lane loads 2 dims of
//     every part, all parts in one round;
//   * many parts (S > 32, the in-GPU split combine of one long request): one
//     CTA per (row, 32 value dims); the eight warps split the parts, each lane
//     owns one dim; the values of the first 256 parts load in the same round
//     as the normalisers, and the warps' sums meet in shared memory.
#include "mla_merge_dev.cuh"

namespace mla {
namespace {

using namespace mergedev;

// Launched as a programmatic dependent of the decode kernel (pdl): wait for
// its partials, and let the next kernel's CTAs be scheduled meanwhile (the
// decode kernel waits for this one before reading anything).
__device__ __forceinline__ void wait_for_producer(const MergeParams& p) {
    if (p.pdl) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

template <bool kBf16In>
__global__ void __launch_bounds__(256) merge_warp_kernel(MergeParams p) {
    wait_for_producer(p);
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (gw >= p.rows * 8) return;
    merge_warp<kBf16In>(p, gw >> 3, static_cast<int>(gw & 7), threadIdx.x & 31);
}

template <bool kBf16In>
__global__ void __launch_bounds__(256, kBf16In ? 3 : 2) merge_row_kernel(MergeParams p) {
    wait_for_producer(p);
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= p.rows) return;
    merge_row<kBf16In>(p, row, threadIdx.x & 31);
}

template <bool kBf16In>
__global__ void __launch_bounds__(256) merge_cta_kernel(MergeParams p) {
    wait_for_producer(p);
    __shared__ CtaScratch sh;
    merge_cta<kBf16In>(p, blockIdx.x >> 4, static_cast<int>(blockIdx.x & 15), threadIdx.x, sh,
                       [] { __syncthreads(); });
}

template <typename K>
cudaError_t launch_with_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t stream,
                            const MergeParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Rows from which the one-warp-per-row kernel takes a merge of S <= 32 parts.
// fp32 parts (the decode's own split combine): one 8-row CTA per SM of a GB300;
// below that the (row, 64 dims) warps finish sooner inside a decode step (768
// rows x 14 parts: 179.7 vs 180.8 us per verify step; 96 rows x 19 parts: 3.4
// vs 10.5 us alone).  bf16 parts (answers of DCP shards) move only 4 bytes per
// lane and part on the warp path, so the row kernel wins from far fewer rows
// (768 rows x 8 parts: 4.7 vs 10.3 us).
constexpr int64_t kRowPathMinRows = 8 * 152;
constexpr int64_t kRowPathMinRowsBf16 = 256;

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
    if (p.S <= 32 && p.rows >= (p.in_bf16 ? kRowPathMinRowsBf16 : kRowPathMinRows)) {
        // enough rows for a full wave of one-warp-per-row CTAs: stream whole rows
        const dim3 grid((unsigned)((p.rows + 7) / 8));
        return p.in_bf16 ? launch_with_pdl(merge_row_kernel<true>, grid, dim3(256), stream, p)
                         : launch_with_pdl(merge_row_kernel<false>, grid, dim3(256), stream, p);
    }
    if (p.S <= 32) {
        const int64_t warps = p.rows * 8;
        const dim3 grid((unsigned)((warps + 7) / 8));
        return p.in_bf16 ? launch_with_pdl(merge_warp_kernel<true>, grid, dim3(256), stream, p)
                         : launch_with_pdl(merge_warp_kernel<false>, grid, dim3(256), stream, p);
    }
    const dim3 grid((unsigned)(p.rows * 16));
    return p.in_bf16 ? launch_with_pdl(merge_cta_kernel<true>, grid, dim3(256), stream, p)
                     : launch_with_pdl(merge_cta_kernel<false>, grid, dim3(256), stream, p);
}

}  // namespace mla
