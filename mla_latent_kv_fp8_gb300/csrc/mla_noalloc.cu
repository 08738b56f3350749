// mla_noalloc.cu -- mla_decode_paged_noalloc: the split-KV decode with its
// split scratch in a fixed, statically allocated device array, for callers
// that must not have the library allocate device memory.
//
// Who needs it: a serving engine that reserves (nearly) all of the GPU's memory
// up front for its own page pool and accounts for every byte itself, where an
// allocation made inside a library could fail or fragment that pool; and code
// on a latency-critical path that must not pay for a first-use allocation in
// the middle of a decode step.  Such callers pass inputs and outputs as usual
// and this entry point uses no cudaMalloc, cudaMallocAsync or cudaFree at all.
#include <cstdio>
#include <mutex>

#include "mla_host.h"

namespace mla {
namespace {

// The fixed split scratch: fp32 partial outputs and log-sum-exps of every
// history partition.  Each GPU that loads the library holds it until exit.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (in host code the symbol itself is only a host-side
// stand-in).  The library does not survive cudaDeviceReset: a reset rebuilds
// the context and its module, and the cached address would be stale.
std::mutex g_mu;
void* g_scratch_ptr[64];

mla_status_t scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return internal_cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return internal_fail(MLA_ERR_UNSUPPORTED, "device ordinal >= 64");
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return internal_cuda_fail(e, "cudaGetSymbolAddress(no-allocation scratch)");
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return MLA_OK;
}

// The largest partition count whose partials fit the array (at least 1: an
// unsplit call needs no scratch).
int32_t max_splits_that_fit(int64_t rows) {
    const int64_t per_split = rows * (kDv + 1) * (int64_t)sizeof(float);
    int64_t n = (int64_t)kNoAllocScratchBytes / per_split;
    if (n > 4096) n = 4096;
    while (n > 1 && mla_decode_workspace_bytes(1, 1, (int32_t)rows, (int32_t)n) > kNoAllocScratchBytes) --n;
    return n < 1 ? 1 : (int32_t)n;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_decode_paged_noalloc(const mla_tensor_t* q, const mla_tensor_t* kv_cache,
                                                 const float* kv_scale, const mla_tensor_t* block_table,
                                                 const mla_tensor_t* seq_lens, int32_t n_splits,
                                                 float sm_scale, const mla_tensor_t* out,
                                                 const mla_tensor_t* lse, void* stream) {
    internal_clear_error();
    // n_splits = 0: the automatic count, capped to what the array holds
    int32_t cap = 1;
    if (q && q->ndim == 4 && q->shape[0] > 0 && q->shape[1] > 0 && q->shape[2] > 0)
        cap = max_splits_that_fit(q->shape[0] * q->shape[1] * q->shape[2]);
    DecodeParams p{};
    bool empty = false;
    mla_status_t st = internal_prepare_decode(q, kv_cache, kv_scale, block_table, seq_lens, n_splits, cap,
                                              sm_scale, out, lse, &p, &empty);
    if (st != MLA_OK || empty) return st;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != MLA_OK) return st;
    const size_t need = mla_decode_workspace_bytes(p.B, p.T, p.H, p.n_splits);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "split scratch of %zu bytes exceeds the fixed %zu-byte array of the no-allocation "
                 "entry point; pass fewer n_splits (or 0) or use mla_decode_paged",
                 need, kNoAllocScratchBytes);
        return internal_fail(MLA_ERR_UNSUPPORTED, msg);
    }
    if (p.n_splits > 1) internal_carve_scratch(p, scratch);
    return internal_launch_decode(p, static_cast<cudaStream_t>(stream));
}
