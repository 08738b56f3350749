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

#include "../../include/mla_decode.h"
#include "mla_internal.cuh"

namespace mla {

mla_status_t internal_fail(mla_status_t st, const char* msg);
mla_status_t internal_cuda_fail(cudaError_t e, const char* what);
void internal_clear_error();
void internal_set_last_impl(int impl);
mla_status_t internal_device(int** err_word, int* sm_count);
mla_status_t internal_check_tensor(const mla_tensor_t* t, const char* name, int ndim, int dtype,
                                   bool need_contig, size_t align);
cudaError_t launch_tc_decode(const DecodeParams& p, cudaStream_t stream, bool* handled);

namespace {

// The fixed split scratch: fp32 partial outputs and log-sum-exps of every
// history partition.  Each GPU that loads the library holds it until exit.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device with that
// device current (in host code the symbol itself is only a host-side stand-in).
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

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_decode_paged_noalloc(const mla_tensor_t* q, const mla_tensor_t* kv_cache,
                                                 const float* kv_scale, const mla_tensor_t* block_table,
                                                 const mla_tensor_t* seq_lens, int32_t n_splits,
                                                 float sm_scale, const mla_tensor_t* out,
                                                 const mla_tensor_t* lse, void* stream) {
    internal_clear_error();
    mla_status_t st;
    if ((st = internal_check_tensor(q, "q", 4, MLA_DTYPE_BF16, true, 16)) != MLA_OK) return st;
    const int64_t B = q->shape[0], T = q->shape[1], H = q->shape[2];
    if (q->shape[3] != kDqk) return internal_fail(MLA_ERR_UNSUPPORTED, "q: last dim must be 576");
    if (T < 1 || H < 1) return internal_fail(MLA_ERR_INVALID_ARG, "q: T and H must be >= 1");
    if (H * T > kMaxRows) return internal_fail(MLA_ERR_UNSUPPORTED, "H*T exceeds 128");
    if ((st = internal_check_tensor(kv_cache, "kv_cache", 3, MLA_DTYPE_E4M3FN, true, 16)) != MLA_OK) return st;
    if (kv_cache->shape[1] != kPage || kv_cache->shape[2] != kDqk)
        return internal_fail(MLA_ERR_UNSUPPORTED, "kv_cache: must be [num_pages, 64, 576]");
    if (!kv_scale) return internal_fail(MLA_ERR_INVALID_ARG, "kv_scale: null pointer");
    if ((st = internal_check_tensor(block_table, "block_table", 2, MLA_DTYPE_I32, false, 4)) != MLA_OK) return st;
    if (block_table->shape[0] != B) return internal_fail(MLA_ERR_INVALID_ARG, "block_table: first dim must be B");
    const int64_t max_pages = block_table->shape[1];
    if (block_table->stride[1] != 1 || block_table->stride[0] < max_pages)
        return internal_fail(MLA_ERR_UNSUPPORTED, "block_table: rows must be contiguous");
    if ((st = internal_check_tensor(seq_lens, "seq_lens", 1, MLA_DTYPE_I32, true, 4)) != MLA_OK) return st;
    if (seq_lens->shape[0] != B) return internal_fail(MLA_ERR_INVALID_ARG, "seq_lens: must have B entries");
    if ((st = internal_check_tensor(out, "out", 4, MLA_DTYPE_BF16, true, 16)) != MLA_OK) return st;
    if (out->shape[0] != B || out->shape[1] != T || out->shape[2] != H || out->shape[3] != kDv)
        return internal_fail(MLA_ERR_INVALID_ARG, "out: must be [B, T, H, 512]");
    if (lse) {
        if ((st = internal_check_tensor(lse, "lse", 3, MLA_DTYPE_F32, true, 4)) != MLA_OK) return st;
        if (lse->shape[0] != B || lse->shape[1] != T || lse->shape[2] != H)
            return internal_fail(MLA_ERR_INVALID_ARG, "lse: must be [B, T, H]");
    }
    if (n_splits < 0) return internal_fail(MLA_ERR_INVALID_ARG, "n_splits must be >= 0");
    if (max_pages < 1 && B > 0) return internal_fail(MLA_ERR_INVALID_ARG, "block_table: needs >= 1 column");
    if (max_pages > (1 << 24)) return internal_fail(MLA_ERR_UNSUPPORTED, "block_table: too many pages");
    if (B > 65535) return internal_fail(MLA_ERR_UNSUPPORTED, "B > 65535");
    if (B == 0) return MLA_OK;

    int* err_word = nullptr;
    int sm_count = 0;
    if ((st = internal_device(&err_word, &sm_count)) != MLA_OK) return st;
    void* scratch = nullptr;
    if ((st = scratch_address(&scratch)) != MLA_OK) return st;

    const int32_t req = n_splits > 0 ? n_splits
                                     : mla_auto_splits((int32_t)B, (int32_t)T, (int32_t)H,
                                                       (int32_t)max_pages, sm_count);
    const int32_t chunk = mla_split_chunk_pages((int32_t)max_pages, req);
    const int32_t n_eff = (int32_t)cdiv(max_pages, chunk);
    const size_t need = mla_decode_workspace_bytes((int32_t)B, (int32_t)T, (int32_t)H, n_eff);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "split scratch of %zu bytes exceeds the fixed %zu-byte array of the no-allocation "
                 "entry point; pass fewer n_splits or use mla_decode_paged",
                 need, kNoAllocScratchBytes);
        return internal_fail(MLA_ERR_UNSUPPORTED, msg);
    }

    DecodeParams p{};
    p.q = static_cast<const uint16_t*>(q->data);
    p.kv = static_cast<const uint8_t*>(kv_cache->data);
    p.kv_scale = kv_scale;
    p.block_table = static_cast<const int32_t*>(block_table->data);
    p.seq_lens = static_cast<const int32_t*>(seq_lens->data);
    p.bt_stride = block_table->stride[0];
    p.num_pages = kv_cache->shape[0];
    p.B = (int)B;
    p.T = (int)T;
    p.H = (int)H;
    p.max_pages = (int)max_pages;
    p.n_splits = n_eff;
    p.chunk_pages = chunk;
    p.sm_scale_log2 = sm_scale * kLog2e;
    p.out = static_cast<uint16_t*>(out->data);
    p.lse = lse ? static_cast<float*>(lse->data) : nullptr;
    p.err = err_word;
    if (n_eff > 1) {
        const size_t out_bytes = (size_t)n_eff * B * T * H * kDv * sizeof(float);
        p.part_out = static_cast<float*>(scratch);
        p.part_lse = reinterpret_cast<float*>(static_cast<char*>(scratch) + ((out_bytes + 255) & ~size_t(255)));
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool handled = false;
    cudaError_t e = launch_tc_decode(p, s, &handled);
    if (e != cudaSuccess) return internal_cuda_fail(e, "tcgen05 decode launch");
    if (!handled) {
        e = launch_simt_decode(p, s);
        if (e != cudaSuccess) return internal_cuda_fail(e, "decode launch");
    }
    internal_set_last_impl(handled ? MLA_IMPL_TCGEN05 : MLA_IMPL_SIMT);
    if (n_eff > 1) {
        MergeParams m{};
        m.part_out = p.part_out;
        m.part_lse = p.part_lse;
        m.S = n_eff;
        m.rows = B * T * H;
        m.in_bf16 = 0;
        m.out = p.out;
        m.lse = p.lse;
        m.pdl = 1;
        e = launch_merge(m, s);
        if (e != cudaSuccess) return internal_cuda_fail(e, "split combine launch");
    }
    return MLA_OK;
}
