// mla_append.cu -- mla_append_latent: quantise the new latents of a decode
// step to E4M3FN and write them into their paged cache slots.
//
// Method: "Kimi K3 on AMD Instinct MI355X" post -- model section (every MLA
// layer's compressed history grows by one 576-wide latent per new position),
// section 1 "Cache" (576 FP8 bytes per position and layer, no per-position
// scale bytes), benchmark section (FP8 KV).  The code of each value is
// e4m3fn(x / kv_scale): one correctly rounded binary32 division, then round to
// nearest even with saturation to +-448 (cvt.rn.satfinite).
//
// One CTA of 72 threads per new position: each thread reads 16 bytes (8 bf16
// values) and writes 8 code bytes, so a position's 1,152 input bytes and 576
// output bytes move as fully coalesced 16- and 8-byte accesses.  The work is a
// few KB per step; the kernel is launch-bound by design.
#include <cuda_fp8.h>

#include "mla_host.h"

namespace mla {

namespace {

constexpr int kAppendThreads = kDqk / 8;  // 72: 8 values each

__global__ void __launch_bounds__(kAppendThreads)
    append_latent_kernel(const uint16_t* __restrict__ latent, int T, const float* __restrict__ kv_scale,
                         const int32_t* __restrict__ block_table, int64_t bt_stride, int max_pages,
                         const int32_t* __restrict__ start_pos, uint8_t* __restrict__ kv, int64_t num_pages,
                         int* err) {
    const int64_t row = blockIdx.x;  // b * T + t
    const int b = static_cast<int>(row / T), t = static_cast<int>(row % T);
    const int lane = threadIdx.x;
    const int64_t pos = static_cast<int64_t>(__ldg(start_pos + b)) + t;
    if (pos < 0 || pos >= static_cast<int64_t>(max_pages) * kPage) {
        if (lane == 0) atomicCAS(err, 0, kErrSeqRange);
        return;
    }
    const int32_t page = __ldg(block_table + b * bt_stride + pos / kPage);
    if (page < 0 || page >= num_pages) {
        if (lane == 0) atomicCAS(err, 0, kErrPageRange);
        return;
    }
    const float s = __ldg(kv_scale);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(latent + row * kDqk) + lane);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t code[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float x0 = __fdiv_rn(__uint_as_float(w[j] << 16), s);          // element 2j
        const float x1 = __fdiv_rn(__uint_as_float(w[j] & 0xffff0000u), s);  // element 2j + 1
        const uint32_t c = static_cast<uint32_t>(
            __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3));
        code[j >> 1] |= (c & 0xffffu) << (16 * (j & 1));
    }
    uint8_t* dst = kv + (static_cast<int64_t>(page) * kPage + pos % kPage) * kDqk;
    reinterpret_cast<uint2*>(dst)[lane] = make_uint2(code[0], code[1]);
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status_t mla_append_latent(const mla_tensor_t* latent, const float* kv_scale,
                                          const mla_tensor_t* block_table, const mla_tensor_t* start_pos,
                                          const mla_tensor_t* kv_cache, void* stream) {
    internal_clear_error();
    mla_status_t st;
    if ((st = internal_check_tensor(latent, "latent", 3, MLA_DTYPE_BF16, true, 16)) != MLA_OK) return st;
    const int64_t B = latent->shape[0], T = latent->shape[1];
    if (latent->shape[2] != kDqk) return internal_fail(MLA_ERR_UNSUPPORTED, "latent: last dim must be 576");
    if (!kv_scale) return internal_fail(MLA_ERR_INVALID_ARG, "kv_scale: null pointer");
    if ((st = internal_check_tensor(block_table, "block_table", 2, MLA_DTYPE_I32, false, 4)) != MLA_OK) return st;
    if (block_table->shape[0] != B) return internal_fail(MLA_ERR_INVALID_ARG, "block_table: first dim must be B");
    const int64_t max_pages = block_table->shape[1];
    if (block_table->stride[1] != 1 || block_table->stride[0] < max_pages)
        return internal_fail(MLA_ERR_UNSUPPORTED, "block_table: rows must be contiguous");
    if ((st = internal_check_tensor(start_pos, "start_pos", 1, MLA_DTYPE_I32, true, 4)) != MLA_OK) return st;
    if (start_pos->shape[0] != B) return internal_fail(MLA_ERR_INVALID_ARG, "start_pos: must have B entries");
    if ((st = internal_check_tensor(kv_cache, "kv_cache", 3, MLA_DTYPE_E4M3FN, true, 16)) != MLA_OK) return st;
    if (kv_cache->shape[1] != kPage || kv_cache->shape[2] != kDqk)
        return internal_fail(MLA_ERR_UNSUPPORTED, "kv_cache: must be [num_pages, 64, 576]");
    if (max_pages > (1 << 24)) return internal_fail(MLA_ERR_UNSUPPORTED, "block_table: too many pages");
    if (B * T == 0) return MLA_OK;
    if (B * T > (int64_t(1) << 31) - 1) return internal_fail(MLA_ERR_UNSUPPORTED, "B * T >= 2^31");
    int* err_word = nullptr;
    int sm_count = 0;
    if ((st = internal_device(&err_word, &sm_count)) != MLA_OK) return st;
    append_latent_kernel<<<static_cast<unsigned>(B * T), kAppendThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t*>(latent->data), static_cast<int>(T), kv_scale,
        static_cast<const int32_t*>(block_table->data), block_table->stride[0], static_cast<int>(max_pages),
        static_cast<const int32_t*>(start_pos->data), static_cast<uint8_t*>(kv_cache->data), kv_cache->shape[0],
        err_word);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return internal_cuda_fail(e, "append launch");
    return MLA_OK;
}
