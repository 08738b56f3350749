// mla_host.h -- host-side helpers shared by the library's entry-point
// translation units (mla_api.cu, mla_noalloc.cu, mla_append.cu).  Internal:
// nothing here is exported (the library is built with hidden visibility).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

#include "../../include/mla_decode.h"
#include "mla_internal.cuh"

namespace mla {

// Error reporting: set the calling thread's last-error message and return st.
mla_status_t internal_fail(mla_status_t st, const char* msg);
mla_status_t internal_cuda_fail(cudaError_t e, const char* what);
void internal_clear_error();

// Facts of the current device, filled once per device: its device error word
// and SM count.
mla_status_t internal_device(int** err_word, int* sm_count);

mla_status_t internal_check_tensor(const mla_tensor_t* t, const char* name, int ndim, int dtype,
                                   bool need_contig, size_t align);

// Checks the arguments of a decode call (mla_decode_paged and
// mla_decode_paged_noalloc take the same ones) and fills *p with everything
// but the split scratch: shapes, pointers, the resolved partition count
// (p->n_splits, from n_splits or, when it is 0, from auto_splits) and chunk.
// *empty is set when B == 0 (nothing to launch).  Nothing is launched.
mla_status_t internal_prepare_decode(const mla_tensor_t* q, const mla_tensor_t* kv_cache, const float* kv_scale,
                                     const mla_tensor_t* block_table, const mla_tensor_t* seq_lens,
                                     int32_t n_splits, int32_t auto_splits_cap, float sm_scale,
                                     const mla_tensor_t* out, const mla_tensor_t* lse, DecodeParams* p,
                                     bool* empty);

// Points p.part_out and p.part_lse (the fp32 partials of the split-KV kernel)
// into split scratch of at least mla_decode_workspace_bytes(...) bytes.
void internal_carve_scratch(DecodeParams& p, void* ws);

// Launches a prepared decode on `stream`: the split-KV kernel of the family
// mla_set_impl selected (with the calling thread's profile events and test
// hooks), then, when p.n_splits > 1, the split combine over p.part_out /
// p.part_lse, which the caller has pointed at enough scratch.
mla_status_t internal_launch_decode(DecodeParams& p, cudaStream_t stream);

}  // namespace mla
