// mla_tc.cu -- tcgen05 tensor-core split-KV MLA decode (sm_103a).
#include "mla_internal.cuh"

namespace mla {

cudaError_t launch_tc_decode(const DecodeParams& p, cudaStream_t stream, bool* handled) {
    (void)p;
    (void)stream;
    *handled = false;
    return cudaSuccess;
}

}  // namespace mla
