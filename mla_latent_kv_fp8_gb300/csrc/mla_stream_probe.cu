// mla_stream_probe.cu -- benchmark instrumentation: the HBM ceiling of the
// decode's access pattern.
//
// Each CTA pulls its share of 36,864-byte cache pages (64 positions x 576
// bytes, at the page ids it is given) through TMA into a 4-deep shared-memory
// ring, one page per copy instruction, exactly as the tensor-core decode kernel
// does, and discards them: no arithmetic, no output.  Its time for a grid and
// page count is the floor that any kernel reading those pages this way meets,
// ramp-up and tail included.  Not part of the decode operation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kProbeStages = 4;
constexpr int kProbePageBytes = kPage * kDqk;  // 36,864
constexpr uint64_t kProbeTimeoutNs = 2000000000ull;

struct ProbeSmem {
    alignas(1024) uint8_t slot[kProbeStages][kProbePageBytes];
    alignas(8) uint64_t full[kProbeStages];
    uint64_t empty[kProbeStages];
};

__device__ __forceinline__ uint32_t probe_smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t probe_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait on an mbarrier phase; false (and device error 1) on timeout.
__device__ __forceinline__ bool probe_wait(uint64_t* bar, uint32_t parity, int* err) {
    const uint64_t t0 = probe_ns();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(probe_smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (probe_ns() - t0 > kProbeTimeoutNs) {
            atomicCAS(err, 0, kErrWaitTimeout);
            return false;
        }
    }
}

// Thread 0 issues copies; thread 32 waits for each page, touches one byte of
// it and frees the slot.  A timeout on either side stops both (abort flag),
// and the CTA leaves only after every copy it issued has landed or the wait
// for it has run out.
__global__ void __launch_bounds__(64, 1)
    stream_pages_kernel(const __grid_constant__ CUtensorMap map, const int32_t* page_ids, int pages_per_cta,
                        int64_t num_pages, int* err) {
    extern __shared__ uint8_t smem_raw[];
    ProbeSmem& S = *reinterpret_cast<ProbeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ int abort_flag;
    __shared__ int issued_count;
    __shared__ uint32_t touched;
    const int tid = threadIdx.x;
    const int32_t* ids = page_ids + static_cast<int64_t>(blockIdx.x) * pages_per_cta;
    if (tid == 0) {
        for (int s = 0; s < kProbeStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(probe_smem_u32(&S.full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(probe_smem_u32(&S.empty[s])));
        }
        abort_flag = 0;
        issued_count = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort = &abort_flag;
    if (tid == 0) {
        int i = 0;
        for (; i < pages_per_cta && !*abort; ++i) {
            const int s = i % kProbeStages;
            if (i >= kProbeStages && !probe_wait(&S.empty[s], ((i / kProbeStages) & 1) ^ 1, err)) {
                *abort = 1;
                break;
            }
            int32_t pid = __ldg(ids + i);
            if (pid < 0 || pid >= num_pages) {
                atomicCAS(err, 0, kErrPageRange);
                pid = 0;
            }
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(probe_smem_u32(&S.full[s])),
                         "r"(kProbePageBytes)
                         : "memory");
            asm volatile(
                "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
                "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(probe_smem_u32(S.slot[s])),
                "l"(reinterpret_cast<uint64_t>(&map)), "r"(0), "r"(pid * kPage), "r"(0),
                "r"(probe_smem_u32(&S.full[s]))
                : "memory");
        }
        issued_count = i;
    } else if (tid == 32) {
        uint32_t acc = 0;
        for (int i = 0; i < pages_per_cta && !*abort; ++i) {
            const int s = i % kProbeStages;
            if (!probe_wait(&S.full[s], (i / kProbeStages) & 1, err)) {
                *abort = 1;
                break;
            }
            acc += S.slot[s][i & 1023];
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(probe_smem_u32(&S.empty[s])) : "memory");
        }
        *reinterpret_cast<volatile uint32_t*>(&touched) = acc;  // keeps the touches
    }
    __syncthreads();
    if (tid == 0 && *abort) {
        // Drain: every issued copy lands (or its wait runs out) before exit.
        const int n = issued_count;
        for (int i = n > kProbeStages ? n - kProbeStages : 0; i < n; ++i)
            probe_wait(&S.full[i % kProbeStages], (i / kProbeStages) & 1, err);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 probe_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    });
    return fn;
}

}  // namespace

cudaError_t launch_stream_probe(const uint8_t* kv, int64_t num_pages, const int32_t* page_ids, int ctas,
                                int pages_per_cta, int* err, cudaStream_t stream) {
    auto fn = probe_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(stream_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(sizeof(ProbeSmem)) + 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // The decode kernel's whole-page view: {64-byte column, row, 64-byte chunk}.
    CUtensorMap map;
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(num_pages * kPage), static_cast<cuuint64_t>(kDqk / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(kDqk), 64};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kPage), static_cast<cuuint32_t>(kDqk / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(kv), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    stream_pages_kernel<<<ctas, 64, sizeof(ProbeSmem) + 1024, stream>>>(map, page_ids, pages_per_cta, num_pages,
                                                                         err);
    return cudaGetLastError();
}

}  // namespace mla
