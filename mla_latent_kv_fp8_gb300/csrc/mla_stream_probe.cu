// mla_stream_probe.cu -- benchmark instrumentation: the HBM ceiling of the
// decode's access pattern.
//
// Each CTA pulls its share of 36,864-byte cache pages (64 positions x 576
// bytes, at the page ids it is given) through TMA into a 4-deep shared-memory
// ring, one page per copy instruction, exactly as the tensor-core decode kernel
// does, and discards them: no arithmetic, no output.  Its time for a grid and
// page count is the floor that any kernel reading those pages this way meets,
// ramp-up and tail included.  Not part of the decode operation.
#include <mutex>

#include "mla_tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kProbeStages = 4;
constexpr int kProbePageBytes = kPage * kDqk;  // 36,864

struct ProbeSmem {
    alignas(1024) uint8_t slot[kProbeStages][kProbePageBytes];
    alignas(8) uint64_t full[kProbeStages];
    uint64_t empty[kProbeStages];
    int abort_flag;
    int issued;
    uint32_t sink;
};

// Thread 0 issues copies; thread 32 waits for each page, reads one byte of it
// and frees the slot.  A timeout on either side stops both (abort flag), and
// the CTA leaves only after every copy it issued has landed or the wait for it
// has run out.
__global__ void __launch_bounds__(64, 1)
    stream_pages_kernel(const __grid_constant__ CUtensorMap map, const int32_t* page_ids, int pages_per_cta,
                        int64_t num_pages, int* err) {
    extern __shared__ uint8_t smem_raw[];
    ProbeSmem& S = *reinterpret_cast<ProbeSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int32_t* ids = page_ids + static_cast<int64_t>(blockIdx.x) * pages_per_cta;
    if (tid == 0) {
        for (int s = 0; s < kProbeStages; ++s) {
            mbar_init(&S.full[s], 1);
            mbar_init(&S.empty[s], 1);
        }
        S.abort_flag = 0;
        S.issued = 0;
        S.sink = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int* abort = &S.abort_flag;
    if (tid == 0) {
        int i = 0;
        for (; i < pages_per_cta && !*abort; ++i) {
            const int s = i % kProbeStages;
            if (i >= kProbeStages && !wait_bounded(&S.empty[s], ((i / kProbeStages) & 1) ^ 1, abort, err)) break;
            int32_t pid = __ldg(ids + i);
            if (pid < 0 || pid >= num_pages) {
                atomicCAS(err, 0, kErrPageRange);
                pid = 0;
            }
            mbar_expect_tx(&S.full[s], kProbePageBytes);
            tma_load_page(smem_u32(S.slot[s]), &map, pid * kPage, &S.full[s]);
        }
        S.issued = i;
    } else if (tid == 32) {
        uint32_t acc = 0;
        for (int i = 0; i < pages_per_cta && !*abort; ++i) {
            const int s = i % kProbeStages;
            if (!wait_bounded(&S.full[s], (i / kProbeStages) & 1, abort, err)) break;
            acc += S.slot[s][i & 1023];
            mbar_arrive(&S.empty[s]);
        }
        *reinterpret_cast<volatile uint32_t*>(&S.sink) = acc;  // keeps the reads
    }
    __syncthreads();
    if (tid == 0 && *abort) {
        // Drain: every issued copy lands (or its wait runs out) before exit.
        // The abort flag is already set, so each wait is a plain deadline wait.
        const int n = S.issued;
        for (int i = n > kProbeStages ? n - kProbeStages : 0; i < n; ++i) {
            const uint64_t t0 = global_ns();
            while (!mbar_try_wait(&S.full[i % kProbeStages], (i / kProbeStages) & 1))
                if (global_ns() - t0 > kTimeoutNs) break;
        }
    }
}

}  // namespace

cudaError_t launch_stream_probe(const uint8_t* kv, int64_t num_pages, const int32_t* page_ids, int ctas,
                                int pages_per_cta, int* err, cudaStream_t stream) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(stream_pages_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(sizeof(ProbeSmem)) + 1024);
    });
    if (attr_err != cudaSuccess) return attr_err;
    // The decode kernel's whole-page view: {64-byte column, row, 64-byte chunk}.
    CUtensorMap map, map_box;
    cudaError_t e = encode_cache_maps(&map, &map_box, kv, num_pages);
    if (e != cudaSuccess) return e;
    stream_pages_kernel<<<ctas, 64, sizeof(ProbeSmem) + 1024, stream>>>(map, page_ids, pages_per_cta, num_pages,
                                                                         err);
    return cudaGetLastError();
}

}  // namespace mla
