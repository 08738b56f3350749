// mla_merge.cu -- merge of partial attention answers by their log-sum-exp.
//
// "Kimi K3 on AMD Instinct MI355X" post, section 1 (DCP paragraph): each
// partial answer over a part of the history carries normalisation information
// so that the merge weighs the parts correctly.  With lse_s the natural-log
// normaliser of part s:
//     lse = M + ln sum_s exp(lse_s - M),   M = max_s lse_s
//     out = sum_s exp(lse_s - lse) * o_s
// Parts with lse_s = -inf weigh exactly 0 and are not read.
//
// Two kernels:
//   * few parts (S <= 32): one warp per (row, 64 value dims); lane s holds
//     lse_s, the normaliser is a shuffle reduction, each lane loads 2 dims of
//     every part, all parts in one round;
//   * many parts (S > 32, the in-GPU split combine of one long request): one
//     CTA per (row, 32 value dims); the eight warps split the parts, each lane
//     owns one dim, and the warps' sums meet in shared memory.
#include <cuda_bf16.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Launched as a programmatic dependent of the decode kernel (pdl): wait for
// its partials, and let the next kernel's CTAs be scheduled meanwhile (the
// decode kernel waits for this one before reading anything).
__device__ __forceinline__ void wait_for_producer(int pdl) {
    if (pdl) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

template <bool kBf16In>
__device__ __forceinline__ float load1(const void* base, int64_t idx) {
    if constexpr (kBf16In) {
        return __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16);
    } else {
        return static_cast<const float*>(base)[idx];
    }
}

template <bool kBf16In>
__device__ __forceinline__ float2 load2(const void* base, int64_t idx) {
    if constexpr (kBf16In) {
        const uint32_t raw = *reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(base) + idx);
        return make_float2(__uint_as_float(raw << 16), __uint_as_float(raw & 0xffff0000u));
    } else {
        return *reinterpret_cast<const float2*>(static_cast<const float*>(base) + idx);
    }
}

// One warp per (row, 64 value dims); lane s holds lse_s, each lane owns two
// dims.  Every part's two values are loaded in a single round (all loads in
// flight before the first product), so the kernel costs two memory latencies:
// the normalisers, then the values.
template <bool kBf16In>
__global__ void __launch_bounds__(256) merge_warp_kernel(MergeParams p) {
    wait_for_producer(p.pdl);
    const int lane = threadIdx.x & 31;
    const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (gw >= p.rows * 8) return;
    const int64_t row = gw >> 3;
    const int chunk = (int)(gw & 7);
    const int64_t col = (int64_t)chunk * 64 + lane * 2;

    const float ls = (lane < p.S) ? p.part_lse[(int64_t)lane * p.rows + row] : -INFINITY;
    const float M = warp_max(ls);
    uint16_t* dst = p.out + row * kDv + col;
    if (M == -INFINITY) {
        *reinterpret_cast<uint32_t*>(dst) = 0u;
        if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = -INFINITY;
        return;
    }
    const float e = (ls == -INFINITY) ? 0.f : exp2f((ls - M) * kLog2e);
    const float sum = warp_sum(e);
    const float w = e / sum;  // lanes >= S: 0
    float ws[32];
    float2 v[32];
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        ws[s] = __shfl_sync(0xffffffffu, w, s);
        v[s] = ws[s] != 0.f ? load2<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col)
                            : make_float2(0.f, 0.f);
    }
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 32; ++s) {
        acc.x = fmaf(ws[s], v[s].x, acc.x);
        acc.y = fmaf(ws[s], v[s].y, acc.y);
    }
    __nv_bfloat162 o = __floats2bfloat162_rn(acc.x, acc.y);
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<uint32_t*>(&o);
    if (chunk == 0 && lane == 0 && p.lse) p.lse[row] = M + logf(sum);
}

template <bool kBf16In>
__global__ void __launch_bounds__(256) merge_cta_kernel(MergeParams p) {
    wait_for_producer(p.pdl);
    __shared__ float red[8];
    __shared__ float part[8][32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t row = blockIdx.x >> 4;
    const int col = (blockIdx.x & 15) * 32 + lane;

    float mx = -INFINITY;
    for (int s = tid; s < p.S; s += 256) mx = fmaxf(mx, p.part_lse[(int64_t)s * p.rows + row]);
    mx = warp_max(mx);
    if (lane == 0) red[wid] = mx;
    __syncthreads();
    float M = red[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) M = fmaxf(M, red[i]);
    __syncthreads();
    if (M == -INFINITY) {
        if (wid == 0) {
            p.out[row * kDv + col] = 0;
            if (blockIdx.x % 16 == 0 && lane == 0 && p.lse) p.lse[row] = -INFINITY;
        }
        return;
    }
    float sm = 0.f;
    for (int s = tid; s < p.S; s += 256) {
        const float ls = p.part_lse[(int64_t)s * p.rows + row];
        if (ls != -INFINITY) sm += exp2f((ls - M) * kLog2e);
    }
    sm = warp_sum(sm);
    if (lane == 0) red[wid] = sm;
    __syncthreads();
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) sum += red[i];
    const float lse_out = M + logf(sum);

    // Warp wid takes parts wid, wid + 8, ...; eight of them per round, with
    // every load of the round issued before the first product.  An empty
    // part's output was never written: it is selected away, not multiplied.
    float acc = 0.f;
    for (int s0 = wid; s0 < p.S; s0 += 64) {
        float ls[8], v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int s = s0 + 8 * j;
            ls[j] = s < p.S ? p.part_lse[(int64_t)s * p.rows + row] : -INFINITY;
            v[j] = s < p.S ? load1<kBf16In>(p.part_out, ((int64_t)s * p.rows + row) * kDv + col) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (ls[j] != -INFINITY) acc = fmaf(exp2f((ls[j] - lse_out) * kLog2e), v[j], acc);
    }
    part[wid][lane] = acc;
    __syncthreads();
    if (wid == 0) {
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) t += part[i][lane];
        __nv_bfloat16 v = __float2bfloat16_rn(t);
        p.out[row * kDv + col] = *reinterpret_cast<uint16_t*>(&v);
        if ((blockIdx.x & 15) == 0 && lane == 0 && p.lse) p.lse[row] = lse_out;
    }
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

}  // namespace

cudaError_t launch_merge(const MergeParams& p, cudaStream_t stream) {
    if (p.rows == 0) return cudaSuccess;
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
